"""The C-ABI library on the host: it loads, exports every declared entry
point, and refuses bad configs before touching a device (no GPU needed)."""
import ctypes
import os
import re

import pytest

import quantized_moe_decode_gemv_gb300 as pkg
from quantized_moe_decode_gemv_gb300 import _capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_layer.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_capi.LIB_PATH):
        pytest.fail("libmoe_gb300.so is not built; run __graft_entry__.build()")
    return _capi.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_layer_create", "moe_layer_forward", "moe_layer_destroy"):
        assert n in names
    assert set(names) == set(_capi.SIGNATURES), set(names) ^ set(_capi.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.moe_abi_version() == 4


def test_status_strings(lib):
    for i, name in enumerate(_capi.STATUS_NAMES):
        assert lib.moe_status_string(i).decode() == name


def _cfg(**kw):
    base = dict(hidden=512, n_experts=16, top_k=2, expert_ffn=256, latent=0, group_size=64,
                shared_ffn=256, max_tokens=4, act="swiglu", router="softmax")
    base.update(kw)
    return pkg.MoEConfig(**base)


FAKE = 0x1000  # non-NULL placeholder pointers: validation only checks presence


def _w(**kw):
    w = {n: FAKE for n in ("router_w", "gate_q", "up_q", "down_q", "gate_s", "gate_b", "up_s",
                           "up_b", "down_s", "down_b", "sh_gate", "sh_up", "sh_down")}
    w.update(kw)
    return _capi.moe_layer_weights(**w)


def _validate(lib, cfg, w=None):
    c = cfg.to_c()
    return lib.moe_layer_validate(ctypes.byref(c), ctypes.byref(w) if w is not None else None)


CASES = [
    ("valid", {}, {}, "MOE_OK"),
    ("top_k above E", {"top_k": 17}, {}, "MOE_ERR_TOPK_GT_E"),
    ("top_k zero", {"top_k": 0}, {}, "MOE_ERR_TOPK_GT_E"),
    ("latent without fc1", {"latent": 256}, {"fc2_latent": FAKE}, "MOE_ERR_LATENT_PROJ"),
    ("latent without fc2", {"latent": 256}, {"fc1_latent": FAKE}, "MOE_ERR_LATENT_PROJ"),
    ("latent fp32", {"latent": 256, "act_dtype": "fp32"}, {"fc1_latent": FAKE, "fc2_latent": FAKE},
     "MOE_ERR_LATENT_PROJ"),
    ("latent given to non-latent layer", {}, {"fc1_latent": FAKE, "fc2_latent": FAKE}, "MOE_ERR_LATENT_PROJ"),
    ("latent ok", {"latent": 256}, {"fc1_latent": FAKE, "fc2_latent": FAKE}, "MOE_OK"),
    ("group 48", {"group_size": 48}, {}, "MOE_ERR_SHAPE"),
    ("hidden not multiple of 64", {"hidden": 520}, {}, "MOE_ERR_SHAPE"),
    ("ffn not multiple of group", {"expert_ffn": 192, "group_size": 128}, {}, "MOE_ERR_SHAPE"),
    ("too many experts", {"n_experts": 2048}, {}, "MOE_ERR_UNSUPPORTED"),
    ("top_k above 16", {"n_experts": 64, "top_k": 17}, {}, "MOE_ERR_UNSUPPORTED"),
    ("bias with softmax", {"router_bias": True}, {"router_bias": FAKE}, "MOE_ERR_UNSUPPORTED"),
    ("swiglu without gate", {}, {"gate_q": None}, "MOE_ERR_INVALID_ARG"),
    ("relu2 with gate", {"act": "relu2"}, {"sh_gate": None}, "MOE_ERR_SHAPE"),
    ("shared weights missing", {}, {"sh_down": None}, "MOE_ERR_UNSUPPORTED"),
    ("shared weights without shared_ffn", {"shared_ffn": 0}, {}, "MOE_ERR_SHAPE"),
    ("no router", {}, {"router_w": None}, "MOE_ERR_INVALID_ARG"),
    ("zero max_tokens", {"max_tokens": 0}, {}, "MOE_ERR_INVALID_ARG"),
    ("3-bit codes", {"bits": 3}, {}, "MOE_OK"),
    ("8-bit codes", {"bits": 8}, {}, "MOE_OK"),
    ("bits 0 means 4", {"bits": 0}, {}, "MOE_OK"),
    ("2-bit codes", {"bits": 2}, {}, "MOE_OK"),
    ("5-bit codes", {"bits": 5}, {}, "MOE_OK"),
    ("6-bit codes", {"bits": 6}, {}, "MOE_OK"),
    ("7-bit codes", {"bits": 7}, {}, "MOE_ERR_INVALID_ARG"),
    ("1-bit codes", {"bits": 1}, {}, "MOE_ERR_INVALID_ARG"),
    ("16-bit codes", {"bits": 16}, {}, "MOE_ERR_INVALID_ARG"),
    ("nvfp4", {"fmt": "nvfp4", "group_size": 16}, {}, "MOE_OK"),
    ("nvfp4 bits 0", {"fmt": "nvfp4", "group_size": 16, "bits": 0}, {}, "MOE_OK"),
    ("nvfp4 fp32 scale dtype ignored", {"fmt": "nvfp4", "group_size": 16, "scale_dtype": "fp32"}, {},
     "MOE_OK"),
    ("nvfp4 block 32", {"fmt": "nvfp4", "group_size": 32}, {}, "MOE_ERR_SHAPE"),
    ("nvfp4 8-bit", {"fmt": "nvfp4", "group_size": 16, "bits": 8}, {}, "MOE_ERR_INVALID_ARG"),
    ("affine group 16", {"group_size": 16}, {}, "MOE_ERR_SHAPE"),
    ("mxfp4", {"fmt": "mxfp4", "group_size": 32}, {}, "MOE_OK"),
    ("mxfp4 without bias pointers", {"fmt": "mxfp4", "group_size": 32},
     {"up_b": None, "down_b": None, "gate_b": None}, "MOE_OK"),
    ("mxfp4 block 16", {"fmt": "mxfp4", "group_size": 16}, {}, "MOE_ERR_SHAPE"),
    ("mxfp4 3-bit", {"fmt": "mxfp4", "group_size": 32, "bits": 3}, {}, "MOE_ERR_INVALID_ARG"),
    ("nvfp4 needs matrix scales", {"fmt": "nvfp4", "group_size": 16}, {"up_b": None}, "MOE_ERR_INVALID_ARG"),
]


@pytest.mark.parametrize("name,ckw,wkw,want", CASES, ids=[c[0] for c in CASES])
def test_validate_refusals(lib, name, ckw, wkw, want):
    st = _validate(lib, _cfg(**ckw), _w(**wkw))
    assert _capi.STATUS_NAMES[st] == want, (name, _capi.STATUS_NAMES[st],
                                            lib.moe_layer_last_error(None))


def test_create_refuses_before_any_allocation(lib):
    """An invalid config is refused by create before any device call, and
    nothing stays allocated."""
    before = lib.moe_debug_live_allocations()
    c = _cfg(top_k=40).to_c()
    w = _w()
    h = ctypes.c_void_p()
    st = lib.moe_layer_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h))
    assert _capi.STATUS_NAMES[st] == "MOE_ERR_TOPK_GT_E"
    assert h.value is None
    assert lib.moe_debug_live_allocations() == before
    assert b"top_k" in lib.moe_layer_last_error(None)


# --- bench.py's gate on captured DRAM traffic ------------------------------------

def test_traffic_gate_ignores_comments_but_not_code():
    """The captured-traffic hash follows the code only: comments and blank
    lines do not change it, a changed statement or string literal does."""
    import bench
    a = 'int f() {\n  // launch 304 CTAs\n  return g("a // b", 304); /* grid */\n}\n'
    b = 'int f() {\n\n  return g("a // b", 304);   // comments moved\n}\n'
    c = 'int f() {\n  return g("a // b", 152);\n}\n'
    d = 'int f() {\n  return g("a // c", 304);\n}\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)


def test_traffic_gate_matches_the_committed_capture():
    """Every captured kernel in profiles/traffic.json either matches the
    current sources (reported) or is reported as null -- never a stale number."""
    import json
    import bench
    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "profiles", "traffic.json")
    if not os.path.exists(path):
        pytest.skip("no captured traffic")
    for key, rec in json.load(open(path))["kernels"].items():
        kernel, tz = key.split("@T")
        zipf = tz.endswith("z")
        T = int(tz.rstrip("z"))
        got = bench.captured_traffic(kernel, T, zipf)
        if rec["source_sha256"] == bench.kernel_source_hash(kernel):
            assert got == float(rec["dram_bytes_per_launch"])
        else:
            assert got is None


def test_unknown_weight_format_refused(lib):
    c = _cfg().to_c()
    c.weight_format = 7
    st = lib.moe_layer_validate(ctypes.byref(c), ctypes.byref(_w()))
    assert _capi.STATUS_NAMES[st] == "MOE_ERR_INVALID_ARG"
    assert b"weight_format" in lib.moe_layer_last_error(None)


def test_algorithmic_byte_model():
    """The bench's algorithmic bytes on the latent layer at T = 1 with 9
    distinct experts: router 4.06 + fc1 8.39 + shared gate 30.4 MB in the pass
    over x, 1.07 MB per expert projection (0.95 MB of codes, 0.12 MB of
    scale/bias words at G = 64; NVFP4 the same; MXFP4 0.06 MB of E8M0 bytes),
    fc2 8.39 + shared down 30.4 MB in the output pass; 100.9 MB in all."""
    import bench
    import moe_inputs as mi
    sp = mi.SPECS["latent"]
    H, E, L, F, Fs = 4096, 496, 1024, 1856, 3712
    b = bench.stage_bytes(sp, 1, 9)
    assert b["dense_in"] == E * H * 2 + L * H * 2 + Fs * H * 2 + H * 2 + E * 4
    assert b["dense_out"] == H * L * 2 + H * Fs * 2 + 2 * H * 2
    assert bench.expert_bytes(sp) == (F * L // 2 + 4 * F * L // 64,) * 2
    assert b["expert_up"] == b["expert_down"] == 9 * (F * L // 2 + F * L // 16)
    assert abs(bench.layer_bytes(sp, 1, 9) - 100.9e6) < 0.1e6
    nv = bench.expert_bytes(sp.with_(fmt="nvfp4", group_size=16))
    mx = bench.expert_bytes(sp.with_(fmt="mxfp4", group_size=32))
    assert nv == (F * L // 2 + F * L // 16 + 4,) * 2
    assert mx == (F * L // 2 + F * L // 32,) * 2
