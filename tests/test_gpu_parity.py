"""CUDA layer against the fp64 oracle, through the C ABI (GPU only).

Inputs are seeded and margin-filtered (the k-th and (k+1)-th oracle selection
keys differ by >= 1e-3), so the selected expert set is unambiguous in fp32 and
must match exactly.  Full-size layers are compared on every row where the
oracle takes seconds, and on sampled rows otherwise (the oracle is row
independent, so a sampled row is checked exactly like a full pass).
"""
import os

import numpy as np
import pytest

import moe_inputs as mi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_moe_decode_gemv_gb300 as pkg
    pkg.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


_HANDLES = {}


# create-time knobs a cached handle was built under
KNOBS = ("MOE_UMMA_V", "MOE_UMMA_TMA", "MOE_UMMA_ABUFS", "MOE_UMMA_NTILE", "MOE_UMMA_SUB",
         "MOE_UMMA_SLEEP", "MOE_GATHER_MIN_T")


def handle_for(name, max_tokens, seed=0, zipf=False, layer=None):
    key = (name, seed, zipf, max_tokens) + tuple(os.environ.get(k) for k in KNOBS)
    if key not in _HANDLES:
        lay = layer if layer is not None else gu.cached_layer(name, seed, zipf)
        _HANDLES[key] = (lay, gu.build_layer(lay, max_tokens))
    return _HANDLES[key]


def teardown_module(module):
    for _, h in _HANDLES.values():
        h.close()
    _HANDLES.clear()


def _parity(name, T, rows=None, max_tokens=None, seed=0, zipf=False, paths=("auto",)):
    """Every path in `paths` against one oracle result of the same inputs."""
    lay, h = handle_for(name, max_tokens or max(T, 16), seed, zipf)
    x, redraws = gu.margin_x(lay, T, seed=seed + T)
    sel = list(range(T)) if rows is None else list(rows)
    ref = gu.ora_forward(lay, x[sel])
    rr = None
    try:
        for path in paths:
            h.set_path(path)
            got = gu.run_layer(h, x, lay.spec.act_dtype)
            rr = gu.check_parity(got, ref, rows=sel, what=f"{name} T={T} path={path}")
            assert h.device_status() == 0
    finally:
        h.set_path("auto")
    return rr


# the CUDA-core schedule for few token rows
SMALL_T_PATHS = ("gemv",)


# --- tiny layer (oracle in milliseconds): several tiles and ragged tails ------

@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 13, 16])
def test_tiny_parity(T):
    _parity("tiny", T, paths=SMALL_T_PATHS)


# --- odd shapes covering every option of the config -------------------------

ODD = {
    # latent, softmax without renormalisation, SwiGLU, fp16, group 128, F not a power of 2
    "odd_latent_fp16": mi.LayerSpec(name="odd_latent_fp16", hidden=1024, n_experts=40, top_k=6,
                                    expert_ffn=384, latent=256, group_size=128, shared_ffn=320,
                                    act="swiglu", router="softmax", renormalize=False,
                                    routed_scale=1.5, act_dtype="fp16", scale_dtype="fp16",
                                    router_dtype="fp16", weight_std=0.05),
    # non-latent sigmoid without bias or shared expert, squared ReLU, fp32 router, group 32
    "odd_relu2_noshared": mi.LayerSpec(name="odd_relu2_noshared", hidden=768, n_experts=33,
                                       top_k=4, expert_ffn=192, latent=0, group_size=32,
                                       shared_ffn=0, act="relu2", router="sigmoid",
                                       renormalize=True, routed_scale=2.0, router_dtype="fp32",
                                       weight_std=0.05),
    # latent sigmoid with bias, no shared expert, k = E
    "odd_k_eq_e": mi.LayerSpec(name="odd_k_eq_e", hidden=512, n_experts=8, top_k=8,
                               expert_ffn=128, latent=128, group_size=64, shared_ffn=0,
                               act="relu2", router="sigmoid", renormalize=True,
                               routed_scale=2.5, router_bias=True, weight_std=0.05),
    # the non-latent fp16 sigmoid top-k layer's options at a small size: fp32 router
    # without bias, SwiGLU (gate + up in one launch), fp16 activations, fp16 scales,
    # group 32, fp16 shared expert
    "odd_c3_like": mi.LayerSpec(name="odd_c3_like", hidden=768, n_experts=24, top_k=4,
                                expert_ffn=256, latent=0, group_size=32, shared_ffn=256,
                                act="swiglu", router="sigmoid", renormalize=True,
                                routed_scale=1.0, act_dtype="fp16", scale_dtype="fp16",
                                router_dtype="fp32", weight_std=0.05),
    # a single expert (k = E = 1): the dense MLP special case
    "odd_single": mi.LayerSpec(name="odd_single", hidden=256, n_experts=1, top_k=1,
                               expert_ffn=128, latent=0, group_size=64, shared_ffn=64,
                               act="swiglu", router="softmax", weight_std=0.05),
}


@pytest.mark.parametrize("name", sorted(ODD))
@pytest.mark.parametrize("T", [1, 7, 12])
def test_odd_shapes(name, T):
    spec = ODD[name]
    lay = mi.make_layer(spec, 11)
    h = gu.build_layer(lay, 12)
    try:
        x, _ = gu.margin_x(lay, T, seed=3)
        ref = gu.ora_forward(lay, x)
        for path in SMALL_T_PATHS:
            h.set_path(path)
            got = gu.run_layer(h, x, spec.act_dtype)
            gu.check_parity(got, ref, what=f"{name} T={T} path={path}")
            assert h.device_status() == 0
    finally:
        h.close()


# --- latent Bolt-shaped layer (E=496, k=9, latent 1024) at full size ---------

@pytest.mark.parametrize("T", [1, 2, 9, 16])
def test_latent_parity(T):
    _parity("latent", T, paths=SMALL_T_PATHS)


# --- 3- and 8-bit affine codes (gemv schedule): tiny and latent shapes ---------

def _bits_layer(base, bits, seed=0):
    spec = mi.spec_for(base).with_(name=f"{base}_b{bits}", bits=bits)
    return gu.cached_layer_spec(spec, seed)


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
@pytest.mark.parametrize("T", [1, 2, 3, 5, 16])
def test_code_width_tiny_parity(bits, T):
    """Little-endian b-bit code streams (3-, 5- and 6-bit codes straddle words) through
    the gemv expert kernels, on every row; AUTO keeps the gemv schedule."""
    lay = _bits_layer("tiny", bits)
    _, h = handle_for(lay.spec.name, 16, layer=lay)
    assert h.path_for(T) == "gemv"
    _parity(lay.spec.name, T, max_tokens=16, paths=("auto",))


@pytest.mark.parametrize("bits,T,rows", [(b, T, r) for b in (3, 8) for T, r in ((1, None), (2, None), (9, [0, 4, 8]))]
                         + [(b, T, r) for b in (2, 5, 6) for T, r in ((1, None), (9, [0, 4, 8]))])
def test_code_width_latent_parity(bits, T, rows):
    """The latent layer (E=496, k=9, latent 1024, group 64) with 2-, 3-, 5-,
    6- and 8-bit expert codes at full size."""
    lay = _bits_layer("latent", bits)
    handle_for(lay.spec.name, 16, layer=lay)
    _parity(lay.spec.name, T, rows=rows, max_tokens=16, paths=("auto",))


@pytest.mark.parametrize("bits", [2, 3, 5, 6, 8])
def test_code_width_grouped_refused(bits):
    """The tensor-core schedule decodes 4-bit codes only: forcing it on a 3- or
    8-bit layer is refused and the layer keeps its gemv schedule."""
    import quantized_moe_decode_gemv_gb300 as pkg
    lay = _bits_layer("tiny", bits)
    _, h = handle_for(lay.spec.name, 16, layer=lay)
    with pytest.raises(pkg.MoEError) as ei:
        h.set_path("grouped")
    assert "MOE_ERR_UNSUPPORTED" in str(ei.value)
    assert h.path_for(16) == "gemv"


# --- NVFP4 experts: E2M1 codes, E4M3 block scales, fp32 matrix scales ------------

def _fp4_layer(spec, seed=0, fmt="nvfp4"):
    return gu.cached_layer_spec(spec.with_(name=f"{spec.name}_{fmt}", fmt=fmt,
                                           group_size=16 if fmt == "nvfp4" else 32), seed)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 16, 33])
def test_nvfp4_tiny_parity(T):
    """The tiny SwiGLU layer with NVFP4 experts (gate and up in one kernel),
    every row; 33 rows take several passes of 16 pairs over an expert."""
    lay = _fp4_layer(mi.spec_for("tiny"))
    _, h = handle_for(lay.spec.name, 48, layer=lay)
    assert h.path_for(T) == "gemv"
    _parity(lay.spec.name, T, max_tokens=48, paths=("auto",))


@pytest.mark.parametrize("T,rows", [(1, None), (2, None), (9, [0, 4, 8]), (16, [0, 15])])
def test_nvfp4_latent_parity(T, rows):
    """The latent layer (E=496, k=9, latent 1024, squared ReLU) with NVFP4
    experts at full size."""
    lay = _fp4_layer(mi.spec_for("latent"))
    handle_for(lay.spec.name, 16, layer=lay)
    _parity(lay.spec.name, T, rows=rows, max_tokens=16, paths=("auto",))


@pytest.mark.parametrize("T", [1, 4, 12])
def test_nvfp4_fp16_softmax_parity(T):
    """fp16 activations, softmax without renormalisation, SwiGLU, latent 256,
    F = 384 (not a power of two) with NVFP4 experts."""
    lay = _fp4_layer(ODD["odd_latent_fp16"])
    handle_for(lay.spec.name, 16, layer=lay)
    _parity(lay.spec.name, T, max_tokens=16, paths=("auto",))


@pytest.mark.parametrize("T", [1, 3, 16, 33])
def test_mxfp4_tiny_parity(T):
    """MXFP4 experts (E2M1 codes, E8M0 scale per 32) on the tiny SwiGLU layer,
    every row."""
    lay = _fp4_layer(mi.spec_for("tiny"), fmt="mxfp4")
    _, h = handle_for(lay.spec.name, 48, layer=lay)
    assert h.path_for(T) == "gemv"
    _parity(lay.spec.name, T, max_tokens=48, paths=("auto",))


@pytest.mark.parametrize("T,rows", [(1, None), (9, [0, 4, 8]), (16, [0, 15])])
def test_mxfp4_latent_parity(T, rows):
    """The latent layer with MXFP4 experts at full size (the down projection's
    F = 1856 is not a multiple of 128: two scale bytes per 64-column chunk)."""
    lay = _fp4_layer(mi.spec_for("latent"), fmt="mxfp4")
    handle_for(lay.spec.name, 16, layer=lay)
    _parity(lay.spec.name, T, rows=rows, max_tokens=16, paths=("auto",))


@pytest.mark.parametrize("T", [1, 12])
def test_mxfp4_fp16_softmax_parity(T):
    lay = _fp4_layer(ODD["odd_latent_fp16"], fmt="mxfp4")
    handle_for(lay.spec.name, 16, layer=lay)
    _parity(lay.spec.name, T, max_tokens=16, paths=("auto",))


def test_nvfp4_grouped_refused():
    """The tensor-core schedule decodes affine codes only: forcing it on an
    NVFP4 layer is refused and AUTO keeps the gemv schedule at every T."""
    import quantized_moe_decode_gemv_gb300 as pkg
    lay = _fp4_layer(mi.spec_for("tiny"))
    _, h = handle_for(lay.spec.name, 48, layer=lay)
    with pytest.raises(pkg.MoEError) as ei:
        h.set_path("grouped")
    assert "MOE_ERR_UNSUPPORTED" in str(ei.value)
    assert [h.path_for(T) for T in (1, 32, 48)] == ["gemv"] * 3


# --- non-latent fp16 sigmoid top-8 layer (H=6144, E=256) at full size ---------

@pytest.mark.parametrize("T,rows", [(1, None), (4, [0, 3]), (32, [0, 17, 31])])
def test_nonlatent_parity(T, rows):
    """Every path AUTO or a forced schedule gives this layer at its configured
    batch sizes; at 32 rows AUTO takes the grouped tcgen05 path (SwiGLU gate and
    up in one GEMM launch, fp16 scale/bias of group 32)."""
    paths = SMALL_T_PATHS + (("auto",) if T >= 16 else ())
    if T >= 16:
        lay, h = handle_for("nonlatent", 32)
        assert h.path_for(T) == "grouped"
    _parity("nonlatent", T, rows=rows, max_tokens=32, paths=paths)


# --- batched decode rows with Zipf-skewed expert load -------------------------

@pytest.mark.parametrize("T,rows", [(32, [0, 31]), (64, [5, 63]), (256, [0, 128, 255])])
def test_batched_zipf_parity(T, rows):
    _parity("latent", T, rows=rows, max_tokens=256, zipf=True,
            paths=SMALL_T_PATHS + ("auto",) if T < 64 else ("auto",))


# --- prefill-sized batches: the routing over row blocks, then one list CTA ----

@pytest.mark.parametrize("T,rows,gemm", [(65, [0, 64], "k_umma2"), (512, [0, 255, 511], "k_umma2"),
                                         (512, [0, 255, 511], "k_umma"),
                                         (2048, [0, 1023, 2047], "k_umma2")])
def test_prefill_parity(T, rows, gemm, monkeypatch):
    """Above 64 rows the top-k runs over 16-row blocks in parallel and one CTA
    builds the distinct-expert lists from per-expert row bitmasks; the
    grouped tcgen05 path takes every projection (token tiles of a dense
    matrix or of a busy expert spread over CTAs)."""
    for k, v in GEMM_ENV[gemm].items():
        monkeypatch.setenv(k, v)
    _parity("latent", T, rows=rows, max_tokens=2048, zipf=True)


# --- the tcgen05 grouped path (forced at small T, automatic from T = 64) ------

# grouped GEMM variants, selected at create time: the CTA-synchronised K loop
# (k_umma); the warp-specialised roles (k_umma2) with every operand by tensor
# copies, two chunks per ring slot and three dequantised A tiles (default),
# with every operand by cp.async, with two A tiles, with one chunk per slot
# and back-to-back polls, with the up GEMM's B rows gathered by cp.async
GEMM_ENV = {"k_umma": {"MOE_UMMA_V": "1"},
            "k_umma2": {"MOE_UMMA_V": "2"},
            "k_umma2_cpasync": {"MOE_UMMA_V": "2", "MOE_UMMA_TMA": "0"},
            "k_umma2_2buf": {"MOE_UMMA_V": "2", "MOE_UMMA_ABUFS": "2"},
            "k_umma2_slot1": {"MOE_UMMA_V": "2", "MOE_UMMA_SUB": "1", "MOE_UMMA_SLEEP": "0"},
            "k_umma2_nogather": {"MOE_UMMA_V": "2", "MOE_GATHER_MIN_T": "100000"}}


@pytest.mark.parametrize("gemm", list(GEMM_ENV))
@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 16), ("tiny", 37), ("latent", 4),
                                    ("latent", 16), ("odd_latent_fp16", 12),
                                    ("odd_relu2_noshared", 9), ("odd_c3_like", 1),
                                    ("odd_c3_like", 20)])
def test_grouped_path_parity(name, T, gemm, monkeypatch):
    """Every grouped GEMM variant on the tiny, latent and odd layers."""
    for k, v in GEMM_ENV[gemm].items():
        monkeypatch.setenv(k, v)
    if name in ODD:
        lay = mi.make_layer(ODD[name], 11)
    else:
        lay = gu.cached_layer(name)
    h = gu.build_layer(lay, max(T, 16))
    try:
        h.set_path("grouped")
        x, _ = gu.margin_x(lay, T, seed=90 + T)
        got = gu.run_layer(h, x, lay.spec.act_dtype)
        ref = gu.ora_forward(lay, x)
        gu.check_parity(got, ref, what=f"grouped {name} T={T}")
        assert h.device_status() == 0
    finally:
        h.close()


def test_grouped_matches_gemv_path():
    """Both expert paths on the same batch: identical expert choice, outputs
    within the parity bound of each other."""
    lay, h = handle_for("latent", 64, zipf=True)
    x, _ = gu.margin_x(lay, 64, seed=95)
    try:
        h.set_path("gemv")
        a = gu.run_layer(h, x, "bf16")
        h.set_path("grouped")
        b = gu.run_layer(h, x, "bf16")
    finally:
        h.set_path("auto")
    assert np.array_equal(a["ids"], b["ids"])
    assert gu.rel_rms(b["delta"], a["delta"]) <= gu.REL_RMS


# --- heterogeneous five-layer stack, residual stream carried -----------------

_STACK = {}


def stack_layers():
    if "layers" not in _STACK:
        _STACK["layers"] = [mi.make_layer(s, i) for i, s in enumerate(mi.stack_specs())]
    return _STACK["layers"]


@pytest.mark.parametrize("T,rows", [(2, None), (9, [0, 4, 8]), (16, [0, 7, 15])])
def test_stack_parity(T, rows):
    """Five stacked layers (E = 240..496), the output of each the input of the
    next.  Checked rows are margin-filtered at every layer along the oracle's
    own residual stream; the other rows are plain draws.

    The free-running output is compared with the oracle's own stream: its
    error is the sum of five layers' errors carried along the residual path,
    so its max-abs bound is five single-layer bounds (relative RMS stays at
    the single-layer bound).  Re-running the oracle on the GPU's input to each
    layer is no test here: with relu^2 experts and no normalisation the
    synthetic stream grows about quadratically per layer, the later routers'
    logits saturate, and a 1e-4 relative change of the input already moves
    the oracle's own expert choice.

    Each layer is also run on the oracle's stream itself (its bf16 input to
    that layer, on which the checked rows keep the routing margin): the same
    input bits on both sides, held to the single-layer parity gate."""
    layers = stack_layers()
    sel = list(range(T)) if rows is None else rows
    xs, _ = gu.margin_x(layers[0], len(sel), seed=40 + T, stack=layers)
    x = mi.make_x(layers[0].spec, T, 50 + T)
    x[sel] = xs
    handles = [gu.build_layer(l, 16) for l in layers]
    try:
        cur = gu.to_torch_x(x, "bf16")
        ref_in = x[sel]
        for li, (lay, h) in enumerate(zip(layers, handles)):
            out, ids, w, delta = h.forward_ex(cur)
            torch.cuda.synchronize()
            ref = gu.ora_forward(lay, ref_in)
            assert np.array_equal(ids.cpu().numpy()[sel], ref["ids"]), f"layer {li}"
            # Layer 0 sees the same input on both sides: the weights match to the
            # fp32 routing bound.  A later layer's GPU input is the GPU's previous
            # output, within the parity bound (rel. RMS <= 1e-2) of the oracle's;
            # a relative input error e moves a logit by about e * |z| and a
            # sigmoid weight by at most e * |z| / 4 of its unit scale, so those
            # layers are held to the parity bound itself.
            rtol, atol = (gu.W_RTOL, gu.W_ATOL) if li == 0 else (gu.REL_RMS, gu.REL_RMS * 0.1)
            np.testing.assert_allclose(w.cpu().numpy()[sel], ref["w"], rtol=rtol, atol=atol)
            # the same layer on the oracle's input to it
            same = gu.run_layer(h, ref_in, "bf16")
            gu.check_parity(same, ref, what=f"stack layer {li} on the oracle's stream")
            ref_in = mi._round_to_dtype(ref["out"], "bf16")
            cur = out
        final = cur.float().cpu().numpy().astype(np.float64)[sel]
        want = ref["out"]
        assert gu.rel_rms(final, want) <= gu.REL_RMS
        assert gu.max_abs_frac(final, want) <= len(layers) * gu.MAX_ABS_FRAC
        assert np.isfinite(final).all()
    finally:
        for h in handles:
            h.close()


# --- properties of the CUDA path ------------------------------------------------

def test_path_selection_and_launch_counts():
    """AUTO takes the grouped tcgen05 path from 32 rows and the gemv path below;
    a forced path is honoured; a gemv forward of the latent layer is four
    launches (dense pass with the routing, expert up, expert down with the
    combine, output pass)."""
    lay, h = handle_for("latent", 256, zipf=True)
    x = gu.to_torch_x(mi.make_x(lay.spec, 64, 5), "bf16")
    assert [h.path_for(T) for T in (32, 64, 256)] == ["grouped"] * 3
    assert [h.path_for(T) for T in (1, 8, 16, 31)] == ["gemv"] * 4
    try:
        h.set_path("gemv")
        assert h.path_for(64) == "gemv"
        h.forward(x[:1].contiguous())
        assert h.last_launch_count() == 4
        h.set_path("grouped")
        assert h.path_for(1) == "grouped"
    finally:
        h.set_path("auto")
    torch.cuda.synchronize()
    assert h.device_status() == 0

@pytest.mark.parametrize("path", ["gemv", "grouped"])
def test_row_invariance_bit_exact(path):
    """On one path, each row of a 16-row pass equals its own one-row pass, bit
    for bit (no reduction order depends on the other rows of the batch)."""
    lay, h = handle_for("latent", 16)
    x, _ = gu.margin_x(lay, 16, seed=77)
    xt = gu.to_torch_x(x, "bf16")
    try:
        h.set_path(path)
        full = h.forward(xt).clone()
        for t in range(16):
            one = h.forward(xt[t:t + 1].contiguous())
            torch.cuda.synchronize()
            assert torch.equal(one.view(torch.int16), full[t:t + 1].view(torch.int16)), (path, t)
    finally:
        h.set_path("auto")


def test_graph_replay_equals_eager():
    """The forward is stream-capturable: a captured CUDA graph replays to the
    same bits as the eager call."""
    lay, h = handle_for("latent", 16)
    x, _ = gu.margin_x(lay, 4, seed=82)
    xt = gu.to_torch_x(x, "bf16")
    out = torch.empty_like(xt)
    eager = h.forward(xt).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        h.forward(xt, out)          # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h.forward(xt, out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_repeat_is_deterministic():
    lay, h = handle_for("latent", 16)
    x, _ = gu.margin_x(lay, 9, seed=78)
    xt = gu.to_torch_x(x, "bf16")
    a = h.forward(xt).clone()
    b = h.forward(xt)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_host_buffer_forward_matches_device_forward():
    lay, h = handle_for("latent", 16)
    x, _ = gu.margin_x(lay, 4, seed=79)
    xt = gu.to_torch_x(x, "bf16")
    dev = h.forward(xt).cpu()
    xh = xt.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    h.forward_host(xh, oh)
    assert torch.equal(dev.view(torch.int16), oh.view(torch.int16))


def test_two_handles_on_two_streams_equal_solo():
    lay = gu.cached_layer("tiny")
    h1, h2 = gu.build_layer(lay, 16), gu.build_layer(lay, 16)
    try:
        x, _ = gu.margin_x(lay, 16, seed=80)
        xt = gu.to_torch_x(x, "bf16")
        solo = h1.forward(xt).clone()
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        outs = []
        for _ in range(8):
            with torch.cuda.stream(s1):
                a = h1.forward(xt)
            with torch.cuda.stream(s2):
                b = h2.forward(xt)
            outs.append((a, b))
        torch.cuda.synchronize()
        for a, b in outs:
            assert torch.equal(a.view(torch.int16), solo.view(torch.int16))
            assert torch.equal(b.view(torch.int16), solo.view(torch.int16))
    finally:
        h1.close()
        h2.close()


def test_nonfinite_router_keys_rank_last_and_are_reported():
    """A NaN selection bias makes that expert's key non-finite: it ranks below
    every finite key (as in the oracle) and the device status reports it."""
    spec = mi.LayerSpec(name="nan_bias", hidden=512, n_experts=16, top_k=3, expert_ffn=128,
                        latent=0, group_size=64, shared_ffn=0, act="relu2", router="sigmoid",
                        routed_scale=1.0, router_bias=True, weight_std=0.05)
    lay = mi.make_layer(spec, 5)
    lay.router_bias[[2, 7, 11]] = np.nan
    h = gu.build_layer(lay, 4)
    try:
        x, _ = gu.margin_x(lay, 4, seed=81)
        got = gu.run_layer(h, x, "bf16")
        ref = gu.ora_forward(lay, x)
        gu.check_parity(got, ref, what="nan bias")
        assert not np.isin(got["ids"], [2, 7, 11]).any()
        assert h.device_status() == 10  # MOE_ERR_NONFINITE
        assert h.device_status() == 0   # cleared by the read
    finally:
        h.close()


def test_forward_argument_errors():
    import quantized_moe_decode_gemv_gb300 as pkg
    lay, h = handle_for("tiny", 16)
    xt = gu.to_torch_x(mi.make_x(lay.spec, 16, 0), "bf16")
    with pytest.raises(pkg.MoEError, match="INVALID_ARG"):
        pkg.moe_layer_forward(h.handle, xt, 0, torch.empty_like(xt))
    with pytest.raises(pkg.MoEError, match="INVALID_ARG"):
        pkg.moe_layer_forward(h.handle, xt, 17, torch.empty_like(xt))
    with pytest.raises(pkg.MoEError, match="INVALID_ARG"):   # out overlaps x
        pkg.moe_layer_forward(h.handle, xt, 8, xt[4:])
    with pytest.raises(pkg.MoEError, match="INVALID_ARG"):   # unknown path id
        pkg._capi._check(pkg.load_library().moe_layer_set_path(h.handle, 7), h.handle)


def test_refusals_and_allocation_failures_leak_nothing():
    """Refused creates and creates whose n-th device allocation fails free
    everything they allocated (the live-allocation count returns to its
    starting value)."""
    import quantized_moe_decode_gemv_gb300 as pkg
    lib = pkg.load_library()
    lay = gu.cached_layer("tiny")
    cfg = pkg.MoEConfig.from_spec(lay.spec, max_tokens=4)
    dev = pkg.upload_arrays(lay.arrays())
    base = lib.moe_debug_live_allocations()
    bad = pkg.MoEConfig.from_spec(lay.spec, max_tokens=4)
    bad.top_k = 17
    with pytest.raises(pkg.MoEError, match="TOPK_GT_E"):
        pkg.moe_layer_create(bad, dev)
    assert lib.moe_debug_live_allocations() == base
    n_ok = 0
    for n in range(1, 80):
        lib.moe_debug_fail_allocation(n)
        try:
            hh = pkg.moe_layer_create(cfg, dev)
        except pkg.MoEError as e:
            assert e.status == 7  # MOE_ERR_OOM
            assert lib.moe_debug_live_allocations() == base
            continue
        finally:
            lib.moe_debug_fail_allocation(0)
        pkg.moe_layer_destroy(hh)   # n beyond the number of allocations
        n_ok = n
        break
    assert n_ok > 5
    assert lib.moe_debug_live_allocations() == base


def test_smoke_entry():
    import __graft_entry__
    __graft_entry__.smoke()
