"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` takes the oracle module and raises ``AssertionError`` when it
disagrees with a fixed point: hand-derived fixtures under ``tests/golden``,
closed forms, invariants of the method, brute force on tiny layers.  They are
functions (not tests) so that ``test_oracle_planted.py`` can run the whole
suite against deliberately broken copies of the oracle and check that each
planted mistake is caught.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np

import moe_inputs as mi
from tests import pure_python_layer as ppl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# Tiny layers: every feature of the method at sizes brute force can handle.
TINY_SOFTMAX = mi.LayerSpec(name="t_softmax", hidden=16, n_experts=4, top_k=2, expert_ffn=8,
                            latent=0, group_size=8, shared_ffn=8, act="swiglu",
                            router="softmax", weight_std=0.3)
TINY_LATENT = mi.LayerSpec(name="t_latent", hidden=16, n_experts=5, top_k=3, expert_ffn=16,
                           latent=8, group_size=8, shared_ffn=8, act="relu2",
                           router="sigmoid", renormalize=True, routed_scale=2.5,
                           router_bias=True, weight_std=0.3, bias_std=0.05)
TINY_FP16 = mi.LayerSpec(name="t_fp16", hidden=24, n_experts=6, top_k=3, expert_ffn=8,
                         latent=0, group_size=8, shared_ffn=16, act="swiglu",
                         router="sigmoid", renormalize=True, routed_scale=1.0,
                         act_dtype="fp16", scale_dtype="fp16", router_dtype="fp32",
                         weight_std=0.3)
TINY_UNNORM = TINY_SOFTMAX.with_(name="t_unnorm", renormalize=False, n_experts=5, top_k=3)
# 2-, 3-, 5-, 6- and 8-bit expert codes (rows of K codes fill whole words: K * bits % 32 == 0)
TINY_B3 = TINY_SOFTMAX.with_(name="t_b3", hidden=32, expert_ffn=32, bits=3)
TINY_B8 = TINY_LATENT.with_(name="t_b8", bits=8)
TINY_B2 = TINY_SOFTMAX.with_(name="t_b2", hidden=32, expert_ffn=32, bits=2)
TINY_B5 = TINY_LATENT.with_(name="t_b5", bits=5, latent=32, hidden=32, expert_ffn=32)
TINY_B6 = TINY_FP16.with_(name="t_b6", bits=6, hidden=32, expert_ffn=32)
TINY_SPECS = (TINY_SOFTMAX, TINY_LATENT, TINY_FP16, TINY_UNNORM, TINY_B3, TINY_B8, TINY_B2, TINY_B5,
              TINY_B6)


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


def _layer_and_x(spec, seed=0, T=3):
    layer = mi.make_layer(spec, seed)
    x = mi.make_x(spec, T, seed)
    return layer, x


# --- storage ---------------------------------------------------------------

def pin_unpack_fixture(ora):
    """Code order of packed words against hand-written words: 4-bit codes
    (int4_words.txt) and 3-bit and 8-bit codes (packed_words.txt, codes that
    straddle two words included)."""
    with open(os.path.join(GOLDEN, "int4_words.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            word = np.array([int(line[0], 16)], dtype=np.uint32)
            want = [int(v) for v in line[1:]]
            got = ora.unpack_codes(word).tolist()
            assert got == want, (line[0], got, want)
    n = 0
    with open(os.path.join(GOLDEN, "packed_words.txt")) as f:
        for line in f:
            line = line.split("#")[0]
            if not line.strip():
                continue
            head, codes = line.split("|")
            head = head.split()
            bits = int(head[0])
            words = np.array([int(v, 16) for v in head[1:]], dtype=np.uint32)
            want = [int(v) for v in codes.split()]
            got = ora.unpack_codes(words, bits).tolist()
            assert got == want, (bits, head[1:], got, want)
            n += 1
    assert n >= 7


def pin_dequant_closed_form(ora):
    """code 0 -> bias; code 15 -> 15*scale + bias; each element uses the scale
    of its own group (k // G), checked with exactly representable values."""
    N, K, G = 3, 32, 8
    ng = K // G
    scale = np.array([[0.5 * (g + 1) + n for g in range(ng)] for n in range(N)])
    bias = np.array([[-(g + 1) * 0.25 - n for g in range(ng)] for n in range(N)])
    s_st, b_st = mi.round_to_bf16_bits(scale), mi.round_to_bf16_bits(bias)
    for code in (0, 1, 7, 15):
        packed = mi.pack_int4(np.full((N, K), code, dtype=np.uint8))
        got = ora.dequantize(packed, s_st, b_st, G, "bf16")
        for n in range(N):
            for kk in range(K):
                assert got[n, kk] == code * scale[n, kk // G] + bias[n, kk // G]
    # distinct codes along a row: element kk gets code kk % 16
    codes = np.array([[kk % 16 for kk in range(K)]] * N, dtype=np.uint8)
    got = ora.dequantize(mi.pack_int4(codes), s_st, b_st, G, "bf16")
    for n in range(N):
        for kk in range(K):
            assert got[n, kk] == (kk % 16) * scale[n, kk // G] + bias[n, kk // G]


def pin_dequant_closed_form_bits(ora):
    """2-, 3-, 5-, 6- and 8-bit codes: code 0 -> bias, the top code 2^b - 1 -> (2^b - 1)*scale +
    bias, every element on its own group's scale and bias."""
    N, K, G = 2, 64, 32
    ng = K // G
    scale = np.array([[0.25 * (g + 1) + n for g in range(ng)] for n in range(N)])
    bias = np.array([[-(g + 1) * 0.5 - n for g in range(ng)] for n in range(N)])
    s_st, b_st = mi.round_to_bf16_bits(scale), mi.round_to_bf16_bits(bias)
    for bits in (2, 3, 5, 6, 8):
        top = (1 << bits) - 1
        for code in (0, 1, top // 2, top):
            packed = mi.pack_codes(np.full((N, K), code, dtype=np.uint8), bits)
            got = ora.dequantize(packed, s_st, b_st, G, "bf16", bits)
            for n in range(N):
                for kk in range(K):
                    assert got[n, kk] == code * scale[n, kk // G] + bias[n, kk // G], (bits, code)
        codes = np.array([[(7 * kk + n) % (top + 1) for kk in range(K)] for n in range(N)], dtype=np.uint8)
        got = ora.dequantize(mi.pack_codes(codes, bits), s_st, b_st, G, "bf16", bits)
        for n in range(N):
            for kk in range(K):
                assert got[n, kk] == codes[n, kk] * scale[n, kk // G] + bias[n, kk // G]


def pin_quant_roundtrip_bits(ora):
    """2-, 3-, 5-, 6- and 8-bit: the generator's quantiser applied to the oracle's
    dequantised weights gives back the same codes where a group holds both end
    codes (its min/max reproduce scale and bias), and the error of a round trip
    is at most half a step plus the scale/bias storage rounding."""
    rng = np.random.Generator(np.random.PCG64(21))
    for bits, sdt, G, eps in ((3, "bf16", 64, 2.0 ** -8), (8, "fp16", 32, 2.0 ** -11),
                              (2, "bf16", 32, 2.0 ** -8), (5, "fp16", 128, 2.0 ** -11),
                              (6, "bf16", 64, 2.0 ** -8)):
        top = (1 << bits) - 1
        w = rng.normal(0, 0.02, size=(6, 256))
        q, s, b = mi.quantize_affine(w, G, bits, sdt)
        deq = ora.dequantize(mi.pack_codes(q, bits), s, b, G, sdt, bits)
        qg = q.reshape(6, 256 // G, G)
        keep = (qg.min(-1) == 0) & (qg.max(-1) == top)
        q2, _, _ = mi.quantize_affine(deq, G, bits, sdt)
        assert keep.mean() > 0.9
        assert np.array_equal(q2.reshape(6, 256 // G, G)[keep], qg[keep])
        sf = np.repeat(mi.bf16_bits_to_f32(s) if sdt == "bf16" else s.astype(np.float64), G, -1)
        bf = np.repeat(mi.bf16_bits_to_f32(b) if sdt == "bf16" else b.astype(np.float64), G, -1)
        bound = sf / 2 + top * eps * np.abs(sf) + eps * np.abs(bf) + 1e-12
        assert np.all(np.abs(w - deq) <= bound)


def _nvfp4_fixture():
    tabs = {"e2m1": {}, "e4m3": {}, "e8m0": {}}
    for line in open(os.path.join(GOLDEN, "nvfp4_formats.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        key, txt = int(f[1], 16), f[2]
        if txt == "nan":
            val = math.nan
        elif txt.startswith("2^"):
            val = math.ldexp(1.0, int(txt[2:]))
        else:
            val = -0.0 if txt == "-0" else float(Fraction(txt))
        tabs[f[0]][key] = val
    return tabs["e2m1"], tabs["e4m3"], tabs["e8m0"]


def pin_nvfp4_format_fixture(ora):
    """Every E2M1 code and the listed E4M3 and E8M0 bytes decode to the
    hand-worked values of nvfp4_formats.txt (signs of zeros included, NaN
    where listed)."""
    e2m1, e4m3, e8m0 = _nvfp4_fixture()
    assert len(e2m1) == 16 and len(e4m3) >= 20 and len(e8m0) >= 8
    for tab, fn in ((e2m1, ora.e2m1_values), (e4m3, ora.e4m3_values), (e8m0, ora.e8m0_values)):
        keys = np.array(sorted(tab))
        got = np.asarray(fn(keys), dtype=np.float64)
        for k, g in zip(keys, got):
            want = tab[int(k)]
            if math.isnan(want):
                assert math.isnan(g), (hex(k), g)
            else:
                assert g == want and math.copysign(1, g) == math.copysign(1, want), (hex(k), g, want)


def pin_e4m3_grid(ora):
    """The 127 non-negative finite E4M3 bytes (0x00..0x7E) decode to strictly
    increasing multiples of 2^-9 from 0 to 448; setting the sign bit negates;
    0x7F and 0xFF are NaN; between consecutive powers of two from 2^-6 on
    there are exactly 8 values (3 mantissa bits)."""
    v = np.asarray(ora.e4m3_values(np.arange(0x7F)), dtype=np.float64)
    assert v[0] == 0 and v[-1] == 448 and np.all(np.diff(v) > 0)
    assert np.all(v * 512 == np.rint(v * 512))
    assert np.array_equal(np.asarray(ora.e4m3_values(np.arange(0x7F) | 0x80)), -v)
    assert np.isnan(ora.e4m3_values(np.array([0x7F, 0xFF]))).all()
    for p2 in range(-6, 8):
        n = int(((v >= 2.0 ** p2) & (v < 2.0 ** (p2 + 1))).sum())
        assert n == 8, (p2, n)


def pin_dequant_nvfp4_worked_example(ora):
    """Two blocks of one row, worked by hand: block 0 holds every code with
    scale byte 0x40 (2.0); block 1 repeats codes 0x7 and 0x9 with scale byte 0x01
    (2^-9); the matrix scale is 0.25."""
    codes = np.array([[0x2, 0xA, 0x7, 0xF, 0x1, 0x9, 0x0, 0x8, 0x3, 0x4, 0x5, 0x6, 0xB, 0xC, 0xD, 0xE]
                      + [0x7, 0x9] * 8], dtype=np.uint8)
    scale = np.array([[0x40, 0x01]], dtype=np.uint8)
    want = [0.5, -0.5, 3, -3, 0.25, -0.25, 0, -0, 0.75, 1, 1.5, 2, -0.75, -1, -1.5, -2] + \
           [6 / 2048, -0.5 / 2048] * 8
    got = ora.dequantize_nvfp4(mi.pack_codes(codes, 4), scale, np.float32(0.25))
    assert got.shape == (1, 32)
    assert np.array_equal(got[0], np.array(want, dtype=np.float64)), got


def pin_dequant_mxfp4_worked_example(ora):
    """Two 32-element blocks of one row, worked by hand: block 0 holds the
    sixteen codes twice with scale byte 0x7F (1), block 1 codes 0x7 and 0xD
    with scale byte 0x7C (1/8)."""
    order = [0x2, 0xA, 0x7, 0xF, 0x1, 0x9, 0x0, 0x8, 0x3, 0x4, 0x5, 0x6, 0xB, 0xC, 0xD, 0xE]
    codes = np.array([order * 2 + [0x7, 0xD] * 16], dtype=np.uint8)
    scale = np.array([[0x7F, 0x7C]], dtype=np.uint8)
    vals = [1, -1, 6, -6, 0.5, -0.5, 0, -0, 1.5, 2, 3, 4, -1.5, -2, -3, -4]
    want = vals * 2 + [0.75, -0.375] * 16
    got = ora.dequantize_mxfp4(mi.pack_codes(codes, 4), scale)
    assert got.shape == (1, 64)
    assert np.array_equal(got[0], np.array(want, dtype=np.float64)), got


def pin_mxfp4_quant_roundtrip(ora):
    """The generator's MXFP4 quantiser and the oracle's decoder: each block's
    scale X puts the block's largest magnitude in [4 X, 8 X) (the largest E2M1
    exponent is 2), and every weight is within 2 X of its value (at most the
    clip from 8 X to 6 X; inside the grid at most half the largest gap)."""
    rng = np.random.Generator(np.random.PCG64(35))
    w = rng.normal(0, 0.02, size=(8, 128))
    q, sb = mi.quantize_mxfp4(w)
    deq = ora.dequantize_mxfp4(mi.pack_codes(q, 4), sb)
    X = ora.e8m0_values(sb)
    bmax = np.abs(w).reshape(8, 4, 32).max(-1)
    assert np.all((bmax >= 4 * X) & (bmax < 8 * X))
    assert np.all(np.abs(w - deq) <= 2 * np.repeat(X, 32, axis=-1) + 1e-15)


def pin_nvfp4_quant_roundtrip(ora):
    """The generator's NVFP4 quantiser and the oracle's decoder: every weight is
    within half the largest E2M1 gap (1.0) of its block scale S of its value,
    each block's largest magnitude is reproduced to within the E4M3 rounding
    (1/16 relative) or is saturated at 6 S, and re-quantising the decoded
    weights gives back the same codes and scales."""
    rng = np.random.Generator(np.random.PCG64(33))
    w = rng.normal(0, 0.02, size=(8, 128))
    q, sb, gs = mi.quantize_nvfp4(w)
    deq = ora.dequantize_nvfp4(mi.pack_codes(q, 4), sb, gs)
    S = np.repeat(ora.e4m3_values(sb), 16, axis=-1) * float(gs)
    assert np.all(np.abs(w - deq) <= S * 1.0 + 1e-15)
    bmax = np.abs(w).reshape(8, 8, 16).max(-1)
    dmax = np.abs(deq).reshape(8, 8, 16).max(-1)
    assert np.all(np.abs(dmax - bmax) <= bmax / 16 + 1e-12)
    q2, sb2, gs2 = mi.quantize_nvfp4(deq)
    assert np.float32(gs2) <= np.float32(gs)
    deq2 = ora.dequantize_nvfp4(mi.pack_codes(q2, 4), sb2, gs2)
    assert np.allclose(deq2, deq, rtol=0, atol=float(np.max(S)))


def pin_quant_roundtrip(ora):
    """The generator's quantiser applied to the oracle's dequantised weights
    gives back the same codes (groups hold codes 0 and 15, so the recomputed
    min/max reproduce scale and bias)."""
    rng = np.random.Generator(np.random.PCG64(5))
    for sdt, G in (("bf16", 64), ("fp16", 32), ("bf16", 128)):
        w = rng.normal(0, 0.02, size=(6, 256))
        q, s, b = mi.quantize_affine_int4(w, G, sdt)
        qg = q.reshape(6, 256 // G, G)
        keep = (qg.min(-1) == 0) & (qg.max(-1) == 15)
        deq = ora.dequantize(mi.pack_int4(q), s, b, G, sdt)
        q2, s2, b2 = mi.quantize_affine_int4(deq, G, sdt)
        q2g = q2.reshape(6, 256 // G, G)
        assert keep.mean() > 0.9
        assert np.array_equal(q2g[keep], qg[keep])


def pin_quant_error_bound(ora):
    """|w - deq(quant(w))| <= scale/2 plus the scale/bias storage rounding
    (15 steps of half an ulp of the scale, half an ulp of the bias)."""
    rng = np.random.Generator(np.random.PCG64(9))
    for sdt, G, eps in (("bf16", 64, 2.0 ** -8), ("fp16", 32, 2.0 ** -11)):
        w = rng.normal(0, 0.02, size=(8, 512))
        q, s, b = mi.quantize_affine_int4(w, G, sdt)
        deq = ora.dequantize(mi.pack_int4(q), s, b, G, sdt)
        sf = np.repeat(mi.bf16_bits_to_f32(s) if sdt == "bf16" else s.astype(np.float64), G, -1)
        bf = np.repeat(mi.bf16_bits_to_f32(b) if sdt == "bf16" else b.astype(np.float64), G, -1)
        bound = sf / 2 + 15 * eps * np.abs(sf) + eps * np.abs(bf) + 1e-12
        assert np.all(np.abs(w - deq) <= bound)
        assert np.max(np.abs(w - deq) / sf) > 0.3     # not trivially exact


# --- routing ---------------------------------------------------------------

def pin_topk_bruteforce(ora):
    """Top-k = the k-subset with the largest key sum (exhaustive search), in
    descending key order."""
    rng = np.random.Generator(np.random.PCG64(11))
    for trial in range(200):
        E = int(rng.integers(2, 11))
        k = int(rng.integers(1, E + 1))
        keys = rng.normal(size=E)
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(keys[i] for i in c))
        got = ora.topk_order(keys, k).tolist()
        assert sorted(got) == sorted(best), (keys, k, got, best)
        assert all(keys[got[i]] >= keys[got[i + 1]] for i in range(k - 1))


def _golden_routing():
    with open(os.path.join(GOLDEN, "routing_cases.json")) as f:
        return json.load(f)


def pin_topk_fixture(ora):
    """Ties go to the lower index; non-finite keys rank after every finite key."""
    for case in _golden_routing()["topk_keys"]:
        keys = np.array([float(v) for v in case["keys"]])
        got = ora.topk_order(keys, case["k"]).tolist()
        assert got == case["ids"], (case["name"], got)


def pin_route_closed_forms(ora):
    """Routing weights against hand-derived fractions (logits ln of rationals)."""
    for case in _golden_routing()["cases"]:
        spec = mi.LayerSpec(name="r", hidden=8, n_experts=len(case["z_ln"]), top_k=case["k"],
                            expert_ffn=8, group_size=8, router=case["router"],
                            renormalize=case["renormalize"],
                            routed_scale=case["routed_scale"],
                            router_bias=case["bias"] is not None)
        z = np.array([math.log(float(Fraction(v))) for v in case["z_ln"]])
        bias = None if case["bias"] is None else np.array(case["bias"])
        ids, w = ora.route(z, spec, bias)
        assert ids.tolist() == case["ids"], (case["name"], ids)
        want = [float(Fraction(v)) for v in case["w"]]
        assert np.allclose(w, want, rtol=1e-13, atol=0), (case["name"], w, want)


def pin_routing_margin(ora):
    """The k-th minus the (k+1)-th selection key against hand-derived gaps: on
    the key (score + bias for sigmoid routing, not the logit), with
    non-finite keys ranked last, infinite when no (k+1)-th finite key exists."""
    for case in _golden_routing()["margin_cases"]:
        if "z_ln" in case:
            z = np.array([math.log(float(Fraction(v))) for v in case["z_ln"]])
        else:
            z = np.array([float(v) for v in case["z"]])
        spec = mi.LayerSpec(name="m", hidden=8, n_experts=len(z), top_k=case["k"],
                            expert_ffn=8, group_size=8, router=case["router"],
                            router_bias=case["bias"] is not None)
        bias = None if case["bias"] is None else np.array(case["bias"])
        got = ora.routing_margin(z, spec, bias)
        if case["margin"] == "inf":
            assert got == math.inf, (case["name"], got)
        else:
            want = float(Fraction(case["margin"]))
            assert abs(got - want) <= 1e-12, (case["name"], got, want)


def pin_weight_sums(ora):
    """Normalised weights sum to the routed scale; a full softmax sums to 1
    over all experts."""
    rng = np.random.Generator(np.random.PCG64(13))
    for spec in (mi.SPECS["latent"], mi.SPECS["nonlatent"], mi.SPECS["tiny"]):
        for _ in range(20):
            z = rng.normal(0, 1.5, size=spec.n_experts)
            bias = rng.normal(0, 0.01, size=spec.n_experts) if spec.router_bias else None
            ids, w = ora.route(z, spec, bias)
            assert len(set(ids.tolist())) == spec.top_k
            assert abs(w.sum() - spec.routed_scale) < 1e-12
    spec = TINY_UNNORM.with_(top_k=TINY_UNNORM.n_experts)
    z = rng.normal(size=spec.n_experts)
    _, w = ora.route(z, spec, None)
    assert abs(w.sum() - 1.0) < 1e-12


def pin_activation_closed_forms(ora):
    """silu(ln 3) = (3/4) ln 3, silu(0) = 0, relu^2 of (-1, 0, 2) = (0, 0, 4)."""
    sw = mi.SPECS["tiny"]
    lr = mi.SPECS["latent"]
    g = np.array([math.log(3.0), 0.0, -math.log(3.0)])
    u = np.array([2.0, 5.0, 4.0])
    got = ora.activation(sw, u, g)
    want = np.array([0.75 * math.log(3.0) * 2.0, 0.0, 0.25 * -math.log(3.0) * 4.0])
    assert np.allclose(got, want, rtol=1e-14, atol=1e-300)
    assert np.array_equal(ora.activation(lr, np.array([-1.0, 0.0, 2.0]), None), [0.0, 0.0, 4.0])


# --- the layer ---------------------------------------------------------------

def pin_pure_python(ora):
    """The whole layer against a brute-force pure-Python forward on tiny layers
    (all routers, activations, dtypes, latent and non-latent)."""
    for spec in TINY_SPECS:
        for seed in (0, 1):
            layer, x = _layer_and_x(spec, seed, T=3)
            out, ids, w = ppl.forward(layer, x)
            r = ora.oracle_forward(layer, x)
            assert r["ids"].tolist() == ids, (spec.name, r["ids"], ids)
            assert _rel(r["w"], w) < 1e-12, spec.name
            assert _rel(r["out"], out) < 1e-12, (spec.name, _rel(r["out"], out))


def pin_k_equals_e(ora):
    """With k = E every expert is used: the routed output is the dense sum over
    all experts with full softmax (or normalised sigmoid) weights, computed
    here by direct matrix products on independently unpacked weights."""
    for spec in (TINY_SOFTMAX, TINY_LATENT):
        spec = spec.with_(top_k=spec.n_experts)
        layer, x = _layer_and_x(spec, 3, T=2)
        r = ora.oracle_forward(layer, x)
        G, sdt, adt = spec.group_size, spec.scale_dtype, spec.act_dtype
        to64 = (lambda a: mi.bf16_bits_to_f32(a).astype(np.float64)) if adt == "bf16" else \
            (lambda a: np.asarray(a, np.float64))
        sto64 = (lambda a: mi.bf16_bits_to_f32(a).astype(np.float64))

        def deq(qw, s, b):
            return (mi.unpack_int4(qw).astype(np.float64) * np.repeat(sto64(s), G, -1)
                    + np.repeat(sto64(b), G, -1))
        xs = to64(x)
        Wr = to64(layer.router_w)
        for t in range(xs.shape[0]):
            z = Wr @ xs[t]
            if spec.router == "softmax":
                p = np.exp(z - z.max())
                wts = p / p.sum()
            else:
                sg = 1.0 / (1.0 + np.exp(-z))
                wts = spec.routed_scale * sg / sg.sum()
            xin = to64(layer.fc1) @ xs[t] if spec.latent else xs[t]
            y = np.zeros(spec.k_in)
            for e in range(spec.n_experts):
                u = deq(layer.up_q[e], layer.up_s[e], layer.up_b[e]) @ xin
                if spec.gated:
                    g = deq(layer.gate_q[e], layer.gate_s[e], layer.gate_b[e]) @ xin
                    h = g / (1 + np.exp(-g)) * u
                else:
                    h = np.maximum(u, 0) ** 2
                y += wts[e] * (deq(layer.down_q[e], layer.down_s[e], layer.down_b[e]) @ h)
            assert _rel(r["y"][t], y) < 1e-12, (spec.name, t)
            assert sorted(r["ids"][t].tolist()) == list(range(spec.n_experts))


def pin_expert_permutation(ora):
    """Relabelling the experts (router rows, router bias, expert tensors) leaves
    the output unchanged and maps the selected ids through the relabelling."""
    for spec in (TINY_SOFTMAX, TINY_LATENT, TINY_FP16):
        layer, x = _layer_and_x(spec, 4, T=3)
        r = ora.oracle_forward(layer, x)
        perm = np.random.Generator(np.random.PCG64(21)).permutation(spec.n_experts)
        inv = np.argsort(perm)           # new expert i is old expert perm[i]
        arrays = {}
        for name in ("router_w", "router_bias", "gate_q", "gate_s", "gate_b", "up_q", "up_s",
                     "up_b", "down_q", "down_s", "down_b"):
            v = getattr(layer, name)
            arrays[name] = None if v is None else v[perm]
        import dataclasses
        layer_p = dataclasses.replace(layer, **arrays)
        rp = ora.oracle_forward(layer_p, x)
        assert _rel(rp["out"], r["out"]) < 1e-12
        assert np.array_equal(perm[rp["ids"]], r["ids"])
        assert np.array_equal(inv[r["ids"]], rp["ids"])


def pin_single_expert_is_dense_mlp(ora):
    """E = 1, k = 1 with softmax routing: weight 1, and the layer is the
    textbook residual MLP x + down(silu(gate x) * up x) + shared(x)."""
    spec = TINY_SOFTMAX.with_(n_experts=1, top_k=1)
    layer, x = _layer_and_x(spec, 6, T=2)
    r = ora.oracle_forward(layer, x)
    assert np.array_equal(r["w"], np.ones((2, 1)))
    xs = mi.bf16_bits_to_f32(x).astype(np.float64)
    G = spec.group_size

    def deq(qw, s, b):
        return (mi.unpack_int4(qw).astype(np.float64)
                * np.repeat(mi.bf16_bits_to_f32(s).astype(np.float64), G, -1)
                + np.repeat(mi.bf16_bits_to_f32(b).astype(np.float64), G, -1))
    up = deq(layer.up_q[0], layer.up_s[0], layer.up_b[0])
    gate = deq(layer.gate_q[0], layer.gate_s[0], layer.gate_b[0])
    down = deq(layer.down_q[0], layer.down_s[0], layer.down_b[0])
    f64 = lambda a: mi.bf16_bits_to_f32(a).astype(np.float64)
    silu = lambda v: v / (1 + np.exp(-v))
    want = (xs + (silu(xs @ gate.T) * (xs @ up.T)) @ down.T
            + (silu(xs @ f64(layer.sh_gate).T) * (xs @ f64(layer.sh_up).T)) @ f64(layer.sh_down).T)
    assert _rel(r["out"], want) < 1e-12


def pin_zero_input(ora):
    """x = 0 gives out = 0 exactly: every product of the layer has a zero
    factor (routing still picks experts and weights, which multiply zeros)."""
    for spec in TINY_SPECS:
        layer = mi.make_layer(spec, 0)
        dt = np.uint16 if spec.act_dtype == "bf16" else np.float16
        x = np.zeros((2, spec.hidden), dtype=dt)
        r = ora.oracle_forward(layer, x)
        assert np.all(r["out"] == 0.0), spec.name
        if spec.renormalize:
            assert np.abs(r["w"].sum(axis=1) - spec.routed_scale).max() < 1e-12


def pin_row_invariance(ora):
    """A T-row pass equals T one-row passes, bit for bit."""
    for spec in (TINY_SOFTMAX, TINY_LATENT):
        layer, x = _layer_and_x(spec, 8, T=5)
        r = ora.oracle_forward(layer, x)
        for t in range(5):
            rt = ora.oracle_forward(layer, x[t:t + 1])
            assert np.array_equal(rt["out"][0], r["out"][t])
            assert np.array_equal(rt["ids"][0], r["ids"][t])


def pin_residual_and_shared_terms(ora):
    """Removing the shared expert removes exactly the shared MLP's output, and
    scaling the routed scale by c scales the routed part (out - x - shared)
    by c."""
    spec = TINY_LATENT
    layer, x = _layer_and_x(spec, 10, T=2)
    r = ora.oracle_forward(layer, x)
    import dataclasses
    no_sh = dataclasses.replace(layer, spec=spec.with_(shared_ffn=0), sh_up=None, sh_down=None,
                                sh_gate=None)
    r0 = ora.oracle_forward(no_sh, x)
    xs = mi.bf16_bits_to_f32(x).astype(np.float64)
    f64 = lambda a: mi.bf16_bits_to_f32(a).astype(np.float64)
    shared = (np.maximum(xs @ f64(layer.sh_up).T, 0) ** 2) @ f64(layer.sh_down).T
    assert _rel(r["out"] - r0["out"], shared) < 1e-12
    routed = r0["out"] - xs
    scaled = dataclasses.replace(no_sh, spec=no_sh.spec.with_(routed_scale=5.0))
    r2 = ora.oracle_forward(scaled, x)
    assert _rel(r2["out"] - xs, 2.0 * routed) < 1e-12


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
