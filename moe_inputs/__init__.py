"""Seeded synthetic inputs for the quantized MoE decode layer.

This module only *draws* data: layer shapes, random weights, their int4 affine
group quantisation and packing (the storage format), token activations, and the
per-expert router bias used to skew expert load.  It holds none of the layer's
forward arithmetic (no gemv, routing, activation or combine).  Both the CPU
oracle (``oracle/``) and the CUDA library's tests and bench take their inputs
from here, so the two sides see bit-identical data.

Storage conventions (the library's input format):

* bf16 tensors are numpy ``uint16`` arrays of bf16 bit patterns; fp16 tensors
  are numpy ``float16``; fp32 tensors are ``float32``.
* Expert matrices are row-major ``[E, N_out, K_in]`` with the quantisation
  groups of ``G`` consecutive elements along ``K_in``.  ``q`` holds b-bit
  codes (b = 2, 3, 4, 5, 6 or 8) packed into ``uint32`` words as one little-endian bit
  stream per row, code ``i`` in bits ``b*i .. b*i+b-1`` (for b = 4: eight per
  word, lowest nibble first), giving ``[E, N_out, K_in*b/32]``.  ``scale`` and
  ``bias`` are ``[E, N_out, K_in/G]`` in the layer's scale dtype and a weight
  is reconstructed as ``scale * q + bias`` (MLX-style affine quantisation, as
  the mlx-bun decode-speed program describes its "affine 2/3/4/5/6/8-bit with
  supported group sizes 32/64/128" weights).
* The quantiser used to make synthetic weights is round-to-nearest over each
  group's min/max: ``bias = min``, ``scale = (max - min) / (2^b - 1)`` (both
  rounded to the scale dtype), ``q = clip(rint((w - bias) / scale), 0, 2^b - 1)``.  The pages
  give no quantiser; this one only shapes the test weights.
* NVFP4 experts (``LayerSpec.fmt == "nvfp4"``, group size 16): ``q`` holds
  4-bit E2M1 codes packed as above, ``scale`` one E4M3 byte per 16 elements
  (``uint8 [E, N_out, K_in/16]``) and ``bias`` one float32 scale per expert
  matrix (``[E]``); a weight is ``e2m1(q) * e4m3(scale) * bias``.  The
  synthetic quantiser takes the matrix scale ``amax / (6 * 448)``, each block's
  E4M3 scale as the nearest to ``block amax / (6 * matrix scale)`` and each
  code as the nearest E2M1 value of ``w / (block scale * matrix scale)``.
* MXFP4 experts (``fmt == "mxfp4"``, group size 32): ``q`` as for NVFP4,
  ``scale`` one E8M0 byte per 32 elements (``uint8 [E, N_out, K_in/32]``, the
  power of two ``2^(byte - 127)``) and no ``bias``; the synthetic quantiser
  takes each block's scale as ``2^(floor(log2(block amax)) - 2)`` (2 being the
  largest E2M1 exponent) and each code as the nearest E2M1 value of
  ``w / scale`` (saturating at 6).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "LayerSpec", "LayerWeights", "SPECS", "stack_specs", "make_layer", "make_x",
    "draw_x_rows", "round_to_bf16_bits", "bf16_bits_to_f32", "quantize_affine_int4",
    "quantize_affine", "pack_codes", "unpack_codes", "CODE_BITS", "pack_int4", "unpack_int4",
    "zipf_router_bias", "spec_for", "ROUTED_BYTES", "quantize_nvfp4", "e4m3_round",
    "e2m1_round", "quantize_mxfp4",
]


# ---------------------------------------------------------------------------
# bf16 storage helpers (bit manipulation only)
# ---------------------------------------------------------------------------

def round_to_bf16_bits(a) -> np.ndarray:
    """Round float values to bf16 (round to nearest, ties to even) and return the
    16-bit patterns as ``uint16``.  NaN stays a quiet NaN."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    nan = np.isnan(f)
    r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u16) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def _round_to_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the named storage dtype; returns the storage array."""
    if dtype == "bf16":
        return round_to_bf16_bits(a)
    if dtype == "fp16":
        return np.asarray(a, dtype=np.float64).astype(np.float16)
    if dtype == "fp32":
        return np.asarray(a, dtype=np.float64).astype(np.float32)
    raise ValueError(dtype)


def _storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


# ---------------------------------------------------------------------------
# b-bit packing and the synthetic-weight quantiser
# ---------------------------------------------------------------------------

CODE_BITS = (3, 4, 8)   # code widths of the expert weight formats


def pack_codes(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack b-bit codes ``[..., K]`` (values 0..2^b-1) into ``uint32 [..., K*b/32]``
    as one little-endian bit stream per row: code ``i`` occupies bits
    ``b*i .. b*i+b-1`` of the row, counted from bit 0 of word 0 (a code may
    straddle two words).  For b = 4 this is eight codes per word, lowest
    nibble first; for b = 8 four per word, lowest byte first."""
    q = np.asarray(q)
    K = q.shape[-1]
    if (K * bits) % 32:
        raise ValueError("K * bits must be a multiple of 32")
    if q.size and (q.min() < 0 or q.max() > (1 << bits) - 1):
        raise ValueError(f"codes must be in 0..{(1 << bits) - 1}")
    bitarr = ((q.astype(np.uint32)[..., None] >> np.arange(bits, dtype=np.uint32)) & 1).astype(np.uint8)
    bitarr = bitarr.reshape(*q.shape[:-1], K * bits)
    by = np.packbits(bitarr, axis=-1, bitorder="little")
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32)


def unpack_codes(packed: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of :func:`pack_codes` (used by the generator's own checks)."""
    p = np.ascontiguousarray(np.asarray(packed, dtype=np.uint32))
    K = p.shape[-1] * 32 // bits
    out = np.zeros(p.shape[:-1] + (K,), dtype=np.uint8)
    for i in range(K):
        pos = bits * i
        w, off = pos >> 5, pos & 31
        v = p[..., w].astype(np.uint64) >> np.uint64(off)
        if off + bits > 32:
            v = v | (p[..., w + 1].astype(np.uint64) << np.uint64(32 - off))
        out[..., i] = (v & np.uint64((1 << bits) - 1)).astype(np.uint8)
    return out


def pack_int4(q: np.ndarray) -> np.ndarray:
    """4-bit codes ``[..., K]`` into ``uint32 [..., K/8]``, element ``8*w + i``
    at bits ``4*i``."""
    return pack_codes(q, 4)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_int4` (used by the generator's own checks)."""
    p = np.asarray(packed, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = (p[..., None] >> shifts) & np.uint32(0xF)
    return q.reshape(*p.shape[:-1], p.shape[-1] * 8).astype(np.uint8)


def quantize_affine(w: np.ndarray, group: int, bits: int, scale_dtype: str):
    """Round-to-nearest b-bit affine quantisation of ``w [..., K]`` in groups of
    ``group`` along the last axis: bias = group min, scale = (max - min) /
    (2^b - 1), both rounded to the scale dtype, q = clip(rint((w - bias) /
    scale), 0, 2^b - 1).  Returns ``(q uint8 [..., K], scale, bias)`` with
    scale/bias in storage form ``[..., K/group]``."""
    levels = (1 << bits) - 1
    w = np.asarray(w, dtype=np.float64)
    K = w.shape[-1]
    if K % group:
        raise ValueError("group must divide K")
    wg = w.reshape(*w.shape[:-1], K // group, group)
    lo = wg.min(axis=-1)
    hi = wg.max(axis=-1)
    bias_st = _round_to_dtype(lo, scale_dtype)
    scale_st = _round_to_dtype((hi - lo) / float(levels), scale_dtype)
    b = _storage_to_f64(bias_st, scale_dtype)[..., None]
    s = _storage_to_f64(scale_st, scale_dtype)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.where(s > 0, np.rint((wg - b) / np.where(s > 0, s, 1.0)), 0.0)
    q = np.clip(qf, 0, levels).astype(np.uint8).reshape(w.shape)
    return q, scale_st, bias_st


def quantize_affine_int4(w: np.ndarray, group: int, scale_dtype: str):
    """:func:`quantize_affine` with 4-bit codes."""
    return quantize_affine(w, group, 4, scale_dtype)


# E2M1 magnitudes by the low three code bits (the encoder's grid)
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_round(r: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (sign in bit 3) of each element of ``r`` (magnitudes
    above 6 saturate to 6; an exact tie takes the smaller magnitude)."""
    r = np.asarray(r, dtype=np.float64)
    idx = np.abs(np.abs(r)[..., None] - _E2M1_GRID).argmin(axis=-1)
    return (idx | np.where(r < 0, 8, 0)).astype(np.uint8)


def e4m3_round(a: np.ndarray):
    """Nearest E4M3 byte of each non-negative element of ``a`` (round half to
    even on the mantissa, saturating at 448).  Returns ``(bytes uint8, values
    float64)``: normal values (1 + m/8) 2^(e-7) for e = 1..15 (e = 15 stops at
    m = 6), subnormal m/8 2^-6."""
    a = np.asarray(a, dtype=np.float64)
    if (a < 0).any() or not np.isfinite(a).all():
        raise ValueError("E4M3 scales are encoded from finite non-negative values")
    a = np.minimum(a, 448.0)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)                       # unbiased exponent; below -6: subnormal grid
    step = np.exp2(e - 3)                       # mantissa step at that exponent
    m8 = np.rint(a / step)                      # 8 + m (normal) or m (subnormal, e = -6)
    norm = a >= 2.0 ** -6
    # a carry to 16 moves to the next exponent (still exact: 16 * step = 8 * 2 step)
    carry = norm & (m8 >= 16)
    e = np.where(carry, e + 1, e)
    m8 = np.where(carry, 8, m8)
    val = m8 * np.exp2(e - 3)
    sub_m = np.where(norm, 0, m8).astype(np.int64)            # subnormal 0..8 (8: rounds up to 2^-6)
    byte_norm = ((e + 7).astype(np.int64) << 3) | (m8.astype(np.int64) - 8)
    byte_sub = np.where(sub_m >= 8, 1 << 3, sub_m)
    byte = np.where(norm, byte_norm, byte_sub)
    val = np.where(norm, val, np.where(sub_m >= 8, 2.0 ** -6, sub_m * 2.0 ** -9))
    return byte.astype(np.uint8), val


def quantize_mxfp4(w: np.ndarray):
    """MXFP4 quantisation of ``w [..., N, K]`` (blocks of 32 along K): returns
    ``(q uint8 [..., N, K] E2M1 codes, scale uint8 [..., N, K/32] E8M0 bytes)``
    as described in the module notes (an all-zero block takes 2^0)."""
    w = np.asarray(w, dtype=np.float64)
    K = w.shape[-1]
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    wb = w.reshape(*w.shape[:-1], K // 32, 32)
    bmax = np.abs(wb).max(axis=-1)
    e = np.where(bmax > 0, np.floor(np.log2(np.where(bmax > 0, bmax, 1.0))) - 2, 0)
    e = np.clip(e, -127, 127)
    sb = (e + 127).astype(np.uint8)
    q = e2m1_round(wb / np.exp2(e)[..., None]).reshape(w.shape)
    return q, sb


def quantize_nvfp4(w: np.ndarray):
    """NVFP4 quantisation of ``w [..., N, K]`` (blocks of 16 along K): returns
    ``(q uint8 [..., N, K] E2M1 codes, scale uint8 [..., N, K/16] E4M3 bytes,
    matrix scale float32)`` as described in the module notes."""
    w = np.asarray(w, dtype=np.float64)
    K = w.shape[-1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    amax = float(np.abs(w).max())
    gs = np.float32(amax / (6.0 * 448.0) if amax > 0 else 1.0)
    wb = w.reshape(*w.shape[:-1], K // 16, 16)
    bmax = np.abs(wb).max(axis=-1)
    sb, sv = e4m3_round(bmax / (6.0 * float(gs)))
    S = sv[..., None] * float(gs)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(S > 0, wb / np.where(S > 0, S, 1.0), 0.0)
    q = e2m1_round(r).reshape(w.shape)
    return q, sb, gs


# ---------------------------------------------------------------------------
# Layer shapes
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class LayerSpec:
    """Shape and numeric format of one MoE layer."""
    name: str
    hidden: int                 # H
    n_experts: int              # E
    top_k: int                  # k
    expert_ffn: int             # F
    latent: int = 0             # L (0: experts act on the hidden size)
    group_size: int = 64        # G
    shared_ffn: int = 0         # shared expert width (0: none)
    act: str = "swiglu"         # "swiglu" (gate+up) | "relu2" (up only)
    router: str = "softmax"     # "softmax" | "sigmoid"
    renormalize: bool = True
    routed_scale: float = 1.0
    router_bias: bool = False   # per-expert fp32 selection bias
    act_dtype: str = "bf16"     # x, out, latent projections, shared expert
    scale_dtype: str = "bf16"   # expert scale/bias
    router_dtype: str = "bf16"  # router weight
    weight_std: float = 0.02
    bias_std: float = 0.01
    bits: int = 4               # expert code width (2, 3, 4, 5, 6 or 8)
    fmt: str = "affine"         # "affine", "nvfp4" (group_size 16) or "mxfp4" (group_size 32)

    @property
    def k_in(self) -> int:
        """Input width of the routed experts (latent size or hidden)."""
        return self.latent if self.latent else self.hidden

    @property
    def gated(self) -> bool:
        return self.act == "swiglu"

    def with_(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


SPECS: Dict[str, LayerSpec] = {
    # tiny layer the oracle finishes in milliseconds
    "tiny": LayerSpec(name="tiny", hidden=512, n_experts=16, top_k=2, expert_ffn=256,
                      latent=0, group_size=64, shared_ffn=256, act="swiglu",
                      router="softmax", renormalize=True, routed_scale=1.0),
    # latent layer at the Bolt 74B-A9B shapes (E=496, k=9, latent 1024)
    "latent": LayerSpec(name="latent", hidden=4096, n_experts=496, top_k=9,
                        expert_ffn=1856, latent=1024, group_size=64, shared_ffn=3712,
                        act="relu2", router="sigmoid", renormalize=True,
                        routed_scale=2.5, router_bias=True),
    # non-latent sigmoid top-8 layer with fp16 activations and an fp32 router
    "nonlatent": LayerSpec(name="nonlatent", hidden=6144, n_experts=256, top_k=8,
                           expert_ffn=2048, latent=0, group_size=32, shared_ffn=2048,
                           act="swiglu", router="sigmoid", renormalize=True,
                           routed_scale=1.0, router_bias=False, act_dtype="fp16",
                           scale_dtype="fp16", router_dtype="fp32"),
}

STACK_EXPERTS = (240, 304, 368, 432, 496)


# Weight scale of the stacked layers.  A model puts a norm in front of every
# MoE layer; this layer has none, and with N(0, 0.02) weights the squared-ReLU
# shared expert grows the carried residual stream quadratically from layer to
# layer (RMS 1 -> 3 -> 30 -> 3e3 ...).  At 0.008 each layer adds a delta of
# RMS ~0.2 to a stream of RMS ~1, which stays bounded over the five layers.
STACK_WEIGHT_STD = 0.008


def stack_specs() -> List[LayerSpec]:
    """Five latent layers with the per-layer expert counts of the Bolt stack."""
    return [SPECS["latent"].with_(name=f"latent_e{e}", n_experts=e, weight_std=STACK_WEIGHT_STD)
            for e in STACK_EXPERTS]


def spec_for(name: str) -> LayerSpec:
    if name in SPECS:
        return SPECS[name]
    for s in stack_specs():
        if s.name == name:
            return s
    raise KeyError(name)


# ---------------------------------------------------------------------------
# Weights
# ---------------------------------------------------------------------------

@dataclass
class LayerWeights:
    """Storage-form weights of one layer (numpy, host)."""
    spec: LayerSpec
    router_w: np.ndarray                      # [E, H] router_dtype
    router_bias: Optional[np.ndarray]         # [E] float32 or None
    fc1: Optional[np.ndarray]                 # [L, H] act_dtype (latent only)
    fc2: Optional[np.ndarray]                 # [H, L] act_dtype (latent only)
    gate_q: Optional[np.ndarray]              # [E, F, Kin/8] uint32 (gated only)
    gate_s: Optional[np.ndarray]
    gate_b: Optional[np.ndarray]
    up_q: np.ndarray                          # [E, F, Kin/8]
    up_s: np.ndarray                          # [E, F, Kin/G]
    up_b: np.ndarray
    down_q: np.ndarray                        # [E, Kin, F/8]
    down_s: np.ndarray                        # [E, Kin, F/G]
    down_b: np.ndarray
    sh_gate: Optional[np.ndarray]             # [Fsh, H] act_dtype (gated only)
    sh_up: Optional[np.ndarray]               # [Fsh, H]
    sh_down: Optional[np.ndarray]             # [H, Fsh]
    seed: int = 0

    def arrays(self) -> Dict[str, np.ndarray]:
        out = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, np.ndarray):
                out[f.name] = v
        return out


def _dense(rng, shape, std, dtype):
    w = rng.standard_normal(size=shape, dtype=np.float32).astype(np.float64) * std
    return _round_to_dtype(w, dtype)


# Above this many elements per expert tensor, codes are drawn directly (see
# ``_quant_expert_direct``): drawing and quantising billions of normals on a
# host CPU takes minutes, while the kernels' cost does not depend on values.
EXACT_QUANT_MAX_ELEMS = 1 << 26


def _quant_expert_exact(rng, E, N, K, spec: LayerSpec):
    """Draw N(0, weight_std) weights and quantise them group by group."""
    q_all = np.empty((E, N, K), dtype=np.uint8)
    s_all = None
    b_all = None
    G = spec.group_size
    for e in range(E):
        w = rng.normal(0.0, spec.weight_std, size=(N, K))
        q, s, b = quantize_affine(w, G, spec.bits, spec.scale_dtype)
        if s_all is None:
            s_all = np.empty((E,) + s.shape, dtype=s.dtype)
            b_all = np.empty((E,) + b.shape, dtype=b.dtype)
        q_all[e], s_all[e], b_all[e] = q, s, b
    return pack_codes(q_all, spec.bits), s_all, b_all


def _quant_expert_direct(rng, E, N, K, spec: LayerSpec):
    """Draw packed codes uniformly (uniform bits: each code uniform on
    0..2^b-1) and per-group scale/bias so that the reconstructed weights have
    mean ~0 and standard deviation ~weight_std (a uniform b-bit code has std
    (2^b - 1)/sqrt(12) steps; 4.33 for b = 4)."""
    G = spec.group_size
    levels = (1 << spec.bits) - 1
    words = rng.integers(0, 1 << 32, size=(E, N, K * spec.bits // 32), dtype=np.uint32)
    step = spec.weight_std / (levels / np.sqrt(12.0))
    sg = np.abs(step * (1.0 + 0.1 * rng.standard_normal(size=(E, N, K // G))))
    bg = -0.5 * levels * sg + 0.1 * spec.weight_std * rng.standard_normal(size=(E, N, K // G))
    return words, _round_to_dtype(sg, spec.scale_dtype), _round_to_dtype(bg, spec.scale_dtype)


def _quant_expert_nvfp4(rng, E, N, K, spec: LayerSpec):
    """NVFP4 expert matrices: small layers draw N(0, weight_std) weights and
    quantise them (``quantize_nvfp4``); large ones draw uniform codes (each of
    the 16 E2M1 codes equally likely: RMS 2.93) with E4M3 block scales near 64
    and a matrix scale giving weights of standard deviation ~weight_std."""
    if N * K <= EXACT_QUANT_MAX_ELEMS // max(E, 1):
        q_all = np.empty((E, N, K), dtype=np.uint8)
        s_all = np.empty((E, N, K // 16), dtype=np.uint8)
        g_all = np.empty(E, dtype=np.float32)
        for e in range(E):
            q_all[e], s_all[e], g_all[e] = quantize_nvfp4(rng.normal(0.0, spec.weight_std, size=(N, K)))
        return pack_codes(q_all, 4), s_all, g_all
    words = rng.integers(0, 1 << 32, size=(E, N, K // 8), dtype=np.uint32)
    target = np.abs(64.0 * (1.0 + 0.1 * rng.standard_normal(size=(E, N, K // 16))))
    s_all, _ = e4m3_round(target)
    rms = float(np.sqrt(np.mean(_E2M1_GRID ** 2)))
    g_all = np.full(E, spec.weight_std / (rms * 64.0), dtype=np.float32)
    return words, s_all, g_all


def _quant_expert_mxfp4(rng, E, N, K, spec: LayerSpec):
    """MXFP4 expert matrices (no bias term: the third item is None): small
    layers quantise N(0, weight_std) weights (``quantize_mxfp4``); large ones
    draw uniform codes (RMS 2.93) with E8M0 scales within one binade of
    weight_std / 2.93."""
    if N * K <= EXACT_QUANT_MAX_ELEMS // max(E, 1):
        q_all = np.empty((E, N, K), dtype=np.uint8)
        s_all = np.empty((E, N, K // 32), dtype=np.uint8)
        for e in range(E):
            q_all[e], s_all[e] = quantize_mxfp4(rng.normal(0.0, spec.weight_std, size=(N, K)))
        return pack_codes(q_all, 4), s_all, None
    words = rng.integers(0, 1 << 32, size=(E, N, K // 8), dtype=np.uint32)
    rms = float(np.sqrt(np.mean(_E2M1_GRID ** 2)))
    e0 = int(np.rint(np.log2(spec.weight_std / rms)))
    s_all = (127 + e0 + rng.integers(-1, 1, size=(E, N, K // 32), endpoint=True)).astype(np.uint8)
    return words, s_all, None


def _quant_expert(rng, E, N, K, spec: LayerSpec):
    if spec.fmt == "nvfp4":
        return _quant_expert_nvfp4(rng, E, N, K, spec)
    if spec.fmt == "mxfp4":
        return _quant_expert_mxfp4(rng, E, N, K, spec)
    if N * K <= EXACT_QUANT_MAX_ELEMS // max(E, 1):
        return _quant_expert_exact(rng, E, N, K, spec)
    return _quant_expert_direct(rng, E, N, K, spec)


def make_layer(spec: LayerSpec, seed: int = 0, router_bias: Optional[np.ndarray] = None
               ) -> LayerWeights:
    """Draw one layer's weights from ``PCG64(seed)``.  Dense weights are
    N(0, weight_std) rounded to their storage dtype; router bias N(0, bias_std).
    Expert weights are N(0, weight_std) quantised group by group when the
    layer is small, and drawn directly as uniform codes with matching
    scale/bias statistics when it is large (``EXACT_QUANT_MAX_ELEMS``)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    H, E, F, Kin = spec.hidden, spec.n_experts, spec.expert_ffn, spec.k_in
    for dim, nm in ((H, "hidden"), (F, "expert_ffn"), (Kin, "k_in")):
        if dim % spec.group_size or dim % 8:
            raise ValueError(f"{nm}={dim} is not a multiple of the group size")
    router_w = _dense(rng, (E, H), spec.weight_std, spec.router_dtype)
    rb = None
    if spec.router_bias:
        rb = (rng.normal(0.0, spec.bias_std, size=E).astype(np.float32)
              if router_bias is None else np.asarray(router_bias, dtype=np.float32))
    fc1 = fc2 = None
    if spec.latent:
        fc1 = _dense(rng, (spec.latent, H), spec.weight_std, spec.act_dtype)
        fc2 = _dense(rng, (H, spec.latent), spec.weight_std, spec.act_dtype)
    gate = (None, None, None)
    if spec.gated:
        gate = _quant_expert(rng, E, F, Kin, spec)
    up = _quant_expert(rng, E, F, Kin, spec)
    down = _quant_expert(rng, E, Kin, F, spec)
    shg = shu = shd = None
    if spec.shared_ffn:
        Fs = spec.shared_ffn
        if spec.gated:
            shg = _dense(rng, (Fs, H), spec.weight_std, spec.act_dtype)
        shu = _dense(rng, (Fs, H), spec.weight_std, spec.act_dtype)
        shd = _dense(rng, (H, Fs), spec.weight_std, spec.act_dtype)
    return LayerWeights(spec=spec, router_w=router_w, router_bias=rb, fc1=fc1, fc2=fc2,
                        gate_q=gate[0], gate_s=gate[1], gate_b=gate[2],
                        up_q=up[0], up_s=up[1], up_b=up[2],
                        down_q=down[0], down_s=down[1], down_b=down[2],
                        sh_gate=shg, sh_up=shu, sh_down=shd, seed=seed)


def zipf_router_bias(n_experts: int, seed: int, s: float = 1.1, alpha: float = 0.1
                     ) -> np.ndarray:
    """Per-expert selection bias that skews expert load towards a Zipf(s) shape:
    experts get a random popularity rank r (1 = most popular) and bias
    ``-alpha * s * ln(r)``.  ``alpha`` sets how strongly the bias dominates the
    router scores; with the latent layer's sigmoid scores, alpha = 0.1 gives a
    per-rank load whose log-log slope over the 100 most popular experts is
    about -1.1 (k = 9 distinct picks per token cap the head of the curve).
    The realised load is measured by the benchmark, not assumed."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    rank = rng.permutation(n_experts) + 1
    return (-alpha * s * np.log(rank.astype(np.float64))).astype(np.float32)


# ---------------------------------------------------------------------------
# Activations
# ---------------------------------------------------------------------------

def draw_x_rows(spec: LayerSpec, n: int, rng: np.random.Generator) -> np.ndarray:
    """Draw ``n`` activation rows N(0,1) in the layer's activation storage dtype."""
    return _round_to_dtype(rng.normal(0.0, 1.0, size=(n, spec.hidden)), spec.act_dtype)


def make_x(spec: LayerSpec, T: int, seed: int = 0) -> np.ndarray:
    """``T`` activation rows from ``PCG64(seed)`` (no routing-margin filter)."""
    rng = np.random.Generator(np.random.PCG64(1_000_003 + seed))
    return draw_x_rows(spec, T, rng)


def ROUTED_BYTES(spec: LayerSpec) -> int:
    """Bytes of one routed expert: packed codes + scale + bias of all its matrices."""
    sb = 2 if spec.scale_dtype in ("bf16", "fp16") else 4
    n_mats_in = 2 if spec.gated else 1
    per_in = spec.expert_ffn * spec.k_in          # up (and gate) elements
    per_down = spec.k_in * spec.expert_ffn
    elems = n_mats_in * per_in + per_down
    return elems * spec.bits // 8 + 2 * sb * (elems // spec.group_size)
