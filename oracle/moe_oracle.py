"""fp64 CPU oracle for the decode-time forward of a routed MoE layer with b-bit
(2, 3, 4, 5, 6 or 8) affine group-quantised experts, or NVFP4 / MXFP4 experts.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only the
tests, the smoke check and the benchmark's CPU-baseline leg call it.  It shares
no code with the CUDA path: it decodes the storage formats itself (bf16 bits,
packed codes), and every step is the plain definition written out in float64,
one token row at a time, with no blocking, fusion or reordering.

Sources (page titles and sections):

* TensorFold PR #1038 (native Metal backend for Nemotron 3.5 Bolt 74B-A9B),
  "What's in it": the latent MoE runs in the order gate gemv -> route top-k ->
  fc1_latent_proj -> routed experts -> combine rows -> fc2_latent_proj ->
  + shared -> + residual, with routed experts in the 1024-wide latent.
* TensorFold PR #1295 (Muse Spark Open on two GB10s), "What this changes" and
  "Checklist": an fp32 router with sigmoid top-8 and a per-expert
  normalisation and sum; fp16 activations with fp32 sums.
* mlx-bun decode-speed program, weight-format table and the affine shared-M
  section: MLX affine quantisation, packed codes of 2..8 bits with a scale
  and a bias per group (group sizes 32/64/128); the same table lists
  "mxfp4/nvfp4" among the supported formats.

Where the pages leave a step open, the readings are:

1. affine dequantisation is ``w = scale * q + bias`` with unsigned b-bit codes
   ``q in 0..2^b-1`` (b = 2, 3, 4, 5, 6 or 8) and groups of G consecutive elements
   along the input axis;
2. packed storage: the codes of a row as one little-endian bit stream of
   uint32 words (for b = 4: eight codes per word, lowest nibble first);
3. the router bias only steers *selection* (key = sigmoid(z) + bias); the
   combine weights use sigmoid(z) without it;
4. weights are normalised over the selected set first, then multiplied by the
   routed scale;
5. top-k order: larger key first; equal keys: lower expert index first;
   non-finite keys rank below every finite key (in index order);
6. softmax routing with renormalisation equals a softmax over the selected
   logits; without renormalisation the weights are the full softmax;
7. the shared expert has the routed experts' activation form and weight 1;
8. the residual is the layer input; the layer has no norm;
9. NVFP4 (named, not defined, by the pages): 4-bit E2M1 codes (sign bit 3,
   exponent bits 2..1 with bias 1, mantissa bit 0; exponent 0 is subnormal)
   with one E4M3 scale (sign bit 7, exponent bits 6..3 with bias 7, mantissa
   bits 2..0; exponent 0 subnormal; exponent 15 with mantissa 7 is NaN) per
   16 consecutive elements along the input axis and one fp32 scale per
   expert matrix: w = e2m1(q) * e4m3(s) * matrix scale (the OCP
   Microscaling specification's FP4 E2M1 and FP8 E4M3 element types);
10. MXFP4 (named with NVFP4 by the same table): the same E2M1 codes with one
   E8M0 scale (the power of two 2^(byte - 127); 0xFF is NaN) per 32
   consecutive elements along the input axis and no other term:
   w = e2m1(q) * 2^(s - 127) (the OCP Microscaling specification's MXFP4).

Every function here is pinned by tests that do not reuse its formulas
(brute-force top-k, closed forms, invariants, a pure-Python loop).
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np

__all__ = [
    "widen", "unpack_codes", "dequantize", "e2m1_values", "e4m3_values", "dequantize_nvfp4",
    "e8m0_values", "dequantize_mxfp4",
    "router_logits", "selection_keys",
    "topk_order", "route", "activation", "expert_output", "shared_output",
    "oracle_forward", "routing_margin", "forward_rows", "expert_cache",
]


# ---------------------------------------------------------------------------
# storage decoding
# ---------------------------------------------------------------------------

def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array -> float64.  bf16 arrives as uint16 bit patterns: the
    value is the float32 whose upper 16 bits are the pattern."""
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype in ("fp16", "fp32"):
        return np.asarray(a).astype(np.float64)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def unpack_codes(packed: np.ndarray, bits: int = 4) -> np.ndarray:
    """uint32 words -> b-bit codes.  The words of a row are one little-endian
    bit stream (bit j of word w is stream bit 32*w + j) and code ``i`` is the
    unsigned integer in stream bits ``b*i .. b*i+b-1``, lowest bit first
    (reading 2: for b = 4, element ``8*w + i`` in bits ``4*i``)."""
    p = np.ascontiguousarray(np.asarray(packed, dtype="<u4"))
    stream = np.unpackbits(p.view(np.uint8), axis=-1, bitorder="little")
    n = stream.shape[-1] // bits
    digits = stream[..., : n * bits].reshape(*p.shape[:-1], n, bits).astype(np.int64)
    return (digits << np.arange(bits, dtype=np.int64)).sum(axis=-1)


def dequantize(packed: np.ndarray, scale: np.ndarray, bias: np.ndarray, group: int,
               scale_dtype: str, bits: int = 4) -> np.ndarray:
    """Affine b-bit dequantisation ``w[n, k] = scale[n, k // G] * q[n, k] +
    bias[n, k // G]`` in float64 (mlx-bun decode-speed program, affine
    weight formats of 2..8 bits; reading 1)."""
    q = unpack_codes(packed, bits).astype(np.float64)
    s = widen(scale, scale_dtype)
    b = widen(bias, scale_dtype)
    K = q.shape[-1]
    if s.shape[-1] * group != K:
        raise ValueError("scale shape does not match the group size")
    s_full = np.repeat(s, group, axis=-1)
    b_full = np.repeat(b, group, axis=-1)
    return s_full * q + b_full


def e2m1_values(codes: np.ndarray) -> np.ndarray:
    """Values of 4-bit E2M1 codes (reading 9): sign bit 3; exponent field
    bits 2..1 (bias 1); mantissa bit 0; exponent field 0 is subnormal
    (0.5 * mantissa)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = (c >> 3) & 1
    ef = (c >> 2 & 1) * 2 + (c >> 1 & 1)
    mf = c & 1
    mag = np.where(ef == 0, 0.5 * mf, np.exp2(ef - 1.0) * (1.0 + 0.5 * mf))
    return np.where(sign == 1, -mag, mag)


def e4m3_values(b: np.ndarray) -> np.ndarray:
    """Values of E4M3 bytes (reading 9): sign bit 7; exponent field bits 6..3
    (bias 7); mantissa bits 2..0; exponent field 0 is subnormal (m/8 * 2^-6);
    exponent 15 with mantissa 7 is NaN (there is no infinity)."""
    v = np.asarray(b, dtype=np.int64)
    sign = (v >> 7) & 1
    ef = (v >> 3) & 15
    mf = v & 7
    mag = np.where(ef == 0, (mf / 8.0) * 2.0 ** -6, (1.0 + mf / 8.0) * np.exp2(ef - 7.0))
    mag = np.where((ef == 15) & (mf == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def dequantize_nvfp4(packed: np.ndarray, scale_bytes: np.ndarray, matrix_scale) -> np.ndarray:
    """NVFP4 dequantisation ``w[n, k] = e2m1(q[n, k]) * e4m3(s[n, k // 16]) *
    matrix_scale`` in float64 (reading 9)."""
    q = e2m1_values(unpack_codes(packed, 4))
    s = e4m3_values(scale_bytes)
    if s.shape[-1] * 16 != q.shape[-1]:
        raise ValueError("NVFP4 scales do not match blocks of 16")
    return q * np.repeat(s, 16, axis=-1) * float(np.float32(matrix_scale))


def e8m0_values(b: np.ndarray) -> np.ndarray:
    """Values of E8M0 bytes (reading 10): 2^(b - 127); 0xFF is NaN."""
    v = np.asarray(b, dtype=np.int64)
    return np.where(v == 255, np.nan, np.exp2(v - 127.0))


def dequantize_mxfp4(packed: np.ndarray, scale_bytes: np.ndarray) -> np.ndarray:
    """MXFP4 dequantisation ``w[n, k] = e2m1(q[n, k]) * e8m0(s[n, k // 32])`` in
    float64 (reading 10)."""
    q = e2m1_values(unpack_codes(packed, 4))
    s = e8m0_values(scale_bytes)
    if s.shape[-1] * 32 != q.shape[-1]:
        raise ValueError("MXFP4 scales do not match blocks of 32")
    return q * np.repeat(s, 32, axis=-1)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def router_logits(x_row: np.ndarray, router_w: np.ndarray) -> np.ndarray:
    """Router ("gate") gemv: ``z[e] = sum_h Wr[e, h] * x[h]`` in float64
    (TensorFold #1038, gate gemv; TensorFold #1295, fp32 router)."""
    return router_w @ x_row


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def selection_keys(z: np.ndarray, spec, bias: Optional[np.ndarray]) -> np.ndarray:
    """Key that ranks experts: the logit for softmax routing; sigmoid(z) plus
    the per-expert selection bias for sigmoid routing (reading 3)."""
    if spec.router == "softmax":
        return np.asarray(z, dtype=np.float64)
    s = _sigmoid(np.asarray(z, dtype=np.float64))
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float64)
    return s


def topk_order(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys, larger first, ties to the lower index,
    non-finite keys after every finite one (reading 5).  A plain sort on the
    tuple (finite?, key, -index)."""
    keys = np.asarray(keys, dtype=np.float64)
    order = sorted(range(len(keys)),
                   key=lambda e: (0, -keys[e], e) if math.isfinite(keys[e]) else (1, 0.0, e))
    return np.array(order[:k], dtype=np.int64)


def route(z: np.ndarray, spec, bias: Optional[np.ndarray]):
    """Top-k expert ids and combine weights for one row.

    Softmax: weights ``exp(z_j) / sum_{i in S} exp(z_i)`` with renormalisation,
    else the full softmax at the selected ids (reading 6).
    Sigmoid: ``s_j = sigmoid(z_j)`` (bias excluded), divided by the sum over
    the selected set when normalising, then times the routed scale
    (TensorFold #1295, sigmoid top-8 with a per-expert norm and sum;
    readings 3-4)."""
    z = np.asarray(z, dtype=np.float64)
    keys = selection_keys(z, spec, bias)
    ids = topk_order(keys, spec.top_k)
    if spec.router == "softmax":
        m = np.max(z[np.isfinite(z)]) if np.any(np.isfinite(z)) else 0.0
        ez = np.exp(z - m)
        denom = ez[ids].sum() if spec.renormalize else ez.sum()
        w = ez[ids] / denom
    else:
        s = _sigmoid(z)
        w = s[ids]
        if spec.renormalize:
            w = w / w.sum()
    w = w * float(spec.routed_scale)
    return ids, w


def routing_margin(z: np.ndarray, spec, bias: Optional[np.ndarray]) -> float:
    """Gap between the k-th and (k+1)-th selection key of one row, in the
    selection order of ``topk_order`` (non-finite keys rank last and count as
    -inf); inf if k = E or the (k+1)-th key is non-finite."""
    keys = selection_keys(z, spec, bias)
    k = spec.top_k
    if k >= len(keys):
        return math.inf
    ranked = np.where(np.isfinite(keys), keys, -np.inf)
    srt = np.sort(ranked)[::-1]
    if srt[k] == -np.inf:
        return math.inf if srt[k - 1] > -np.inf else 0.0
    return float(srt[k - 1] - srt[k])


# ---------------------------------------------------------------------------
# expert MLPs
# ---------------------------------------------------------------------------

def activation(spec, u: np.ndarray, g: Optional[np.ndarray]) -> np.ndarray:
    """SwiGLU ``silu(g) * u`` with ``silu(g) = g / (1 + exp(-g))``, or the
    non-gated squared ReLU ``max(u, 0)**2``."""
    if spec.act == "swiglu":
        return (g / (1.0 + np.exp(-g))) * u
    if spec.act == "relu2":
        r = np.maximum(u, 0.0)
        return r * r
    raise ValueError(spec.act)


class _ExpertCache:
    """Dequantises each selected expert once per forward call (only selected
    experts are ever dequantised).  When shared across calls it keeps at most
    ``max_bytes`` of dequantised matrices, evicting the oldest first."""

    def __init__(self, layer, max_bytes: int = 4 << 30):
        self.layer = layer
        self.spec = layer.spec
        self.mats: Dict[int, tuple] = {}
        self.max_bytes = max_bytes
        self.bytes = 0

    def get(self, e: int):
        if e not in self.mats:
            L, sp = self.layer, self.spec
            G, sd, nb = sp.group_size, sp.scale_dtype, getattr(sp, "bits", 4)
            if getattr(sp, "fmt", "affine") == "mxfp4":
                up = dequantize_mxfp4(L.up_q[e], L.up_s[e])
                gate = dequantize_mxfp4(L.gate_q[e], L.gate_s[e]) if sp.gated else None
                down = dequantize_mxfp4(L.down_q[e], L.down_s[e])
            elif getattr(sp, "fmt", "affine") == "nvfp4":
                up = dequantize_nvfp4(L.up_q[e], L.up_s[e], L.up_b[e])
                gate = dequantize_nvfp4(L.gate_q[e], L.gate_s[e], L.gate_b[e]) if sp.gated else None
                down = dequantize_nvfp4(L.down_q[e], L.down_s[e], L.down_b[e])
            else:
                up = dequantize(L.up_q[e], L.up_s[e], L.up_b[e], G, sd, nb)
                gate = dequantize(L.gate_q[e], L.gate_s[e], L.gate_b[e], G, sd, nb) if sp.gated else None
                down = dequantize(L.down_q[e], L.down_s[e], L.down_b[e], G, sd, nb)
            size = up.nbytes + down.nbytes + (gate.nbytes if gate is not None else 0)
            while self.mats and self.bytes + size > self.max_bytes:
                old = next(iter(self.mats))
                self.bytes -= sum(m.nbytes for m in self.mats.pop(old) if m is not None)
            self.mats[e] = (gate, up, down)
            self.bytes += size
        return self.mats[e]


def expert_cache(layer) -> _ExpertCache:
    """A dequantised-expert cache that several ``oracle_forward`` calls on the
    same layer may share (it only avoids repeating identical dequantisation)."""
    return _ExpertCache(layer)


def expert_output(cache: _ExpertCache, e: int, xin: np.ndarray) -> np.ndarray:
    """One routed expert on one row: ``down @ act(up @ xin [, gate @ xin])``."""
    gate, up, down = cache.get(e)
    u = up @ xin
    g = gate @ xin if gate is not None else None
    h = activation(cache.spec, u, g)
    return down @ h


def shared_output(layer, x_row: np.ndarray) -> np.ndarray:
    """The dense shared expert on the hidden row, same activation form as the
    routed experts (reading 7)."""
    sp = layer.spec
    if not sp.shared_ffn:
        return np.zeros(sp.hidden)
    dt = sp.act_dtype
    u = widen(layer.sh_up, dt) @ x_row
    g = widen(layer.sh_gate, dt) @ x_row if sp.gated else None
    h = activation(sp, u, g)
    return widen(layer.sh_down, dt) @ h


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------

def oracle_forward(layer, x: np.ndarray, cache: Optional[_ExpertCache] = None) -> dict:
    """Forward of the whole layer on ``x [T, H]`` (storage dtype), row by row,
    in the Bolt layer order (TensorFold #1038, "What's in it"):

    router gemv -> route top-k -> fc1_latent_proj (latent layers) -> selected
    experts -> weighted combine -> fc2_latent_proj (latent layers) -> + shared
    expert -> + residual.

    Returns float64 ``out [T, H]``, ``delta = out - x``, ``ids [T, k]``,
    ``w [T, k]``, the combined routed output ``y [T, Kin]`` and the router
    logits ``z [T, E]``."""
    sp = layer.spec
    xs = widen(x, sp.act_dtype)
    T = xs.shape[0]
    Wr = widen(layer.router_w, sp.router_dtype)
    bias = None if layer.router_bias is None else np.asarray(layer.router_bias, np.float64)
    W1 = widen(layer.fc1, sp.act_dtype) if sp.latent else None
    W2 = widen(layer.fc2, sp.act_dtype) if sp.latent else None
    if cache is None or cache.layer is not layer:
        cache = _ExpertCache(layer)
    k, Kin = sp.top_k, sp.k_in
    out = np.zeros((T, sp.hidden))
    ids_all = np.zeros((T, k), dtype=np.int64)
    w_all = np.zeros((T, k))
    y_all = np.zeros((T, Kin))
    z_all = np.zeros((T, sp.n_experts))
    for t in range(T):
        xt = xs[t]
        z = router_logits(xt, Wr)
        ids, w = route(z, sp, bias)
        xin = W1 @ xt if sp.latent else xt
        y = np.zeros(Kin)
        for j in range(k):
            y = y + w[j] * expert_output(cache, int(ids[j]), xin)
        r = W2 @ y if sp.latent else y
        out[t] = xt + r + shared_output(layer, xt)
        ids_all[t], w_all[t], y_all[t], z_all[t] = ids, w, y, z
    return {"out": out, "delta": out - xs, "ids": ids_all, "w": w_all,
            "y": y_all, "z": z_all}


def forward_rows(layer, x: np.ndarray, rows: Sequence[int]) -> dict:
    """The oracle on a subset of rows (each row is independent)."""
    return oracle_forward(layer, np.asarray(x)[list(rows)])
