"""Helpers shared by the GPU tests: margin-filtered inputs, running the CUDA
layer through the C ABI, and the parity gate against the oracle."""
from __future__ import annotations

import functools

import numpy as np

import moe_inputs as mi
import oracle

# Parity bounds: expert set identical; output relative RMS error <= 1e-2 and
# max abs error <= 3e-2 * RMS(reference); the same bounds on the layer's delta
# (out - x) so the residual cannot hide an error in the routed or shared part.
REL_RMS = 1e-2
MAX_ABS_FRAC = 3e-2
# Routing weights: fp32 against fp64.  The fp32 logit of an H-long dot product
# carries a relative error of about sqrt(H) * 2^-24 (4e-6 of its scale at
# H = 4096-6144); the sigmoid's slope is at most 1/4, and the normalisation
# and the routed scale add a few fp32 ulps (1.2e-7 each) on weights of order 1.
W_RTOL, W_ATOL = 1e-5, 1e-6
MIN_MARGIN = 1e-3

_CACHES = {}


def ora_forward(layer, x):
    """The oracle with a dequantised-expert cache kept per layer (test speed)."""
    c = _CACHES.get(id(layer))
    if c is None or c.layer is not layer:
        c = _CACHES[id(layer)] = oracle.expert_cache(layer)
    return oracle.oracle_forward(layer, x, cache=c)


def margin_x(layer, T: int, seed: int = 0, min_margin: float = MIN_MARGIN, stack=None):
    """T rows drawn from a seeded stream, keeping only rows whose gap between
    the k-th and (k+1)-th oracle selection key is >= min_margin (at every
    layer of ``stack`` when given, following the oracle's own residual
    stream).  Returns (x, redraws)."""
    spec = layer.spec
    rng = np.random.Generator(np.random.PCG64(2_000_003 + seed))
    layers = stack if stack is not None else [layer]
    routers = [(oracle.widen(l.router_w, l.spec.router_dtype),
                None if l.router_bias is None else l.router_bias.astype(np.float64)) for l in layers]
    rows, redraws = [], 0
    while len(rows) < T:
        cand = mi.draw_x_rows(spec, 8, rng)
        for i in range(cand.shape[0]):
            row = cand[i:i + 1]
            ok = True
            cur = row
            for li, lay in enumerate(layers):
                sp = lay.spec
                Wr, bias = routers[li]
                z = Wr @ oracle.widen(cur, sp.act_dtype)[0]
                if not oracle.routing_margin(z, sp, bias) >= min_margin:   # NaN fails too
                    ok = False
                    break
                if li + 1 < len(layers):
                    nxt = ora_forward(lay, cur)["out"]
                    cur = mi._round_to_dtype(nxt, sp.act_dtype)
            if ok:
                rows.append(row[0])
                if len(rows) == T:
                    break
            else:
                redraws += 1
    return np.stack(rows), redraws


def to_torch_x(x: np.ndarray, act_dtype: str):
    import torch
    if act_dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def build_layer(layer, max_tokens: int):
    import quantized_moe_decode_gemv_gb300 as pkg
    cfg = pkg.MoEConfig.from_spec(layer.spec, max_tokens=max_tokens)
    dev = pkg.upload_arrays(layer.arrays())
    h = pkg.MoELayer(cfg, dev)
    del dev
    return h


def run_layer(h, x: np.ndarray, act_dtype: str):
    import torch
    xt = to_torch_x(x, act_dtype)
    out, ids, w, delta = h.forward_ex(xt)
    torch.cuda.synchronize()
    return {"out": out.float().cpu().numpy().astype(np.float64), "ids": ids.cpu().numpy(),
            "w": w.cpu().numpy().astype(np.float64), "delta": delta.cpu().numpy().astype(np.float64),
            "out_raw": out}


def rel_rms(got, ref):
    return float(np.sqrt(np.mean((got - ref) ** 2)) / max(1e-300, np.sqrt(np.mean(ref ** 2))))


def max_abs_frac(got, ref):
    return float(np.max(np.abs(got - ref)) / max(1e-300, np.sqrt(np.mean(ref ** 2))))


def check_parity(got: dict, ref: dict, rows=None, what=""):
    """The parity gate.  ``rows`` selects the GPU rows that ``ref`` covers."""
    sel = slice(None) if rows is None else list(rows)
    g_ids, g_w = got["ids"][sel], got["w"][sel]
    g_out, g_delta = got["out"][sel], got["delta"][sel]
    assert np.array_equal(g_ids, ref["ids"]), f"{what}: selected experts differ\n{g_ids}\n{ref['ids']}"
    np.testing.assert_allclose(g_w, ref["w"], rtol=W_RTOL, atol=W_ATOL, err_msg=what)
    for name, g, r in (("out", g_out, ref["out"]), ("delta", g_delta, ref["delta"])):
        rr, ma = rel_rms(g, r), max_abs_frac(g, r)
        assert rr <= REL_RMS, f"{what}: {name} rel-RMS {rr:.3e}"
        assert ma <= MAX_ABS_FRAC, f"{what}: {name} max-abs/RMS {ma:.3e}"
    return rel_rms(g_out, ref["out"]), rel_rms(g_delta, ref["delta"])


@functools.lru_cache(maxsize=None)
def cached_layer_spec(spec, seed: int = 0):
    """A layer of any spec (LayerSpec is frozen and hashable), built once."""
    return mi.make_layer(spec, seed)


@functools.lru_cache(maxsize=None)
def cached_layer(name: str, seed: int = 0, zipf: bool = False):
    spec = mi.spec_for(name)
    rb = mi.zipf_router_bias(spec.n_experts, seed) if zipf else None
    return mi.make_layer(spec, seed, router_bias=rb)
