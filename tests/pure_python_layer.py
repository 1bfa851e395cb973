"""Brute-force pure-Python forward of a *tiny* MoE layer, used to pin the oracle.

Written independently of ``oracle/``: plain Python ints and floats, explicit
loops, its own storage decoding (struct for bf16 bits, shifts for codes), a
selection by exhaustive search over all k-subsets, and exact-order sums.  It is
only meant for layers with a handful of experts and rows of a few dozen
elements.
"""
from __future__ import annotations

import itertools
import math
import struct


def _bf16(u):
    return struct.unpack("<f", struct.pack("<I", int(u) << 16))[0]


def _val(a, dtype):
    if dtype == "bf16":
        return _bf16(a)
    return float(a)


def _matrix(arr, dtype):
    return [[_val(v, dtype) for v in row] for row in arr.tolist()] if dtype != "bf16" else \
        [[_bf16(v) for v in row] for row in arr.tolist()]


def _deq(words, scale, bias, G, sdt, bits=4):
    """One expert matrix: words [N][K*bits/32] -> [N][K] floats.  The row's
    words are one integer, word w at bit 32*w; code i is bits bits*i.. of it."""
    rows = []
    for n, wrow in enumerate(words.tolist()):
        big = 0
        for w_i, w in enumerate(wrow):
            big |= int(w) << (32 * w_i)
        K = 32 * len(wrow) // bits
        codes = [(big >> (bits * i)) & ((1 << bits) - 1) for i in range(K)]
        srow = scale[n].tolist()
        brow = bias[n].tolist()
        rows.append([_val(srow[kk // G], sdt) * codes[kk] + _val(brow[kk // G], sdt)
                     for kk in range(len(codes))])
    return rows


def _mv(M, v):
    out = []
    for row in M:
        acc = 0.0
        for a, b in zip(row, v):
            acc += a * b
        out.append(acc)
    return out


def _act(act, u, g):
    if act == "swiglu":
        return [(gi / (1.0 + math.exp(-gi))) * ui for ui, gi in zip(u, g)]
    return [max(ui, 0.0) ** 2 for ui in u]


def _select(keys, k):
    """Exhaustive: the k-subset with the largest key sum; order inside it by key
    descending then index.  Keys must be finite and distinct enough."""
    best, best_sum = None, -math.inf
    for comb in itertools.combinations(range(len(keys)), k):
        s = sum(keys[i] for i in comb)
        if s > best_sum:
            best, best_sum = comb, s
    return sorted(best, key=lambda i: (-keys[i], i))


def forward(layer, x):
    """Returns (out rows, ids rows, weight rows) as Python lists."""
    sp = layer.spec
    adt, rdt, sdt, G = sp.act_dtype, sp.router_dtype, sp.scale_dtype, sp.group_size
    Wr = _matrix(layer.router_w, rdt)
    bias = [float(b) for b in layer.router_bias] if layer.router_bias is not None else None
    W1 = _matrix(layer.fc1, adt) if sp.latent else None
    W2 = _matrix(layer.fc2, adt) if sp.latent else None
    experts = []
    for e in range(sp.n_experts):
        nb = getattr(sp, "bits", 4)
        up = _deq(layer.up_q[e], layer.up_s[e], layer.up_b[e], G, sdt, nb)
        gate = _deq(layer.gate_q[e], layer.gate_s[e], layer.gate_b[e], G, sdt, nb) if sp.gated else None
        down = _deq(layer.down_q[e], layer.down_s[e], layer.down_b[e], G, sdt, nb)
        experts.append((gate, up, down))
    if sp.shared_ffn:
        shu = _matrix(layer.sh_up, adt)
        shg = _matrix(layer.sh_gate, adt) if sp.gated else None
        shd = _matrix(layer.sh_down, adt)
    outs, ids_all, w_all = [], [], []
    for row in x.tolist() if adt != "bf16" else x.tolist():
        xr = [_val(v, adt) for v in row]
        z = _mv(Wr, xr)
        if sp.router == "softmax":
            keys = z
        else:
            sg = [1.0 / (1.0 + math.exp(-zi)) for zi in z]
            keys = [sg[i] + (bias[i] if bias else 0.0) for i in range(len(z))]
        ids = _select(keys, sp.top_k)
        if sp.router == "softmax":
            num = [math.exp(z[i]) for i in ids]
            den = sum(num) if sp.renormalize else sum(math.exp(zi) for zi in z)
            w = [v / den for v in num]
        else:
            num = [sg[i] for i in ids]
            den = sum(num) if sp.renormalize else 1.0
            w = [v / den for v in num]
        w = [v * sp.routed_scale for v in w]
        xin = _mv(W1, xr) if sp.latent else xr
        y = [0.0] * len(xin)
        for j, e in enumerate(ids):
            gate, up, down = experts[e]
            u = _mv(up, xin)
            g = _mv(gate, xin) if gate is not None else None
            yj = _mv(down, _act(sp.act, u, g))
            y = [a + w[j] * b for a, b in zip(y, yj)]
        r = _mv(W2, y) if sp.latent else y
        s = [0.0] * len(xr)
        if sp.shared_ffn:
            su = _mv(shu, xr)
            sgt = _mv(shg, xr) if shg is not None else None
            s = _mv(shd, _act(sp.act, su, sgt))
        outs.append([a + b + c for a, b, c in zip(xr, r, s)])
        ids_all.append(list(ids))
        w_all.append(w)
    return outs, ids_all, w_all
