#!/usr/bin/env python
"""MoE-layer decode benchmark on one GB300 (or N independent replicas).

Headline workload: the latent MoE layer at the Bolt 74B-A9B shapes (H=4096,
latent L=1024, E=496 routed experts, top-k=9 sigmoid router with fp32 bias and
normalised weights x2.5, experts F=1856 squared-ReLU int4 affine group 64 with
bf16 scale/bias, bf16 shared expert F=3712), decoding T=1 token row per step.
Inputs are seeded synthetic data resident in HBM; 32 distinct token batches
are cycled so the selected experts change, and L2 is flushed before every
timed step.

Alongside (``also``), every other configured workload is measured the same way:
the latent layer at T=16; the non-latent sigmoid top-8 layer (H=6144, E=256,
SwiGLU F=2048 int4 g32 fp16) at T=1/4/32; the five-layer heterogeneous stack
(E=240..496) at T=2/9/16, layers run round-robin with the residual carried;
the batched-serving sweep of the latent layer with Zipf(1.1)-skewed expert load
at T=64/256 (grouped tcgen05 path, with tensor-pipe throughput); and the tiny
layer at T=1/4.

Prints ONE JSON line: tokens/s (``value``), achieved HBM GB/s over the
algorithmic bytes, the roofline of the dominant kernel, the end-to-end number
through the host-buffer C-ABI call, and the fp64 CPU oracle timed on the host.
``--impl reference`` times that oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s and achieved HBM GB/s (% of GB300 peak) at T=1/16"
WORKLOAD = ("latent MoE layer, Bolt-like shape: H=4096, fc1/fc2 latent L=1024, E=496, "
            "top-k=9 sigmoid+bias, normalised x2.5, F=1856 relu^2 int4 affine g64 bf16 "
            "scale/bias, shared F=3712 bf16")
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Leaves L2 cold for the next step: writes a 256 MB buffer (twice the L2)
    and then reads another 256 MB buffer, so that L2 holds clean, unrelated
    lines -- the state a decode step finds after other layers' weight reads --
    rather than 126 MB of dirty lines whose write-back the timed step would
    pay for."""

    def __init__(self, torch, device):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def zero_(self):
        self.w.zero_()
        self.r.sum()
STAGES = ["dense_in", "route", "expert_up", "expert_down", "dense_out"]
# the kernels of the gemv path's stages (bf16 layers with 4-bit experts: the
# warp-MMA dense and expert kernels at every batch size; the routing rides in
# the first dense pass)
KERNEL_OF_STAGE = {"dense_in": "k_dense_mma", "route": "k_dense_mma", "expert_up": "k_expert_mma",
                   "expert_down": "k_expert_mma", "dense_out": "k_dense_mma"}
# the grouped path runs every projection through the tcgen05 GEMM (its split-K
# sums and the combine ride in the same stages)
KERNEL_OF_STAGE_GROUPED = {"dense_in": "k_umma2", "route": "k_route", "expert_up": "k_umma2",
                           "expert_down": "k_umma2", "dense_out": "k_umma2"}


# the sources that define each kernel and its launch
KERNEL_SOURCES = {
    "k_dense_in": ["moe_kernels.cuh", "moe_layer.cu"],
    "k_dense_out": ["moe_kernels.cuh", "moe_layer.cu"],
    # the expert gemv kernel: its device code and the host code that launches it
    "k_expert": ["moe_kernels.cuh", "moe_layer.cu:expert_gemv_launch"],
    "k_route": ["moe_kernels.cuh", "moe_layer.cu"],
    "k_umma": ["moe_kernels.cuh", "moe_umma.cuh", "moe_layer.cu"],
    "k_umma2": ["moe_kernels.cuh", "moe_umma.cuh", "moe_umma2.cuh", "moe_layer.cu"],
    "k_expert_bulk": ["moe_kernels.cuh", "moe_expert_bulk.cuh", "moe_layer.cu"],
    "k_expert_mma": ["moe_kernels.cuh", "moe_expert_bulk.cuh", "moe_expert_mma.cuh", "moe_layer.cu"],
    "k_dense_mma": ["moe_kernels.cuh", "moe_expert_bulk.cuh", "moe_expert_mma.cuh", "moe_dense_mma.cuh",
                    "moe_layer.cu"],
    "k_dense_bulk": ["moe_kernels.cuh", "moe_expert_bulk.cuh", "moe_dense_bulk.cuh", "moe_layer.cu"],
}


def _code_only(text):
    """C/C++ source without its comments and blank lines (string literals kept)."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                   # string literal
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def _braced(text, start):
    """text from `start` through the brace that closes the first "{" after it."""
    i = text.index("{", start)
    depth = 0
    for j in range(i, len(text)):
        depth += {"{": 1, "}": -1}.get(text[j], 0)
        if depth == 0:
            return text[start:j + 1]
    raise ValueError("unbalanced braces")


def _expert_gemv_launch(code):
    """The host code that configures and launches the expert gemv kernel: its
    launch helpers, the token-slot and grid sizing statements and the two
    launch blocks of the forward."""
    import re
    parts = []
    for fn in ("expert_pb_cap", "pow2_at_least", "launch_ex", "launch_expert_t", "launch_expert"):
        m = re.search(r"^static [^\n(]*\b" + fn + r"\(", code, flags=re.M)
        parts.append(_braced(code, m.start()))
    for var in ("pb_split", "pb_up", "pb_dn", "slots", "target"):
        i = code.index("const int " + var + " =")
        parts.append(code[i:code.index(";", i) + 1])
    for m in re.finditer(r"if \(experts_gemv\) \{", code):
        parts.append(_braced(code, m.start()))
    return "\n".join(parts)


SOURCE_PARTS = {"expert_gemv_launch": _expert_gemv_launch}


def kernel_source_hash(kernel):
    """sha256 over the code (comments stripped) of a kernel's CUDA sources --
    whole files, or the named part of a file ("file:part") -- so that DRAM
    traffic captured by ncu is only reported for the code it was captured from."""
    import hashlib
    d = os.path.join(ROOT, "quantized_moe_decode_gemv_gb300", "csrc")
    h = hashlib.sha256()
    for entry in KERNEL_SOURCES.get(kernel, sorted(os.listdir(d))):
        name, _, part = entry.partition(":")
        with open(os.path.join(d, name), encoding="utf-8") as f:
            code = _code_only(f.read())
        if part:
            code = SOURCE_PARTS[part](code)
        h.update(entry.encode() + b"\0" + code.encode())
    return h.hexdigest()


def captured_traffic(kernel, T, zipf=False):
    """DRAM bytes (read + write) per launch of a kernel from the committed ncu
    summary profiles/traffic.json, or None when there is none for this kernel,
    T and load (uniform, or Zipf-skewed: key suffix "z") or the kernels changed
    since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get("kernels", {}).get(f"{kernel}@T{T}{'z' if zipf else ''}")
    if not d or d.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return float(d["dram_bytes_per_launch"])


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--T", type=int, default=1, help="token rows per step")
    p.add_argument("--also-T", type=int, default=16, help="second T reported alongside (0: off)")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--path", choices=["auto", "gemv", "grouped"], default="auto",
                   help="kernel schedule (A/B); auto: the gemv path below 16 rows, the grouped "
                        "tcgen05 path from 16")
    p.add_argument("--config", choices=["latent", "nonlatent", "tiny"], default="latent",
                   help="layer of the main line (the headline metric is the latent layer at T=1)")
    p.add_argument("--fmt", choices=["affine", "nvfp4", "mxfp4"], default="affine",
                   help="expert weight format of the main line's layer (nvfp4: blocks of 16, "
                        "mxfp4: blocks of 32)")
    p.add_argument("--no-also", action="store_true", help="skip the other configured workloads")
    p.add_argument("--zipf", action="store_true", help="Zipf-skewed expert load (batched sweep)")
    p.add_argument("--sweep", default="", help="comma-separated T values: time each and write "
                   "one JSON line per T to --sweep-out (the main line is unchanged)")
    p.add_argument("--sweep-out", default="sweep.jsonl")
    return p.parse_args()


# ---------------------------------------------------------------------------
# byte accounting (algorithmic bytes: what the method must move)
# ---------------------------------------------------------------------------

def expert_bytes(spec):
    """(up-side bytes, down-side bytes) of one routed expert: packed b-bit codes
    + scale + bias (2 bytes each per group); NVFP4: 4-bit codes, one E4M3 byte
    per 16 elements and a 4-byte matrix scale per matrix; MXFP4: 4-bit codes and
    one E8M0 byte per 32 elements."""
    n_in = 2 if spec.gated else 1
    e_in = n_in * spec.expert_ffn * spec.k_in
    e_dn = spec.k_in * spec.expert_ffn
    if getattr(spec, "fmt", "affine") == "nvfp4":
        return (e_in // 2 + e_in // 16 + 4 * n_in, e_dn // 2 + e_dn // 16 + 4)
    if getattr(spec, "fmt", "affine") == "mxfp4":
        return (e_in // 2 + e_in // 32, e_dn // 2 + e_dn // 32)
    sb = 2 * 2
    b = spec.bits
    return (e_in * b // 8 + sb * (e_in // spec.group_size), e_dn * b // 8 + sb * (e_dn // spec.group_size))


def stage_bytes(spec, T, n_uniq):
    """Algorithmic bytes per stage for one forward of T rows with n_uniq
    distinct selected experts."""
    H, E, L, Fs, k = spec.hidden, spec.n_experts, spec.latent, spec.shared_ffn, spec.top_k
    rd = 4 if spec.router_dtype == "fp32" else 2
    n_sh_in = 2 if spec.gated else 1
    x_bytes = T * H * 2
    up_b, dn_b = expert_bytes(spec)
    din = E * H * rd + L * H * 2 + n_sh_in * Fs * H * 2 + x_bytes + (E if spec.router_bias else 0) * 4
    dout = H * L * 2 + H * Fs * 2 + x_bytes + T * H * 2
    return {"dense_in": din, "route": T * E * 4, "expert_up": n_uniq * up_b,
            "expert_down": n_uniq * dn_b, "dense_out": dout}


def layer_flops(spec, T):
    """Multiply-add flops of one forward of T rows (2 per MAC): router, latent
    projections, shared expert, and k routed experts per row."""
    H, E, L, Fs, k = spec.hidden, spec.n_experts, spec.latent, spec.shared_ffn, spec.top_k
    n_in = 2 if spec.gated else 1
    dense = E * H + 2 * L * H + (n_in + 1) * Fs * H
    experts = k * (n_in + 1) * spec.expert_ffn * spec.k_in
    return 2 * T * (dense + experts)


def layer_bytes(spec, T, n_uniq):
    b = stage_bytes(spec, T, n_uniq)
    return b["dense_in"] + b["expert_up"] + b["expert_down"] + b["dense_out"] - T * spec.hidden * 2


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def time_oracle(layer, rows: int, seconds: float, seed: int):
    """The fp64 oracle as it stands on host cores: one-row forwards until
    ``rows`` rows or ``seconds`` elapse.  Returns (rows done, seconds)."""
    import moe_inputs as mi
    import oracle
    done, t0 = 0, time.perf_counter()
    while done < rows:
        x = mi.make_x(layer.spec, 1, seed + 1000 + done)
        oracle.oracle_forward(layer, x)
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    return done, time.perf_counter() - t0


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate_replicas(local_ms: float, local_tokens: int, device=None):
    """Whole-job throughput of independent replicas: every rank's tokens over
    the slowest rank's time.  Returns (tokens/s, max ms, total tokens); a
    no-op reduction when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_tokens / (local_ms / 1e3), local_ms, local_tokens
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(local_tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    max_ms, tokens = float(t.item()), int(n.item())
    return tokens / (max_ms / 1e3), max_ms, tokens


def run_reference(args):
    import moe_inputs as mi
    rank, world, _ = dist_env()
    if rank != 0:
        return
    spec = mi.SPECS[args.config]
    layer = mi.make_layer(spec, args.seed)
    for i in range(args.warmup):
        time_oracle(layer, 1, 1e9, args.seed + 500 + i)
    per = []
    for i in range(args.steps):
        n, dt = time_oracle(layer, 1, 1e9, args.seed + i)
        per.append(dt)
    total = sum(per)
    value = args.steps * args.T / total
    cores = host_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.config == "latent" else spec.name + " layer", "T": 1},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} one-row forwards of the fp64 oracle"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(torch, pkg, spec, layer_h, T, steps, warmup, seed, flush, stream, profile=True):
    """Time `steps` forwards of T rows (L2 flushed before each).  Returns a
    dict with per-step times, per-stage times and realised distinct-expert
    counts."""
    import moe_inputs as mi
    nb = 32
    xs = [torch.from_numpy(mi.make_x(spec, T, seed + 100 * T + i).view(np.int16)).cuda()
          .view(torch.bfloat16) for i in range(nb)]
    out = torch.empty_like(xs[0])
    k = spec.top_k
    ids = torch.empty((steps, T, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, k), dtype=torch.float32, device="cuda")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    layer_h.profile(profile)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            flush.zero_()
            pkg.moe_layer_forward(layer_h.handle, xs[i % nb], T, out, stream.cuda_stream)
        stream.synchronize()
        stage_ms = np.zeros(len(STAGES))
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            pkg.moe_layer_forward_ex(layer_h.handle, xs[i % nb], T, out, stream.cuda_stream,
                                     ids[i], wts, None)
            evs[i][1].record(stream)
            if profile:
                stage_ms += np.array(layer_h.stage_times())
        stream.synchronize()
    layer_h.profile(False)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ids_np = ids.cpu().numpy()
    n_uniq = [len(np.unique(ids_np[i])) for i in range(steps)]
    return {"step_ms": step_ms, "stage_ms": stage_ms / steps, "n_uniq": n_uniq, "xs": xs}


def workload_line(torch, pkg, spec, T, steps, warmup, seed, flush, stream, hbm_peak, tc_peak,
                  zipf=False, path="auto", label=None):
    """One configured workload measured like the main line (L2 flushed before
    every timed forward): tokens/s, step time, achieved GB/s over the
    algorithmic bytes and its fraction of the HBM peak, and the flops of the
    step against the bf16 tensor peak."""
    import moe_inputs as mi
    rb = mi.zipf_router_bias(spec.n_experts, seed) if zipf else None
    layer = mi.make_layer(spec, seed, router_bias=rb)
    h = pkg.MoELayer(pkg.MoEConfig.from_spec(spec, max_tokens=max(T, 16)),
                     pkg.upload_arrays(layer.arrays()))
    torch.cuda.empty_cache()
    try:
        h.set_path(path)
        m = measure(torch, pkg, spec, h, T, steps, warmup, seed, flush, stream, profile=False)
        tt = sum(m["step_ms"]) / len(m["step_ms"])
        bb = float(np.mean([layer_bytes(spec, T, u) for u in m["n_uniq"]]))
        fl = layer_flops(spec, T)
        return {"workload": label or spec.name, "T": T, "zipf": bool(zipf), "path": h.path_for(T),
                "tokens_per_s": T / (tt / 1e3), "ms_per_step": tt,
                "ms_p10_p50_p90": [float(np.percentile(m["step_ms"], q)) for q in (10, 50, 90)],
                "gbs": bb / (tt / 1e3) / 1e9, "hbm_frac": bb / (tt / 1e3) / 1e9 / hbm_peak,
                "mean_distinct_experts": float(np.mean(m["n_uniq"])),
                "tflops": fl / (tt / 1e3) / 1e12, "tensor_frac": fl / (tt / 1e3) / 1e12 / tc_peak,
                "launches": h.last_launch_count(), "steps": steps}
    finally:
        h.close()
        torch.cuda.empty_cache()


def stack_line(torch, pkg, T, steps, warmup, flush, stream):
    """The five-layer heterogeneous stack (E = 240..496, latent shapes) run like
    a model: the layers in order on the same rows, the residual carried, L2
    flushed before every timed pass."""
    import moe_inputs as mi
    specs = mi.stack_specs()
    hs = [pkg.MoELayer(pkg.MoEConfig.from_spec(sp, max_tokens=16), pkg.upload_arrays(mi.make_layer(sp, i).arrays()))
          for i, sp in enumerate(specs)]
    torch.cuda.empty_cache()
    try:
        xs = [torch.from_numpy(mi.make_x(specs[0], T, 900 + i).view(np.int16)).cuda()
              .view(torch.bfloat16) for i in range(8)]
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(warmup + steps):
                flush.zero_()
                if i >= warmup:
                    evs[i - warmup][0].record(stream)
                cur = xs[i % 8]
                for hh in hs:
                    cur = hh.forward(cur, stream=stream)
                if i >= warmup:
                    evs[i - warmup][1].record(stream)
            stream.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        return {"workload": "stack of five latent layers, E = " + "/".join(str(sp.n_experts) for sp in specs),
                "T": T, "paths": [hh.path_for(T) for hh in hs], "ms_per_stack_step": ms,
                "tokens_per_s": T / (ms / 1e3), "layer_forwards_per_s": len(hs) / (ms / 1e3),
                "steps": steps}
    finally:
        for hh in hs:
            hh.close()
        torch.cuda.empty_cache()


def run_ours(args):
    import torch

    import moe_inputs as mi
    import quantized_moe_decode_gemv_gb300 as pkg

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = {}
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        peaks = json.load(open(pp))
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    tc_peak = peaks.get("bf16_tflops", 1900.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    spec = mi.SPECS[args.config]
    if args.fmt != "affine":
        spec = spec.with_(name=f"{spec.name}_{args.fmt}", fmt=args.fmt,
                          group_size=16 if args.fmt == "nvfp4" else 32)
    rb = mi.zipf_router_bias(spec.n_experts, args.seed + rank) if args.zipf else None
    layer = mi.make_layer(spec, args.seed + rank, router_bias=rb)
    sweep = [int(v) for v in args.sweep.split(",") if v.strip()]
    maxT = max([args.T, args.also_T or 1] + sweep)
    cfg = pkg.MoEConfig.from_spec(spec, max_tokens=max(maxT, 16))
    h = pkg.MoELayer(cfg, pkg.upload_arrays(layer.arrays(), device=dev))
    h.set_path(args.path)
    torch.cuda.empty_cache()
    flush = L2Flush(torch, dev)
    stream = torch.cuda.Stream()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        m = measure(torch, pkg, spec, h, args.T, args.steps, args.warmup, args.seed, flush, stream,
                    profile=False)
    torch.cuda.synchronize()
    # per-kernel durations: a second pass with an event between every kernel
    # (events serialise the kernels, so this pass has no inter-kernel overlap)
    mp = measure(torch, pkg, spec, h, args.T, max(10, min(args.steps, 50)), 2, args.seed, flush,
                 stream, profile=True)
    value, total_ms, tokens = aggregate_replicas(float(sum(m["step_ms"])), args.steps * args.T,
                                                 device=dev)
    bytes_steps = [layer_bytes(spec, args.T, u) for u in m["n_uniq"]]
    gbs = sum(bytes_steps) / (sum(m["step_ms"]) / 1e3) / 1e9

    # dominant kernel roofline: the kernel with the largest share of the step,
    # its launches pooled (the expert kernel runs twice: up and down)
    st = mp["stage_ms"]
    avg_uniq = float(np.mean(mp["n_uniq"]))
    sb = stage_bytes(spec, args.T, avg_uniq)
    path = h.path_for(args.T)
    launches = h.last_launch_count()
    per_kernel = {}
    kmap = KERNEL_OF_STAGE_GROUPED if path == "grouped" else KERNEL_OF_STAGE
    for i, n in enumerate(STAGES):
        kname = kmap[n]
        b, t = per_kernel.get(kname, (0.0, 0.0))
        per_kernel[kname] = (b + sb[n], t + float(st[i]))
    dom_name = max(per_kernel, key=lambda kn: per_kernel[kn][1])
    achieved = per_kernel[dom_name][0] / (per_kernel[dom_name][1] / 1e3) / 1e9
    stages = {n: {"kernel": kmap[n], "ms": round(float(st[i]), 5), "share": round(float(st[i] / st.sum()), 4),
                  "alg_bytes": int(sb[n]), "gbs": round(sb[n] / (st[i] / 1e3) / 1e9, 1)}
              for i, n in enumerate(STAGES)}

    # every other configured workload, measured the same way
    also = []
    if rank == 0 and not args.no_also:
        st_also = max(30, args.steps // 4)
        if args.also_T and args.also_T != args.T:
            also.append(workload_line(torch, pkg, mi.SPECS["latent"], args.also_T, st_also, args.warmup,
                                      args.seed + 1, flush, stream, hbm_peak, tc_peak,
                                      label="latent layer (uniform load)"))
        for T in (1, 4, 32):
            also.append(workload_line(torch, pkg, mi.SPECS["nonlatent"], T, st_also, args.warmup,
                                      args.seed, flush, stream, hbm_peak, tc_peak,
                                      label="non-latent sigmoid top-8 layer"))
        for T in (64, 256):
            also.append(workload_line(torch, pkg, mi.SPECS["latent"], T, st_also, args.warmup,
                                      args.seed, flush, stream, hbm_peak, tc_peak, zipf=True,
                                      label="latent layer, Zipf(1.1) expert load"))
        for T in (2, 9, 16):
            also.append(stack_line(torch, pkg, T, max(20, args.steps // 8), args.warmup, flush, stream))
        for T in (1, 4):
            also.append(workload_line(torch, pkg, mi.SPECS["tiny"], T, st_also, args.warmup, args.seed,
                                      flush, stream, hbm_peak, tc_peak, label="tiny layer"))
        fp4 = mi.SPECS["latent"].with_(name="latent_nvfp4", fmt="nvfp4", group_size=16)
        for T in (1, 16):
            also.append(workload_line(torch, pkg, fp4, T, st_also, args.warmup, args.seed, flush, stream,
                                      hbm_peak, tc_peak,
                                      label="latent layer, NVFP4 experts (E2M1, E4M3 per 16, fp32 per matrix)"))
        mx = mi.SPECS["latent"].with_(name="latent_mxfp4", fmt="mxfp4", group_size=32)
        also.append(workload_line(torch, pkg, mx, 1, st_also, args.warmup, args.seed, flush, stream,
                                  hbm_peak, tc_peak, label="latent layer, MXFP4 experts (E2M1, E8M0 per 32)"))

    # batched serving sweep (separate output file)
    if sweep and rank == 0:
        with open(args.sweep_out, "w") as f:
            for T in sweep:
                paths = ["grouped"] if T > 256 else ["gemv", "grouped"] if T >= 16 else ["gemv"]
                for pth in paths:
                    h.set_path(pth)
                    ms = measure(torch, pkg, spec, h, T, max(20, args.steps // 4), 3,
                                 args.seed + 7, flush, stream, profile=False)
                    tt = sum(ms["step_ms"])
                    bb = sum(layer_bytes(spec, T, u) for u in ms["n_uniq"])
                    f.write(json.dumps({
                        "T": T, "path": pth, "zipf": bool(args.zipf),
                        "tokens_per_s": len(ms["step_ms"]) * T / (tt / 1e3),
                        "ms_per_step": tt / len(ms["step_ms"]),
                        "gbs": bb / (tt / 1e3) / 1e9, "hbm_frac": bb / (tt / 1e3) / 1e9 / hbm_peak,
                        "mean_distinct_experts": float(np.mean(ms["n_uniq"])),
                        "expert_bytes_per_token": (float(np.mean(ms["n_uniq"])) *
                                                   sum(expert_bytes(spec)) / T),
                        "tflops": layer_flops(spec, T) / (tt / len(ms["step_ms"]) / 1e3) / 1e12,
                        "tensor_frac": (layer_flops(spec, T) / (tt / len(ms["step_ms"]) / 1e3) / 1e12
                                        / tc_peak)}) + "\n")
        h.set_path(args.path)

    # end to end through the host-buffer C-ABI call
    xs_host = [x.cpu().pin_memory() for x in m["xs"][:8]]
    out_host = torch.empty_like(xs_host[0]).pin_memory()
    e2e_steps = max(20, args.steps // 4)
    for i in range(3):
        h.forward_host(xs_host[i % 8], out_host, stream)
    e2e_total = 0.0
    for i in range(e2e_steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        h.forward_host(xs_host[i % 8], out_host, stream)
        e2e_total += time.perf_counter() - t0
    e2e = {"value": e2e_steps * args.T * world / e2e_total, "unit": "tokens/s",
           "h2d_bytes_per_step": args.T * spec.hidden * 2,
           "d2h_bytes_per_step": args.T * spec.hidden * 2}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, dt = time_oracle(layer, 10_000, args.cpu_seconds, args.seed)
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} one-row forwards of the same layer (fp64 NumPy, "
                         f"selected experts dequantised per row), {dt:.1f} s"}

    if rank == 0:
        workload = WORKLOAD if args.config == "latent" else spec.name + " layer"
        if args.fmt != "affine":
            workload += f", {args.fmt.upper()} experts"
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "ms_p10_p50_p90": [float(np.percentile(m["step_ms"], q)) for q in (10, 50, 90)],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random weights and activations)",
            "config": {"workload": workload, "T": args.T, "parallelism": "replicas" if world > 1 else "single",
                       "l2": "flushed before every timed step: 256 MB write, then 256 MB read (clean L2)",
                       "input_batches": 32},
            "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak, "hbm_peak_gbs": hbm_peak,
            "hbm_peak_source": peak_src,
            "mean_distinct_experts": float(np.mean(m["n_uniq"])),
            "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved,
                         "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                         "traffic": captured_traffic(dom_name, args.T, args.zipf), "peak_source": peak_src,
                         "timing": "CUDA events around each kernel on its stream (profiled pass)"},
            "profiled_step_ms": float(np.mean(mp["step_ms"])),
            "stages": stages,
            "also": also,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "path": path,
            "gpu_launches": launches * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
