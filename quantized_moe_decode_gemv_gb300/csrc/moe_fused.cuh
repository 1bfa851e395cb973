// The whole decode-time MoE layer as one persistent kernel (k_fused).
//
// At a few token rows per forward every stage of the layer is an HBM stream
// of its weights, but the routed stages are short and latency-bound: the
// selected experts' 9.6 MB of int4 codes (Bolt-like latent layer) cannot fill
// the HBM pipes between two launches, while the shared expert's 60 MB of bf16
// rows does not depend on the routing at all.  One cooperative launch keeps
// every CTA resident and lets the routing-independent streams run while the
// routed chain waits on its dependencies.
//
// Work of one CTA, in consumption order (the "phases"):
//   ROUTER, FC1, SHIN  its rows of the router, fc1_latent_proj and shared
//                      gate/up matrices (every CTA but CTA 0) -> dense_in
//   route              CTA 0: top-k selection once every router row is done
//   SD                 its rows of the shared-expert down matrix -> sdbuf
//   UP                 its share of the selected experts' up(+gate) rows,
//                      activation fused -> hbuf
//   DN                 its share of the selected experts' down rows -> pexp
//   combine            its slice of y = sum_j w_j * down_j (latent layers)
//   OUT                its rows of fc2_latent_proj . y + sdbuf + residual
//                      (latent), or combine + sdbuf + residual (non-latent)
//
// Weights move by bulk copies (cp.async.bulk, completion on an mbarrier) into
// a ring of shared-memory slots, a chunk of whole rows per slot.  Thread 0 is
// the producer: it keeps the ring full, and its issue order decides where the
// shared-expert down rows (SD) go: first while the routing is not yet
// published, then a few between the expert up and down rows (to cover that
// barrier), the rest before fc2.  All 256 threads consume the chunks in issue
// order with one compact executor for dense rows and one for int4 expert rows,
// so the code of every phase stays small and warm in the instruction cache.
//
// Dependencies between CTAs are counters in global memory: a CTA signals a
// phase after a CTA barrier, a gpu-scope fence and an atomic add; a waiting
// CTA's thread 0 spins on an acquire load (bounded: after FZ_SPIN_LIMIT polls
// the kernel sets the timeout bit of the status word and stops computing, but
// still signals and drains its copies, so no other CTA waits longer).  The
// launch is cooperative, so every CTA is resident and the waits end.  The last
// CTA to finish resets the counters for the next launch.  Every output element
// is computed by exactly one CTA in a fixed order, so results are
// deterministic and do not depend on the other rows of the batch.
#pragma once

#include "moe_kernels.cuh"

namespace moe {

constexpr uint32_t FZ_SPIN_LIMIT = 1u << 20;
constexpr int FZ_MAX_SLOTS = 8;
constexpr int FZ_MAX_JOBS = 12;     // per phase
constexpr int FZ_SYNC_STRIDE = 32;  // ints between counters (one 128-byte line each)

// counters (index * FZ_SYNC_STRIDE)
enum : int {
  FZ_ROUTER = 0,  // router rows done (CTAs 1..G-1)
  FZ_FC1,         // fc1 rows done (CTAs 1..G-1)
  FZ_DIN,         // shared gate/up rows done (CTAs 1..G-1)
  FZ_ROUTED,      // routing published (1)
  FZ_UP,          // expert up rows done (all CTAs)
  FZ_DN,          // expert down rows done (all CTAs)
  FZ_SD,          // shared down rows done (all CTAs)
  FZ_COMB,        // combine slice done (all CTAs)
  FZ_EXIT,        // CTAs finished
  FZ_WORDS = 9
};

// phases
enum : int { PH_ROUTER = 0, PH_FC1, PH_SHIN, PH_SD, PH_UP, PH_DN, PH_OUT, PH_N };

struct FusedArgs {
  int T;
  int H, E, L, Fs, k;
  int act;
  const void* x;
  int x_dt;
  // dense matrices: router [E, H] (router_dt), fc1 [L, H], sh_gate/sh_up [Fs, H],
  // sh_down [H, Fs], fc2 [H, L] (act dtype)
  const void* router_w;
  int router_dt;
  const void* fc1;
  const void* sh_gate;
  const void* sh_up;
  const void* sh_down;
  const void* fc2;
  float* dense_in;   // [T, din_rows]: router logits | fc1 | shared gate | shared up
  int din_rows, off_fc1, off_shg, off_shu;
  RouteArgs route;
  ExpertArgs up, dn;
  float* sdbuf;      // [T, H] shared-expert down output
  const float* pexp;
  const float* wts;
  float* ybuf;       // [T, L]
  void* out;
  float* delta;
  int* sync;         // FZ_WORDS counters, FZ_SYNC_STRIDE ints apart, zero at launch
  int* status;
  // ring
  int slots;         // S
  int slot_bytes;
  int sd_mid;        // SD chunks issued between the expert up and down rows
  unsigned long long* trace;   // diagnostics: [grid][FZ_TRACE] globaltimer stamps, or null
};

constexpr int FZ_TRACE = 32;

// ---------------------------------------------------------------------------
// PTX: mbarrier and bulk copy
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t fz_smem(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void fz_mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(fz_smem(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fz_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fz_smem(b)), "r"(bytes)
               : "memory");
}
// [dst, dst + bytes) <- [src, src + bytes); both 16-byte aligned, bytes % 16 == 0
__device__ __forceinline__ void fz_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          fz_smem(dst)),
      "l"(src), "r"(bytes), "r"(fz_smem(b))
      : "memory");
}
__device__ __forceinline__ bool fz_mbar_wait(uint64_t* b, uint32_t parity) {
  const uint32_t a = fz_smem(b);
  for (uint32_t i = 0; i < FZ_SPIN_LIMIT; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// CTA-wide wait until *p >= target; false (and the timeout bit set) if the
// bound ran out.  `ok` false skips the wait.
__device__ __forceinline__ bool fz_wait(const int* p, int target, int* status, bool ok) {
  bool w = true;
  if (threadIdx.x == 0 && ok) {
    w = false;
    for (uint32_t i = 0; i < FZ_SPIN_LIMIT; ++i) {
      if (ld_acquire(p) >= target) { w = true; break; }
      __nanosleep(32);
    }
    if (!w) atomicOr(status, STATUS_TIMEOUT);
    __threadfence();
  }
  return __syncthreads_and(w && ok) != 0;
}

// thread 0 only: publish after the CTA's writes are complete (caller barrier)
__device__ __forceinline__ void fz_post(int* p) {
  __threadfence();
  atomicAdd(p, 1);
}

__device__ __forceinline__ void span(int64_t n, int c, int g, int64_t& b, int64_t& e) {
  b = n * c / g;
  e = n * (c + 1) / g;
}

// ---------------------------------------------------------------------------
// jobs and chunks
// ---------------------------------------------------------------------------

// Dense job: rows [row0, row0 + nrows) of one matrix, R rows per chunk.
// Expert job: rows [row0, row0 + nrows) of distinct-expert slot u (expert e),
// all pairs [pa, pa + np) of the slot in groups of PB; chunk = (group, R rows).
struct FzJob {
  const char* w;    // dense: matrix; expert: codes of expert e
  const char* w2;   // expert: gate codes of expert e (gated up), else null
  const char* sb;   // expert: scale/bias words of expert e
  const char* sb2;
  int row0, nrows, R;
  int col;          // dense: output column of row0; expert: slot u
  int pa, np;       // expert pairs
  int nchunks, first;
};

struct FzPhase {
  int njobs, nchunks, passes;   // nchunks per pass
  int ready;                    // job table built
  int K, dt;                    // reduction width, weight dtype (dense)
  FzJob job[FZ_MAX_JOBS];
};

// Shared bookkeeping of a CTA (dynamic shared memory, after the ring).
struct FzShared {
  FzPhase ph[PH_N];
  int slot_phase[FZ_MAX_SLOTS];
  int slot_idx[FZ_MAX_SLOTS];
  int issued;        // chunks issued (written by thread 0)
  int done_all;      // producer has nothing left
  int routed;        // thread 0's last view of the routing flag
  int pid[8];        // expert staging: pair ids of the staged group
};

// ---------------------------------------------------------------------------
// staging (all threads)
// ---------------------------------------------------------------------------

// fp32 [TB][K] vector swizzled for 8-element (16-bit weights) or 4-element
// (fp32 weights) readers: element f4 of token row t at xs4[t * K4 + swz(f4, 1)].
// kind 0: x (16-bit); 1: act(shared gate, shared up) from dense_in; 2: ybuf.
template <int TB>
__device__ __forceinline__ void fz_stage_dense(const FusedArgs& A, int kind, int t0, int tb, int K,
                                               float4* xs4) {
  const int K4 = K >> 2;
  for (int i = threadIdx.x; i < TB * K4; i += NT) {
    const int t = i / K4, f4 = i - t * K4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < tb) {
      const int64_t tt = t0 + t;
      if (kind == 0) {
        const int64_t e = tt * A.H + 4 * f4;
        v.x = ld16(A.x, e, A.x_dt); v.y = ld16(A.x, e + 1, A.x_dt);
        v.z = ld16(A.x, e + 2, A.x_dt); v.w = ld16(A.x, e + 3, A.x_dt);
      } else if (kind == 1) {
        // the shared columns start at any column of dense_in: scalar loads
        const float* du = A.dense_in + tt * A.din_rows + A.off_shu + 4 * f4;
        const float* dg = A.dense_in + tt * A.din_rows + A.off_shg + 4 * f4;
        const bool gl = A.act == ACT_SWIGLU;
        const float u0 = __ldcg(du), u1 = __ldcg(du + 1), u2 = __ldcg(du + 2), u3 = __ldcg(du + 3);
        float g0 = 0.f, g1 = 0.f, g2 = 0.f, g3 = 0.f;
        if (gl) { g0 = __ldcg(dg); g1 = __ldcg(dg + 1); g2 = __ldcg(dg + 2); g3 = __ldcg(dg + 3); }
        v = make_float4(act_fn(A.act, g0, u0), act_fn(A.act, g1, u1), act_fn(A.act, g2, u2),
                        act_fn(A.act, g3, u3));
      } else {
        v = __ldcg(reinterpret_cast<const float4*>(A.ybuf + tt * A.L) + f4);
      }
    }
    xs4[t * K4 + swz(f4, 1)] = v;
  }
}

// Input rows of pairs [pa, pa + np) of an expert launch (PB slots), swizzled
// for 32-element chunk readers, their 32-element chunk sums and pair ids.
template <int PB>
__device__ __forceinline__ void fz_stage_expert(const ExpertArgs& X, int pa, int np, float4* xs4,
                                                int* pid_s) {
  const int K = X.K, K4 = K >> 2, nchunk = K >> 5;
  float* xsum = reinterpret_cast<float*>(xs4 + PB * K4);
  const int* pairs = X.meta + 2 + 2 * X.umax;
  if (threadIdx.x < PB) pid_s[threadIdx.x] = static_cast<int>(threadIdx.x) < np ? __ldcg(pairs + pa + threadIdx.x) : 0;
  for (int i = threadIdx.x; i < PB * K4; i += NT) {
    const int pp = i / K4, f4 = i - pp * K4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (pp < np) {
      const int pid = __ldcg(pairs + pa + pp);
      const int64_t row = X.xin_by_pair ? pid : (pid / X.k);
      const int64_t base = X.xin_off + row * X.xin_stride + 4 * f4;
      if (X.xin_dt == DT_FP32) {
        const float* src = static_cast<const float*>(X.xin) + base;
        if (((X.xin_off | X.xin_stride) & 3) == 0) {
          v = __ldcg(reinterpret_cast<const float4*>(src));
        } else {
          v.x = __ldcg(src); v.y = __ldcg(src + 1); v.z = __ldcg(src + 2); v.w = __ldcg(src + 3);
        }
      } else {
        v.x = ld16(X.xin, base, X.xin_dt); v.y = ld16(X.xin, base + 1, X.xin_dt);
        v.z = ld16(X.xin, base + 2, X.xin_dt); v.w = ld16(X.xin, base + 3, X.xin_dt);
      }
    }
    xs4[pp * K4 + swz(f4, 7)] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < PB * nchunk; i += NT) {
    const int pp = i / nchunk, c = i - pp * nchunk;
    const float4* x8 = xs4 + pp * K4 + 8 * c;
    float sx = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) { const float4 a = x8[j]; sx += (a.x + a.y) + (a.z + a.w); }
    xsum[pp * nchunk + c] = sx;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// executors (one copy each, shared by every phase)
// ---------------------------------------------------------------------------

// Epilogue of a dense chunk.
struct FzEpi {
  int mode;          // 0: store fp32 to out[t * ld + col]; 1: final output row
  float* out;
  int64_t ld;
};

// Rows [0, n) of a chunk of R rows (K elements of dtype dt each) in shared
// memory against TB staged token rows; v(t, r) goes to the epilogue for token
// row t0 + t (t < tb) and output column col + r.  R in {1, 2, 4, 8}: 8 / R
// warps share a row, each a contiguous K slice.
template <int TB>
__device__ __noinline__ void fz_dense_chunk(const FusedArgs& A, const char* slot, int n, int R, int K,
                                            int dt, const float4* xs4, float* red, int t0, int tb,
                                            int col, FzEpi ep) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpr = NW / R;
  const int rl = warp / wpr, q = warp - rl * wpr;
  const int K4 = K >> 2;
  float acc[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) acc[t] = 0.f;
  if (rl < n) {
    if (dt != DT_FP32) {
      const int pieces = K >> 3, per = pieces / wpr;   // 8 elements per piece
      const uint4* wr = reinterpret_cast<const uint4*>(slot + static_cast<int64_t>(rl) * K * 2);
#pragma unroll 2
      for (int p = q * per + lane; p < (q + 1) * per; p += 32) {
        float wf[8];
        cvt8(wr[p], dt, wf);
        const int s0 = swz(2 * p, 1), s1 = swz(2 * p + 1, 1);
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          const float4 a = xs4[t * K4 + s0], b = xs4[t * K4 + s1];
          float s = acc[t];
          s = fmaf(wf[0], a.x, s); s = fmaf(wf[1], a.y, s); s = fmaf(wf[2], a.z, s); s = fmaf(wf[3], a.w, s);
          s = fmaf(wf[4], b.x, s); s = fmaf(wf[5], b.y, s); s = fmaf(wf[6], b.z, s); s = fmaf(wf[7], b.w, s);
          acc[t] = s;
        }
      }
    } else {
      const int pieces = K >> 2, per = pieces / wpr;   // 4 elements per piece
      const float4* wr = reinterpret_cast<const float4*>(slot + static_cast<int64_t>(rl) * K * 4);
#pragma unroll 2
      for (int p = q * per + lane; p < (q + 1) * per; p += 32) {
        const float4 w = wr[p];
        const int s0 = swz(p, 1);
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          const float4 a = xs4[t * K4 + s0];
          float s = acc[t];
          s = fmaf(w.x, a.x, s); s = fmaf(w.y, a.y, s); s = fmaf(w.z, a.z, s); s = fmaf(w.w, a.w, s);
          acc[t] = s;
        }
      }
    }
  }
  const float tot = warp_reduce_scatter<TB>(acc, lane);
  constexpr int LPV = 32 / TB;
  if ((lane & (LPV - 1)) == 0) red[warp * TB + lane / LPV] = tot;
  __syncthreads();
  for (int o = threadIdx.x; o < n * TB; o += NT) {
    const int r = o / TB, t = o - r * TB;
    if (t >= tb) continue;
    float s = 0.f;
    for (int qq = 0; qq < wpr; ++qq) s += red[(r * wpr + qq) * TB + t];
    const int tt = t0 + t, cc = col + r;
    if (ep.mode == 0) {
      ep.out[tt * ep.ld + cc] = s;
    } else {
      const int64_t e = static_cast<int64_t>(tt) * A.H + cc;
      if (A.Fs) s += __ldcg(A.sdbuf + e);
      const float xv = ld16(A.x, e, A.x_dt);
      reinterpret_cast<unsigned short*>(A.out)[e] = st16_bits(xv + s, A.x_dt);
      if (A.delta) A.delta[e] = s;
    }
  }
}

// Rows [0, n) of a chunk of int4 expert rows in shared memory: codes
// [n][K/2 bytes], then scale/bias words [n][K/G] at sb (and the gate's at
// q2/sb2), against the np staged pair rows.  Warp w takes rows w, w + 8, ...;
// a lane takes 32-code pieces lane, lane + 32, ...
template <int PB, bool GATED>
__device__ __noinline__ void fz_expert_chunk(const ExpertArgs& X, const char* q, const uint32_t* sb,
                                             const char* q2, const uint32_t* sb2, int n, int row0,
                                             const float4* xs4, const int* pid_s, int np) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = X.K, K4 = K >> 2, nchunk = K >> 5, ngr = K / X.G;
  const float* xsum = reinterpret_cast<const float*>(xs4 + PB * K4);
  constexpr int NV = 2 * PB;
  constexpr int LPV = 32 / NV;
#pragma unroll 1
  for (int r = warp; r < n; r += NW) {
    float acc[PB], accg[PB];
#pragma unroll
    for (int pp = 0; pp < PB; ++pp) { acc[pp] = 0.f; accg[pp] = 0.f; }
    const uint4* qr = reinterpret_cast<const uint4*>(q + static_cast<int64_t>(r) * (K >> 1));
    const uint32_t* sr = sb + r * ngr;
#pragma unroll 1
    for (int cc = lane; cc < nchunk; cc += 32) {
      const uint4 w = qr[cc];
      float sc, bi;
      sb_decode(sr[(cc << 5) / X.G], X.s_dt, sc, bi);
      const float s16 = 16.f * sc, bb = bi - s16;
      uint4 wg = make_uint4(0u, 0u, 0u, 0u);
      float sg16 = 0.f, bbg = 0.f;
      if (GATED) {
        wg = reinterpret_cast<const uint4*>(q2 + static_cast<int64_t>(r) * (K >> 1))[cc];
        float sg, bg;
        sb_decode(sb2[r * ngr + (cc << 5) / X.G], X.s_dt, sg, bg);
        sg16 = 16.f * sg;
        bbg = bg - sg16;
      }
#pragma unroll
      for (int pp = 0; pp < PB; ++pp) {
        if (pp < np) {
          const float4* x8 = xs4 + pp * K4 + 8 * cc;
          const float xs = xsum[pp * nchunk + cc];
          acc[pp] = fmaf(s16, chunk_dot(w, x8, cc), fmaf(bb, xs, acc[pp]));
          if (GATED) accg[pp] = fmaf(sg16, chunk_dot(wg, x8, cc), fmaf(bbg, xs, accg[pp]));
        }
      }
    }
    float v[NV];
#pragma unroll
    for (int pp = 0; pp < PB; ++pp) { v[2 * pp] = acc[pp]; v[2 * pp + 1] = accg[pp]; }
    const float tot = warp_reduce_scatter<NV>(v, lane);
    const float other = __shfl_down_sync(0xffffffffu, tot, LPV);   // gate partner
    if ((lane & (2 * LPV - 1)) == 0) {
      const int pp = (lane / LPV) >> 1;
      if (pp < np) {
        const float val = (X.act >= 0) ? act_fn(X.act, other, tot) : tot;
        X.out[static_cast<int64_t>(pid_s[pp]) * X.n_rows + row0 + r] = val;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int TB, int PB, bool GATED>
__global__ void __launch_bounds__(NT, TB >= 8 ? 1 : 2) k_fused(const __grid_constant__ FusedArgs A) {
  extern __shared__ __align__(128) char fz_smem_raw[];
  const int c = blockIdx.x, G = gridDim.x;
  const int S = A.slots;
  const int SB = A.slot_bytes;
  char* ring = fz_smem_raw;
  uint64_t* bar = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(S) * SB);
  FzShared* sh = reinterpret_cast<FzShared*>(bar + FZ_MAX_SLOTS);
  float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(sh) + ((sizeof(FzShared) + 15) & ~size_t(15)));
  float4* xs4 = reinterpret_cast<float4*>(red + NW * 8);   // staged vectors / route scratch
  int* sync = A.sync;
  const int T = A.T;
  const int tid = threadIdx.x;
  bool ok = true;
  auto stamp = [&](int i) {
    if (A.trace && tid == 0) A.trace[c * FZ_TRACE + i] = global_ns();
  };
  stamp(0);

  // ---- job tables of the routing-independent phases (thread 0) ----
  const int passes = (T + TB - 1) / TB;
  const bool din_cta = c > 0;
  if (tid == 0) {
    for (int s = 0; s < FZ_MAX_SLOTS; ++s) fz_mbar_init(bar + s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    auto dense_job = [&](FzPhase& P, const void* w, int dt, int K, int rows, int cc, int gg, int col0) {
      int64_t b, e;
      span(rows, cc, gg, b, e);
      if (e <= b) return;
      const int rb = K * (dt == DT_FP32 ? 4 : 2);
      int R = 8;
      while (R > 1 && R * rb > SB) R >>= 1;
      FzJob& J = P.job[P.njobs++];
      J.w = static_cast<const char*>(w);
      J.w2 = nullptr; J.sb = nullptr; J.sb2 = nullptr;
      J.row0 = static_cast<int>(b);
      J.nrows = static_cast<int>(e - b);
      J.R = R;
      J.col = col0 + static_cast<int>(b);
      J.pa = 0; J.np = 0;
      J.nchunks = (J.nrows + R - 1) / R;
      J.first = P.nchunks;
      P.nchunks += J.nchunks;
    };
    for (int p = 0; p < PH_N; ++p) {
      FzPhase& P = sh->ph[p];
      P.njobs = 0; P.nchunks = 0; P.passes = 1; P.ready = 0; P.K = A.H; P.dt = A.x_dt;
    }
    const int gd = G - 1, cd = c - 1;
    if (din_cta) {
      FzPhase& P0 = sh->ph[PH_ROUTER];
      P0.dt = A.router_dt; P0.passes = passes;
      dense_job(P0, A.router_w, A.router_dt, A.H, A.E, cd, gd, 0);
      FzPhase& P1 = sh->ph[PH_FC1];
      P1.passes = passes;
      if (A.L) dense_job(P1, A.fc1, A.x_dt, A.H, A.L, cd, gd, A.off_fc1);
      FzPhase& P2 = sh->ph[PH_SHIN];
      P2.passes = passes;
      if (A.Fs) {
        if (A.act == ACT_SWIGLU) dense_job(P2, A.sh_gate, A.x_dt, A.H, A.Fs, cd, gd, A.off_shg);
        dense_job(P2, A.sh_up, A.x_dt, A.H, A.Fs, cd, gd, A.off_shu);
      }
    }
    sh->ph[PH_ROUTER].ready = sh->ph[PH_FC1].ready = sh->ph[PH_SHIN].ready = 1;
    FzPhase& Ps = sh->ph[PH_SD];
    Ps.K = A.Fs; Ps.passes = passes;
    if (A.Fs) dense_job(Ps, A.sh_down, A.x_dt, A.Fs, A.H, c, G, 0);
    Ps.ready = 1;
    FzPhase& Po = sh->ph[PH_OUT];
    Po.K = A.L; Po.passes = passes;
    if (A.L) dense_job(Po, A.fc2, A.x_dt, A.L, A.H, c, G, 0);
    Po.ready = 1;
    sh->issued = 0;
    sh->done_all = 0;
    sh->routed = 0;
    // phases without rows are complete at once
    if (din_cta) {
      if (sh->ph[PH_ROUTER].nchunks == 0) fz_post(sync + FZ_ROUTER * FZ_SYNC_STRIDE);
      if (sh->ph[PH_FC1].nchunks == 0) fz_post(sync + FZ_FC1 * FZ_SYNC_STRIDE);
      if (sh->ph[PH_SHIN].nchunks == 0) fz_post(sync + FZ_DIN * FZ_SYNC_STRIDE);
    }
    if (sh->ph[PH_SD].nchunks == 0) fz_post(sync + FZ_SD * FZ_SYNC_STRIDE);
  }
  __syncthreads();

  // ---- routing (CTA 0) ----
  if (c == 0) {
    ok = fz_wait(sync + FZ_ROUTER * FZ_SYNC_STRIDE, G - 1, A.status, ok);
    stamp(1);
    if (ok)
      route_block(A.route, reinterpret_cast<int*>(xs4));
    else if (tid == 0)
      A.route.meta[0] = 0;   // no routing: the expert phases find no work
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicExch(sync + FZ_ROUTED * FZ_SYNC_STRIDE, 1);
    }
    stamp(2);
  }

  // ---- producer (thread 0): the next chunk in issue order ----
  // steps: 0 ROUTER, 1 FC1, 2 SHIN, 3 SD until routed, 4 UP, 5 SD (sd_mid), 6 DN,
  // 7 SD rest, 8 OUT, 9 done
  int step = 0, sd_mid_left = A.sd_mid;
  int cur[PH_N];
  for (int p = 0; p < PH_N; ++p) cur[p] = 0;

  // expert job tables from the route metadata (thread 0; after the routing flag)
  auto build_expert = [&](int ph, const ExpertArgs& X, bool gated_up) {
    FzPhase& P = sh->ph[ph];
    P.njobs = 0; P.nchunks = 0; P.passes = 1; P.K = X.K;
    const int nu = min(max(__ldcg(X.meta), 0), X.umax);
    const int ngr = X.K / X.G;
    const int rowb = (gated_up ? 2 : 1) * (X.K / 2 + ngr * 4);
    int R = (SB - (gated_up ? 32 : 16)) / rowb;
    R = max(1, min(R, 32));
    int64_t b, e;
    span(static_cast<int64_t>(nu) * X.n_rows, c, G, b, e);
    while (b < e && P.njobs < FZ_MAX_JOBS) {
      const int u = static_cast<int>(b / X.n_rows);
      const int n0 = static_cast<int>(b - static_cast<int64_t>(u) * X.n_rows);
      const int n1 = static_cast<int>(min(static_cast<int64_t>(X.n_rows), n0 + (e - b)));
      const int64_t ex = __ldcg(X.meta + 1 + u);
      const int pa = __ldcg(X.meta + 1 + X.umax + u), pe = __ldcg(X.meta + 2 + X.umax + u);
      FzJob& J = P.job[P.njobs++];
      J.w = reinterpret_cast<const char*>(X.q) + ex * X.n_rows * (X.K / 2);
      J.sb = reinterpret_cast<const char*>(X.sb) + ex * X.n_rows * ngr * 4;
      J.w2 = gated_up ? reinterpret_cast<const char*>(X.q_gate) + ex * X.n_rows * (X.K / 2) : nullptr;
      J.sb2 = gated_up ? reinterpret_cast<const char*>(X.sb_gate) + ex * X.n_rows * ngr * 4 : nullptr;
      J.row0 = n0;
      J.nrows = n1 - n0;
      J.R = R;
      J.col = u;
      J.pa = pa;
      J.np = max(0, pe - pa);
      const int groups = (J.np + PB - 1) / PB;
      J.nchunks = groups * ((J.nrows + R - 1) / R);
      J.first = P.nchunks;
      P.nchunks += J.nchunks;
      b += n1 - n0;
    }
    if (b < e) atomicOr(A.status, STATUS_TIMEOUT);   // job table overflow (not expected)
    P.ready = 1;
  };

  // chunk i of a phase: job j, pass (dense) and chunk lc within the job
  auto locate = [&](const FzPhase& P, int i, int& j, int& pass, int& lc) {
    pass = i / max(P.nchunks, 1);
    const int ci = i - pass * P.nchunks;
    j = 0;
    while (j + 1 < P.njobs && ci >= P.job[j + 1].first) ++j;
    lc = ci - P.job[j].first;
  };

  auto issue = [&](int p, int i) {
    const int seq = sh->issued;
    const int s = seq % S;
    const FzPhase& P = sh->ph[p];
    int j, pass, lc;
    locate(P, i, j, pass, lc);
    const FzJob& J = P.job[j];
    char* dst = ring + static_cast<size_t>(s) * SB;
    sh->slot_phase[s] = p;
    sh->slot_idx[s] = i;
    if (p == PH_UP || p == PH_DN) {
      const ExpertArgs& X = (p == PH_UP) ? A.up : A.dn;
      const int nrc = (J.nrows + J.R - 1) / J.R;
      const int rc = lc % nrc;
      const int r = J.row0 + rc * J.R, n = min(J.R, J.row0 + J.nrows - r);
      const int ngr = X.K / X.G;
      const uint32_t qb = static_cast<uint32_t>(n) * (X.K / 2);
      const uint64_t sa = reinterpret_cast<uint64_t>(J.sb + static_cast<int64_t>(r) * ngr * 4);
      const uint64_t sa0 = sa & ~uint64_t(15);
      const uint32_t sbb = static_cast<uint32_t>((sa + static_cast<uint64_t>(n) * ngr * 4 - sa0 + 15) & ~uint64_t(15));
      uint32_t tx = qb + sbb;
      uint32_t sbb2 = 0;
      uint64_t sa2_0 = 0;
      if (J.w2) {
        const uint64_t sa2 = reinterpret_cast<uint64_t>(J.sb2 + static_cast<int64_t>(r) * ngr * 4);
        sa2_0 = sa2 & ~uint64_t(15);
        sbb2 = static_cast<uint32_t>((sa2 + static_cast<uint64_t>(n) * ngr * 4 - sa2_0 + 15) & ~uint64_t(15));
        tx += qb + sbb2;
      }
      fz_expect_tx(bar + s, tx);
      fz_bulk(dst, J.w + static_cast<int64_t>(r) * (X.K / 2), qb, bar + s);
      fz_bulk(dst + qb, reinterpret_cast<const void*>(sa0), sbb, bar + s);
      if (J.w2) {
        fz_bulk(dst + qb + sbb, J.w2 + static_cast<int64_t>(r) * (X.K / 2), qb, bar + s);
        fz_bulk(dst + 2 * qb + sbb, reinterpret_cast<const void*>(sa2_0), sbb2, bar + s);
      }
    } else {
      const int esz = P.dt == DT_FP32 ? 4 : 2;
      const int r = J.row0 + lc * J.R, n = min(J.R, J.row0 + J.nrows - r);
      const uint32_t bytes = static_cast<uint32_t>(n) * P.K * esz;
      fz_expect_tx(bar + s, bytes);
      fz_bulk(dst, J.w + static_cast<int64_t>(r) * P.K * esz, bytes, bar + s);
    }
    sh->issued = seq + 1;
  };

  // thread 0: issue while a slot is free and the next chunk is known
  auto produce = [&](int consumed) {
    // one poll of the routing flag per call while the issue order waits on it
    if ((step == 3 || step == 4) && !sh->routed && ld_acquire(sync + FZ_ROUTED * FZ_SYNC_STRIDE) >= 1)
      sh->routed = 1;
    if (sh->routed && !sh->ph[PH_UP].ready) {
      build_expert(PH_UP, A.up, GATED);
      build_expert(PH_DN, A.dn, false);
      if (sh->ph[PH_UP].nchunks == 0) fz_post(sync + FZ_UP * FZ_SYNC_STRIDE);
      if (sh->ph[PH_DN].nchunks == 0) fz_post(sync + FZ_DN * FZ_SYNC_STRIDE);
    }
    while (sh->issued - consumed < S && step < 9) {
      if (step == 3) {
        const FzPhase& Ps = sh->ph[PH_SD];
        if (sh->routed) { ++step; continue; }
        if (cur[PH_SD] < Ps.nchunks * Ps.passes) { issue(PH_SD, cur[PH_SD]++); continue; }
        break;   // nothing to issue until the routing is published
      }
      if (step == 4 && !sh->routed) break;
      const int p = step == 0 ? PH_ROUTER : step == 1 ? PH_FC1 : step == 2 ? PH_SHIN
                  : step == 4 ? PH_UP : step == 6 ? PH_DN : step == 8 ? PH_OUT : PH_SD;
      const FzPhase& P = sh->ph[p];
      const int total = P.nchunks * P.passes;
      if (step == 5) {
        if (sd_mid_left > 0 && cur[PH_SD] < total) { --sd_mid_left; issue(PH_SD, cur[PH_SD]++); continue; }
        ++step;
        continue;
      }
      if (cur[p] < total) { issue(p, cur[p]++); continue; }
      ++step;
    }
    sh->done_all = step >= 9;
  };

  // ---- consumer loop (all threads) ----
  int consumed = 0;
  int done_cnt[PH_N];
  for (int p = 0; p < PH_N; ++p) done_cnt[p] = 0;
  int staged = -1;          // what xs holds: kind * 65536 + pass (dense), 0x40000 + job (expert)
  uint32_t waited = 0;      // dependency waits already satisfied (bit per counter)
  bool comb_done = false;
  auto need = [&](int ctr, int target) {
    if (waited & (1u << ctr)) return;
    ok = fz_wait(sync + ctr * FZ_SYNC_STRIDE, target, A.status, ok);
    waited |= 1u << ctr;
  };
  auto combine = [&]() {
    // y[t, l] = sum_j w[t, j] * pexp[t k + j, l] over this CTA's slice
    need(FZ_DN, G);
    int64_t b, e;
    span(static_cast<int64_t>(T) * A.L, c, G, b, e);
    for (int64_t i = b + tid; ok && i < e; i += NT) {
      const int t = static_cast<int>(i / A.L), l = static_cast<int>(i - static_cast<int64_t>(t) * A.L);
      float y = 0.f;
      for (int j = 0; j < A.k; ++j)
        y = fmaf(__ldcg(A.wts + t * A.k + j), __ldcg(A.pexp + static_cast<int64_t>(t * A.k + j) * A.L + l), y);
      A.ybuf[i] = y;
    }
    __syncthreads();
    if (tid == 0) fz_post(sync + FZ_COMB * FZ_SYNC_STRIDE);
    comb_done = true;
  };

  while (true) {
    if (tid == 0) produce(consumed);
    __syncthreads();
    if (consumed == sh->issued) {
      if (sh->done_all || !ok) break;
      // the ring is empty and the next chunks need the routing
      need(FZ_ROUTED, 1);
      if (!ok) break;
      continue;
    }
    const int s = consumed % S;
    const int p = sh->slot_phase[s], i = sh->slot_idx[s];
    const FzPhase& P = sh->ph[p];
    int j, pass, lc;
    locate(P, i, j, pass, lc);
    const FzJob& J = P.job[j];
    // dependencies of the phase
    if (p == PH_SD) need(FZ_DIN, G - 1);
    if (p == PH_UP && A.L) need(FZ_FC1, G - 1);
    if (p == PH_DN) need(FZ_UP, G);
    if (p == PH_OUT) {
      if (!comb_done) combine();
      need(FZ_COMB, G);
      need(FZ_SD, G);
    }
    const bool wok = __syncthreads_and(tid != 0 || fz_mbar_wait(bar + s, (consumed / S) & 1)) != 0;
    if (!wok && tid == 0) atomicOr(A.status, STATUS_TIMEOUT);
    ok = ok && wok;
    const char* slot = ring + static_cast<size_t>(s) * SB;
    if (p == PH_UP || p == PH_DN) {
      const ExpertArgs& X = (p == PH_UP) ? A.up : A.dn;
      const int nrc = (J.nrows + J.R - 1) / J.R;
      const int g = lc / nrc, rc = lc - g * nrc;
      const int r = J.row0 + rc * J.R, n = min(J.R, J.row0 + J.nrows - r);
      const int pa = J.pa + g * PB, np = min(PB, J.np - g * PB);
      const int tag = 0x40000 + (p << 12) + (j << 6) + g;
      if (ok && staged != tag) {
        fz_stage_expert<PB>(X, pa, np, xs4, sh->pid);
        staged = tag;
      }
      const int ngr = X.K / X.G;
      const uint32_t qb = static_cast<uint32_t>(n) * (X.K / 2);
      const uint64_t sa = reinterpret_cast<uint64_t>(J.sb + static_cast<int64_t>(r) * ngr * 4);
      const uint32_t off = static_cast<uint32_t>(sa & 15);
      const uint32_t sbb = static_cast<uint32_t>((off + static_cast<uint64_t>(n) * ngr * 4 + 15) & ~uint64_t(15));
      const uint32_t* sbp = reinterpret_cast<const uint32_t*>(slot + qb + off);
      const char* q2 = nullptr;
      const uint32_t* sb2p = nullptr;
      if (J.w2) {
        const uint64_t sa2 = reinterpret_cast<uint64_t>(J.sb2 + static_cast<int64_t>(r) * ngr * 4);
        q2 = slot + qb + sbb;
        sb2p = reinterpret_cast<const uint32_t*>(slot + 2 * qb + sbb + (sa2 & 15));
      }
      if (ok) {
        if (p == PH_UP)
          fz_expert_chunk<PB, GATED>(X, slot, sbp, q2, sb2p, n, r, xs4, sh->pid, np);
        else
          fz_expert_chunk<PB, false>(X, slot, sbp, nullptr, nullptr, n, r, xs4, sh->pid, np);
      }
    } else {
      const int kind = (p == PH_SD) ? 1 : (p == PH_OUT) ? 2 : 0;
      const int t0 = pass * TB, tb = min(TB, T - t0);
      const int tag = kind * 65536 + pass;
      if (ok && staged != tag) {
        fz_stage_dense<TB>(A, kind, t0, tb, P.K, xs4);
        __syncthreads();
        staged = tag;
      }
      const int r = J.row0 + lc * J.R, n = min(J.R, J.row0 + J.nrows - r);
      FzEpi ep;
      ep.mode = (p == PH_OUT) ? 1 : 0;
      ep.out = (p == PH_SD) ? A.sdbuf : A.dense_in;
      ep.ld = (p == PH_SD) ? A.H : A.din_rows;
      if (ok) fz_dense_chunk<TB>(A, slot, n, J.R, P.K, P.dt, xs4, red, t0, tb, J.col + (r - J.row0), ep);
    }
    __syncthreads();   // the slot, the staging and the reduction area are free again
    ++consumed;
    if (++done_cnt[p] == P.nchunks * P.passes) {
      const int sg = p == PH_ROUTER ? FZ_ROUTER : p == PH_FC1 ? FZ_FC1 : p == PH_SHIN ? FZ_DIN
                   : p == PH_SD ? FZ_SD : p == PH_UP ? FZ_UP : p == PH_DN ? FZ_DN : -1;
      if (sg >= 0 && tid == 0) fz_post(sync + sg * FZ_SYNC_STRIDE);
      if (p == PH_SHIN) stamp(3);
      if (p == PH_UP) stamp(5);
      if (p == PH_DN) stamp(8);
      if (p == PH_SD) stamp(9);
    }
  }
  stamp(10);

  // ---- tail: the combine (CTAs without fc2 rows) and the non-latent output ----
  if (A.L) {
    if (!comb_done) combine();
  } else {
    need(FZ_DN, G);
    need(FZ_SD, G);
    int64_t b, e;
    span(static_cast<int64_t>(T) * A.H, c, G, b, e);
    for (int64_t i = b + tid; ok && i < e; i += NT) {
      const int t = static_cast<int>(i / A.H), n = static_cast<int>(i - static_cast<int64_t>(t) * A.H);
      float y = 0.f;
      for (int jj = 0; jj < A.k; ++jj)
        y = fmaf(__ldcg(A.wts + t * A.k + jj), __ldcg(A.pexp + static_cast<int64_t>(t * A.k + jj) * A.H + n), y);
      if (A.Fs) y += __ldcg(A.sdbuf + i);
      const float xv = ld16(A.x, i, A.x_dt);
      reinterpret_cast<unsigned short*>(A.out)[i] = st16_bits(xv + y, A.x_dt);
      if (A.delta) A.delta[i] = y;
    }
  }

  // ---- exit: the last CTA clears the counters for the next launch ----
  __syncthreads();
  stamp(12);
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(sync + FZ_EXIT * FZ_SYNC_STRIDE, 1) == G - 1) {
      __threadfence();
      for (int i = 0; i < FZ_WORDS; ++i) atomicExch(sync + i * FZ_SYNC_STRIDE, 0);
    }
  }
}

// Host launchers, one translation unit per TB (moe_fused.cu built with
// -DFZ_TB=1, 2, 4, 8).  The cache holds the cooperative grid for `smem`
// bytes of shared memory (grid 0: not yet queried).  Launched cooperatively:
// the runtime refuses a grid that cannot be resident at once.
struct FusedLaunchCache {
  size_t smem = 0;
  int grid = 0;
};
cudaError_t fused_launch_tb1(const FusedArgs& a, bool gated, size_t smem, int num_sms,
                             FusedLaunchCache* cache, cudaStream_t s);
cudaError_t fused_launch_tb2(const FusedArgs& a, bool gated, size_t smem, int num_sms,
                             FusedLaunchCache* cache, cudaStream_t s);
cudaError_t fused_launch_tb4(const FusedArgs& a, bool gated, size_t smem, int num_sms,
                             FusedLaunchCache* cache, cudaStream_t s);
cudaError_t fused_launch_tb8(const FusedArgs& a, bool gated, size_t smem, int num_sms,
                             FusedLaunchCache* cache, cudaStream_t s);

// Token-pair slots per staging group of k_fused<TB, .>.
__host__ __device__ constexpr int fused_pb(int tb) { return tb <= 1 ? 1 : 2; }

// Shared memory of k_fused<TB, PB>: ring, barriers, bookkeeping, reduction
// area, then the largest staged vector (or the routing block's scratch).
inline size_t fused_smem_bytes(int tb, int slots, int slot_bytes, int H, int Fs, int L, int kin, int F,
                               size_t route_bytes) {
  const int pb = fused_pb(tb);
  const int mx = H > Fs ? (H > L ? H : L) : (Fs > L ? Fs : L);
  size_t st = static_cast<size_t>(tb) * 4 * static_cast<size_t>(mx);
  const size_t e1 = static_cast<size_t>(pb) * (4 * static_cast<size_t>(kin) + 4 * static_cast<size_t>(kin / 32));
  const size_t e2 = static_cast<size_t>(pb) * (4 * static_cast<size_t>(F) + 4 * static_cast<size_t>(F / 32));
  st = st > e1 ? st : e1;
  st = st > e2 ? st : e2;
  st = st > route_bytes ? st : route_bytes;
  return static_cast<size_t>(slots) * slot_bytes + FZ_MAX_SLOTS * 8 + ((sizeof(FzShared) + 15) & ~size_t(15)) +
         NW * 8 * 4 + st;
}

}  // namespace moe
