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
// A CTA works through a list of segments, each a contiguous range of rows of
// one matrix with its dependency (a counter to wait for), the vector it reads
// (staged in shared memory) and the counter it signals when done:
//   router rows, fc1_latent_proj rows, shared gate/up rows -> dense_in
//                      (every CTA but CTA 0, which routes once the router rows
//                      are done and publishes the distinct-expert lists)
//   shared-down rows (first part)        -> sdbuf, while the routing finishes
//   expert up(+gate) rows, activation    -> hbuf  (one segment per distinct
//                      expert and group of its token rows in this CTA's share)
//   shared-down rows (second part)       -> sdbuf, over the up/down barrier
//   expert down rows                     -> pexp
//   shared-down rows (rest)              -> sdbuf
//   combine y = sum_j w_j * down_j (pick order), then fc2_latent_proj . y
//   + sdbuf + residual -> out (latent); or the combine + sdbuf + residual
//
// Weights move by bulk copies (cp.async.bulk, completion on an mbarrier):
// every warp owns a small ring of shared-memory slots and streams its own
// rows of each segment, lane 0 issuing up to `depth` chunks ahead, across
// segment boundaries whenever the next segment is known.  A warp reduces its
// rows on its own (shuffles), so the 256 threads of a CTA meet only at segment
// boundaries.  One compact executor for dense rows and one for int4 expert
// rows serve every segment, so the code stays warm in the instruction cache.
//
// Dependencies between CTAs are counters in global memory: a CTA signals
// after a CTA barrier, a gpu-scope fence and an atomic add; a waiting CTA's
// thread 0 spins on an acquire load (bounded: after FZ_SPIN_LIMIT polls the
// kernel sets the timeout bit of the status word and stops computing, but
// still signals and drains its copies, so no other CTA waits longer).  The
// launch is cooperative, so every CTA is resident and the waits end.  The last
// CTA to finish resets the counters for the next launch.  Every output element
// is computed by exactly one warp in a fixed order, so results are
// deterministic and do not depend on the other rows of the batch.
#pragma once

#include "moe_kernels.cuh"

namespace moe {

constexpr uint32_t FZ_SPIN_LIMIT = 1u << 20;
constexpr int FZ_MAX_DEPTH = 4;     // slots per warp ring
constexpr int FZ_MAX_SEGS = 32;     // segments per CTA (at most 8 dense + 2 x 9 expert)
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

// segment kinds, staged vectors and epilogues
enum : int { SK_DENSE = 0, SK_UP = 1, SK_DN = 2 };
enum : int { ST_X = 0, ST_SH = 1, ST_Y = 2, ST_EXP = 3 };
enum : int { EP_DIN = 0, EP_SD = 1, EP_OUT = 2 };

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
  // per-warp rings and the placement of the shared-down rows
  int depth;         // slots per warp ring (<= FZ_MAX_DEPTH)
  int chunk_bytes;   // slot size (multiple of 128)
  int sd_pre, sd_mid;   // percent of this CTA's shared-down rows before the expert
                        // up rows, and between the expert up and down rows
  unsigned long long* trace;   // diagnostics: [grid][FZ_TRACE] globaltimer stamps, or null
  int debug_stall;   // failure-detection test: CTA 0 first waits on a counter nothing sets
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
__device__ __forceinline__ bool fz_wait(const int* p, int target, int* status, bool ok,
                                        uint32_t limit = FZ_SPIN_LIMIT) {
  bool w = true;
  if (threadIdx.x == 0 && ok) {
    w = false;
    for (uint32_t i = 0; i < limit; ++i) {
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
// segments
// ---------------------------------------------------------------------------

// A segment runs in nsub sub-rounds, each with its own staged vector: the
// token-row passes of a dense segment, the groups of PB token pairs of an
// expert segment.
struct FzSeg {
  int kind, stage, nsub;
  int wait_ctr, wait_tgt;   // counter to wait for before the segment (-1: none)
  int sig;                  // counter to signal after it (-1: none)
  int row0, nrows;          // the CTA's rows of the matrix (dense) or of the expert (experts)
  // dense
  const char* w;
  int dt, esz, K, col0, epi;
  // experts: codes and scale/bias words of expert e (gate: q2/sb2), token pairs [pa, pa + np)
  const char* q;
  const char* sb;
  const char* q2;
  const char* sb2;
  int pa, np, R;            // all token pairs of the slot; R rows per chunk
};

struct FzShared {
  FzSeg seg[FZ_MAX_SEGS];
  volatile int nsegs;       // segments known so far (grows once, after the routing)
  int pid[8];               // expert staging: pair ids of the staged group
};

// Warp w's rows [r0, r1) of the CTA's rows of segment S, and its chunks per sub-round.
__device__ __forceinline__ void fz_warp_rows(const FzSeg& S, int w, int& r0, int& r1) {
  r0 = S.row0 + S.nrows * w / NW;
  r1 = S.row0 + S.nrows * (w + 1) / NW;
}
__device__ __forceinline__ int fz_sub_chunks(const FzSeg& S, int w, int CH) {
  int r0, r1;
  fz_warp_rows(S, w, r0, r1);
  if (r1 <= r0) return 0;
  if (S.kind == SK_DENSE) return (r1 - r0) * ((S.K * S.esz + CH - 1) / CH);
  return (r1 - r0 + S.R - 1) / S.R;
}

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
  const bool al = ((A.din_rows | A.off_shu | A.off_shg) & 3) == 0;
  // four items per thread per round, loads first, so their latencies overlap
  for (int i0 = threadIdx.x; i0 < TB * K4; i0 += 4 * NT) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * NT;
      const int t = i / K4, f4 = i - t * K4;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i >= TB * K4 || t >= tb) continue;
      const int64_t tt = t0 + t;
      if (kind == 0) {
        const uint2 h = *reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(A.x) + tt * A.H + 4 * f4);
        if (A.x_dt == DT_BF16) v[u] = make_float4(bf16lo(h.x), bf16hi(h.x), bf16lo(h.y), bf16hi(h.y));
        else v[u] = make_float4(f16lo(h.x), f16hi(h.x), f16lo(h.y), f16hi(h.y));
      } else if (kind == 1) {
        const float* du = A.dense_in + tt * A.din_rows + A.off_shu + 4 * f4;
        const float* dg = A.dense_in + tt * A.din_rows + A.off_shg + 4 * f4;
        float4 uu, gg = make_float4(0.f, 0.f, 0.f, 0.f);
        if (al) {
          uu = __ldcg(reinterpret_cast<const float4*>(du));
          if (A.act == ACT_SWIGLU) gg = __ldcg(reinterpret_cast<const float4*>(dg));
        } else {   // the shared columns start at a column that is not a multiple of 4
          uu = make_float4(__ldcg(du), __ldcg(du + 1), __ldcg(du + 2), __ldcg(du + 3));
          if (A.act == ACT_SWIGLU) gg = make_float4(__ldcg(dg), __ldcg(dg + 1), __ldcg(dg + 2), __ldcg(dg + 3));
        }
        v[u] = make_float4(act_fn(A.act, gg.x, uu.x), act_fn(A.act, gg.y, uu.y), act_fn(A.act, gg.z, uu.z),
                           act_fn(A.act, gg.w, uu.w));
      } else {
        v[u] = __ldcg(reinterpret_cast<const float4*>(A.ybuf + tt * A.L) + f4);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * NT;
      if (i >= TB * K4) break;
      const int t = i / K4, f4 = i - t * K4;
      xs4[t * K4 + swz(f4, 1)] = v[u];
    }
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
// executors (one copy each, shared by every segment)
// ---------------------------------------------------------------------------

// Bytes [boff, boff + nb) of row r of a dense matrix, in a slot, against TB
// staged token rows: partial sums into acc; on the row's last chunk the warp
// reduces them and writes the epilogue.
template <int TB>
__device__ __noinline__ void fz_dense_piece(const FusedArgs& A, const FzSeg& S, const char* slot, int r,
                                            int boff, int nb, bool last, const float4* xs4, int t0,
                                            int tb, float (&acc)[TB]) {
  const int lane = threadIdx.x & 31;
  const int K4 = S.K >> 2;
  const int np16 = nb >> 4;
  if (S.esz == 2) {
    const int f0 = boff >> 3;   // float4 index of the chunk's first element
    const int dt = S.dt;
    for (int p = lane; p < np16; p += 32) {
      float wf[8];
      cvt8(reinterpret_cast<const uint4*>(slot)[p], dt, wf);
      const int s0 = swz(f0 + 2 * p, 1), s1 = swz(f0 + 2 * p + 1, 1);
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
    const int f0 = boff >> 4;
    for (int p = lane; p < np16; p += 32) {
      const float4 w = reinterpret_cast<const float4*>(slot)[p];
      const int s0 = swz(f0 + p, 1);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const float4 a = xs4[t * K4 + s0];
        float s = acc[t];
        s = fmaf(w.x, a.x, s); s = fmaf(w.y, a.y, s); s = fmaf(w.z, a.z, s); s = fmaf(w.w, a.w, s);
        acc[t] = s;
      }
    }
  }
  if (!last) return;
  const float tot = warp_reduce_scatter<TB>(acc, lane);
#pragma unroll
  for (int t = 0; t < TB; ++t) acc[t] = 0.f;
  constexpr int LPV = 32 / TB;
  const int t = lane / LPV;
  if ((lane & (LPV - 1)) != 0 || t >= tb) return;
  const int tt = t0 + t;
  const int cc = S.col0 + (r - S.row0);
  if (S.epi == EP_DIN) {
    A.dense_in[static_cast<int64_t>(tt) * A.din_rows + cc] = tot;
  } else if (S.epi == EP_SD) {
    A.sdbuf[static_cast<int64_t>(tt) * A.H + cc] = tot;
  } else {
    const int64_t e = static_cast<int64_t>(tt) * A.H + cc;
    float v = tot;
    if (A.Fs) v += __ldcg(A.sdbuf + e);
    const float xv = ld16(A.x, e, A.x_dt);
    reinterpret_cast<unsigned short*>(A.out)[e] = st16_bits(xv + v, A.x_dt);
    if (A.delta) A.delta[e] = v;
  }
}

// Rows [r, r + n) of an expert segment in a slot: codes [n][K/2 bytes], the
// scale/bias words at sb (and the gate's at q2 / sb2), against the np staged
// token rows of the segment.  One warp; a lane takes 32-code pieces.
template <int PB, bool GATED>
__device__ __noinline__ void fz_expert_rows(const ExpertArgs& X, const char* q, const uint32_t* sb,
                                            const char* q2, const uint32_t* sb2, int n, int r,
                                            const float4* xs4, const int* pid_s, int np) {
  const int lane = threadIdx.x & 31;
  const int K = X.K, K4 = K >> 2, nchunk = K >> 5, ngr = K / X.G;
  const float* xsum = reinterpret_cast<const float*>(xs4 + PB * K4);
  constexpr int NV = 2 * PB;
  constexpr int LPV = 32 / NV;
#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    float acc[PB], accg[PB];
#pragma unroll
    for (int pp = 0; pp < PB; ++pp) { acc[pp] = 0.f; accg[pp] = 0.f; }
    const uint4* qr = reinterpret_cast<const uint4*>(q + static_cast<int64_t>(i) * (K >> 1));
    const uint32_t* sr = sb + i * ngr;
#pragma unroll 1
    for (int cc = lane; cc < nchunk; cc += 32) {
      const uint4 w = qr[cc];
      float sc, bi;
      sb_decode(sr[(cc << 5) / X.G], X.s_dt, sc, bi);
      const float s16 = 16.f * sc, bb = bi - s16;
      uint4 wg = make_uint4(0u, 0u, 0u, 0u);
      float sg16 = 0.f, bbg = 0.f;
      if (GATED) {
        wg = reinterpret_cast<const uint4*>(q2 + static_cast<int64_t>(i) * (K >> 1))[cc];
        float sg, bg;
        sb_decode(sb2[i * ngr + (cc << 5) / X.G], X.s_dt, sg, bg);
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
        X.out[static_cast<int64_t>(pid_s[pp]) * X.n_rows + r + i] = val;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// Geometry of chunk ci (within a sub-round) of warp w in segment S: dense ->
// row, byte offset and bytes; expert -> first row and rows.
struct FzChunk {
  int r, boff, nb, n;
  bool last;   // dense: the row's last chunk
};
__device__ __forceinline__ FzChunk fz_chunk(const FzSeg& S, int w, int ci, int CH) {
  int r0, r1;
  fz_warp_rows(S, w, r0, r1);
  FzChunk C;
  if (S.kind == SK_DENSE) {
    const int rb = S.K * S.esz, per = (rb + CH - 1) / CH;
    const int ri = ci / per, k = ci - ri * per;
    C.r = r0 + ri;
    C.boff = k * CH;
    C.nb = min(CH, rb - C.boff);
    C.n = 1;
    C.last = k == per - 1;
  } else {
    C.r = r0 + ci * S.R;
    C.n = min(S.R, r1 - C.r);
    C.boff = 0;
    C.nb = 0;
    C.last = true;
  }
  return C;
}

template <int TB, int PB, bool GATED>
__global__ void __launch_bounds__(NT, TB >= 8 ? 1 : 2) k_fused(const __grid_constant__ FusedArgs A) {
  extern __shared__ __align__(128) char fz_smem_raw[];
  const int c = blockIdx.x, G = gridDim.x;
  const int D = A.depth, CH = A.chunk_bytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  char* rings = fz_smem_raw;                                             // [NW][D][CH]
  uint64_t* bars = reinterpret_cast<uint64_t*>(rings + static_cast<size_t>(NW) * D * CH);   // [NW][FZ_MAX_DEPTH]
  FzShared* sh = reinterpret_cast<FzShared*>(bars + NW * FZ_MAX_DEPTH);
  float4* xs4 = reinterpret_cast<float4*>(reinterpret_cast<char*>(sh) + ((sizeof(FzShared) + 15) & ~size_t(15)));
  char* ring = rings + static_cast<size_t>(warp) * D * CH;
  uint64_t* bar = bars + warp * FZ_MAX_DEPTH;
  int* sync = A.sync;
  const int T = A.T;
  bool ok = true;
  auto stamp = [&](int i) {
    if (A.trace && tid == 0) A.trace[c * FZ_TRACE + i] = global_ns();
  };
  // diagnostics: CTA 1's warp 7 (which holds router row 0) at points of the first segment
  auto dstamp = [&](int i) {
    if (A.trace && c == 1 && tid == 224) A.trace[FZ_TRACE + 13 + i] = global_ns();
  };
  stamp(0);
  const int passes = (T + TB - 1) / TB;

  // ---- the static segments (thread 0) ----
  if (tid == 0) {
    int ns = 0;
    auto dense = [&](const void* w, int dt, int K, int64_t rb, int64_t re, int col0, int epi, int stage,
                     int wctr, int wtgt, int sig) {
      FzSeg& S = sh->seg[ns++];
      S.kind = SK_DENSE; S.stage = stage; S.nsub = passes;
      S.wait_ctr = wctr; S.wait_tgt = wtgt; S.sig = sig;
      S.row0 = static_cast<int>(rb); S.nrows = static_cast<int>(re - rb);
      S.w = static_cast<const char*>(w); S.dt = dt; S.esz = dt == DT_FP32 ? 4 : 2; S.K = K;
      S.col0 = col0 + static_cast<int>(rb); S.epi = epi;
      S.q = S.sb = S.q2 = S.sb2 = nullptr; S.pa = 0; S.np = 0; S.R = 1;
    };
    if (c > 0) {
      // CTA 0 routes; the others share the rows that read x
      const int gd = G - 1, cd = c - 1;
      int64_t b, e;
      span(A.E, cd, gd, b, e);
      dense(A.router_w, A.router_dt, A.H, b, e, 0, EP_DIN, ST_X, -1, 0, FZ_ROUTER);
      span(A.L, cd, gd, b, e);
      dense(A.fc1, A.x_dt, A.H, b, e, A.off_fc1, EP_DIN, ST_X, -1, 0, FZ_FC1);
      span(A.Fs, cd, gd, b, e);
      if (A.act == ACT_SWIGLU) dense(A.sh_gate, A.x_dt, A.H, b, e, A.off_shg, EP_DIN, ST_X, -1, 0, -1);
      dense(A.sh_up, A.x_dt, A.H, b, e, A.off_shu, EP_DIN, ST_X, -1, 0, FZ_DIN);
    }
    // the first part of this CTA's shared-down rows
    if (A.Fs) {
      int64_t b, e;
      span(A.H, c, G, b, e);
      const int64_t n1 = (e - b) * A.sd_pre / 100;
      dense(A.sh_down, A.x_dt, A.Fs, b, b + n1, 0, EP_SD, ST_SH, FZ_DIN, G - 1, -1);
    }
    sh->nsegs = ns;
    for (int w = 0; w < NW; ++w)
      for (int d = 0; d < FZ_MAX_DEPTH; ++d) fz_mbar_init(bars + w * FZ_MAX_DEPTH + d, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  dstamp(0);

  // ---- per-warp ring: lane 0 issues chunks in segment order ----
  int p_seg = 0, p_ci = 0;          // producer cursor (lane 0)
  uint32_t issued = 0, consumed = 0;
  // The router rows go first and alone: the routing (on the critical path)
  // then does not wait behind every other warp's first chunks.
  int seg_limit = c > 0 ? 1 : FZ_MAX_SEGS;
  auto produce = [&]() {
    if (lane != 0) return;
    const int nk = min(static_cast<int>(sh->nsegs), seg_limit);
    while (issued - consumed < static_cast<uint32_t>(D) && p_seg < nk) {
      const FzSeg& S = sh->seg[p_seg];
      const int per = fz_sub_chunks(S, warp, CH);
      if (p_ci >= per * S.nsub) { ++p_seg; p_ci = 0; continue; }
      const FzChunk C = fz_chunk(S, warp, p_ci % per, CH);
      const int sl = issued % D;
      char* dst = ring + static_cast<size_t>(sl) * CH;
      uint64_t* b = bar + sl;
      if (S.kind == SK_DENSE) {
        fz_expect_tx(b, C.nb);
        fz_bulk(dst, S.w + static_cast<int64_t>(C.r) * S.K * S.esz + C.boff, C.nb, b);
      } else {
        const ExpertArgs& X = S.kind == SK_UP ? A.up : A.dn;
        const int ngr = X.K / X.G;
        const uint32_t qb = static_cast<uint32_t>(C.n) * (X.K / 2);
        const uint64_t sa = reinterpret_cast<uint64_t>(S.sb + static_cast<int64_t>(C.r) * ngr * 4);
        const uint64_t sa0 = sa & ~uint64_t(15);
        const uint32_t sbb = static_cast<uint32_t>((sa + static_cast<uint64_t>(C.n) * ngr * 4 - sa0 + 15) & ~uint64_t(15));
        uint32_t tx = qb + sbb, sbb2 = 0;
        uint64_t sa2_0 = 0;
        if (S.q2) {
          const uint64_t sa2 = reinterpret_cast<uint64_t>(S.sb2 + static_cast<int64_t>(C.r) * ngr * 4);
          sa2_0 = sa2 & ~uint64_t(15);
          sbb2 = static_cast<uint32_t>((sa2 + static_cast<uint64_t>(C.n) * ngr * 4 - sa2_0 + 15) & ~uint64_t(15));
          tx += qb + sbb2;
        }
        fz_expect_tx(b, tx);
        fz_bulk(dst, S.q + static_cast<int64_t>(C.r) * (X.K / 2), qb, b);
        fz_bulk(dst + qb, reinterpret_cast<const void*>(sa0), sbb, b);
        if (S.q2) {
          fz_bulk(dst + qb + sbb, S.q2 + static_cast<int64_t>(C.r) * (X.K / 2), qb, b);
          fz_bulk(dst + 2 * qb + sbb, reinterpret_cast<const void*>(sa2_0), sbb2, b);
        }
      }
      ++issued;
      ++p_ci;
    }
  };
  produce();
  dstamp(1);

  // ---- routing (CTA 0) ----
  if (c == 0) {
    // failure-detection test: a short wait on a word that nothing sets runs
    // out, the timeout is recorded and the launch completes without routing
    if (A.debug_stall) ok = fz_wait(sync + FZ_EXIT * FZ_SYNC_STRIDE + 8, 1, A.status, ok, 1u << 12);
    ok = fz_wait(sync + FZ_ROUTER * FZ_SYNC_STRIDE, G - 1, A.status, ok);
    stamp(1);
    if (ok)
      route_block(A.route, reinterpret_cast<int*>(xs4));
    else if (tid == 0)
      A.route.meta[0] = 0;   // no routing: the expert segments find no work
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicExch(sync + FZ_ROUTED * FZ_SYNC_STRIDE, 1);
    }
    stamp(2);
  }

  // the segments after the routing (thread 0, after the routing flag)
  auto build_rest = [&]() {
    int ns = sh->nsegs;
    auto add = [&]() -> FzSeg* {
      if (ns >= FZ_MAX_SEGS) { atomicOr(A.status, STATUS_TIMEOUT); return nullptr; }   // not reachable
      return &sh->seg[ns++];
    };
    auto experts = [&](int kind, const ExpertArgs& X, bool gated_up, int wctr, int wtgt, int sig) {
      const int nu = min(max(__ldcg(X.meta), 0), X.umax);
      const int ngr = X.K / X.G;
      const int rowb = (gated_up ? 2 : 1) * (X.K / 2 + ngr * 4);
      const int R = max(1, min(32, (CH - (gated_up ? 32 : 16)) / rowb));
      int64_t b, e;
      span(static_cast<int64_t>(nu) * X.n_rows, c, G, b, e);
      FzSeg* last = nullptr;
      while (b < e) {
        const int u = static_cast<int>(b / X.n_rows);
        const int n0 = static_cast<int>(b - static_cast<int64_t>(u) * X.n_rows);
        const int n1 = static_cast<int>(min(static_cast<int64_t>(X.n_rows), n0 + (e - b)));
        const int64_t ex = __ldcg(X.meta + 1 + u);
        const int pa = __ldcg(X.meta + 1 + X.umax + u), pe = __ldcg(X.meta + 2 + X.umax + u);
        FzSeg* S = add();
        if (!S) break;
        S->kind = kind; S->stage = ST_EXP; S->nsub = max(1, (pe - pa + PB - 1) / PB);
        S->wait_ctr = wctr; S->wait_tgt = wtgt; S->sig = -1;
        S->row0 = n0; S->nrows = pe > pa ? n1 - n0 : 0;
        S->w = nullptr; S->dt = 0; S->esz = 0; S->K = X.K; S->col0 = u; S->epi = 0;
        S->q = reinterpret_cast<const char*>(X.q) + ex * X.n_rows * (X.K / 2);
        S->sb = reinterpret_cast<const char*>(X.sb) + ex * X.n_rows * ngr * 4;
        S->q2 = gated_up ? reinterpret_cast<const char*>(X.q_gate) + ex * X.n_rows * (X.K / 2) : nullptr;
        S->sb2 = gated_up ? reinterpret_cast<const char*>(X.sb_gate) + ex * X.n_rows * ngr * 4 : nullptr;
        S->pa = pa; S->np = max(0, pe - pa); S->R = R;
        last = S;
        b += n1 - n0;
      }
      if (!last) {
        // no rows here: an empty segment carries the signal
        last = add();
        if (!last) return;
        last->kind = kind; last->stage = -1; last->nsub = 1; last->wait_ctr = -1; last->wait_tgt = 0;
        last->row0 = 0; last->nrows = 0; last->w = nullptr; last->dt = 0; last->esz = 0; last->K = X.K;
        last->col0 = 0; last->epi = 0; last->q = last->sb = last->q2 = last->sb2 = nullptr;
        last->pa = 0; last->np = 0; last->R = 1;
      }
      last->sig = sig;
    };
    auto sdpart = [&](int pct0, int pct1, int sig) {
      int64_t b, e;
      span(A.H, c, G, b, e);
      const int64_t n = e - b;
      FzSeg* S = add();
      if (!S) return;
      S->kind = SK_DENSE; S->stage = ST_SH; S->nsub = passes;
      S->wait_ctr = FZ_DIN; S->wait_tgt = G - 1; S->sig = sig;
      S->row0 = static_cast<int>(b + n * pct0 / 100); S->nrows = static_cast<int>(n * pct1 / 100 - n * pct0 / 100);
      S->w = static_cast<const char*>(A.sh_down); S->dt = A.x_dt; S->esz = 2; S->K = A.Fs;
      S->col0 = S->row0; S->epi = EP_SD;
      S->q = S->sb = S->q2 = S->sb2 = nullptr; S->pa = 0; S->np = 0; S->R = 1;
    };
    experts(SK_UP, A.up, GATED, A.L ? FZ_FC1 : -1, G - 1, FZ_UP);
    const int pre = A.sd_pre, mid = min(100, A.sd_pre + A.sd_mid);
    if (A.Fs) sdpart(pre, mid, -1);
    experts(SK_DN, A.dn, false, FZ_UP, G, FZ_DN);
    if (A.Fs) sdpart(mid, 100, FZ_SD);
    if (A.L) {
      int64_t b, e;
      span(A.H, c, G, b, e);
      FzSeg* S = add();
      if (S) {
        S->kind = SK_DENSE; S->stage = ST_Y; S->nsub = passes;
        S->wait_ctr = FZ_COMB; S->wait_tgt = G; S->sig = -1;
        S->row0 = static_cast<int>(b); S->nrows = static_cast<int>(e - b);
        S->w = static_cast<const char*>(A.fc2); S->dt = A.x_dt; S->esz = 2; S->K = A.L;
        S->col0 = S->row0; S->epi = EP_OUT;
        S->q = S->sb = S->q2 = S->sb2 = nullptr; S->pa = 0; S->np = 0; S->R = 1;
      }
    }
    __threadfence_block();
    sh->nsegs = ns;
  };

  // ---- consume the segments ----
  uint32_t waited = 0;      // counters already waited for (bit per counter)
  int staged = -1;          // what the staging area holds
  bool comb_done = false;
  auto need = [&](int ctr, int target) {
    if (ctr < 0 || (waited & (1u << ctr))) return;
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

  bool rest_built = false;
  for (int si = 0;; ++si) {
    if (si == sh->nsegs) {
      if (rest_built) break;
      // the remaining segments need the routing
      need(FZ_ROUTED, 1);
      if (tid == 0 && ok) build_rest();
      __syncthreads();
      rest_built = true;
      if (!ok) break;
      produce();
      if (si == sh->nsegs) break;
    }
    const FzSeg& S = sh->seg[si];
    if (si == 0 || sh->seg[si - 1].kind != S.kind) {
      if (S.kind == SK_UP) stamp(4);
      if (S.kind == SK_DN) stamp(7);
    }
    // dependencies
    if (S.stage == ST_Y && !comb_done) combine();
    if (S.stage == ST_Y && A.Fs) need(FZ_SD, G);
    need(S.wait_ctr, S.wait_tgt);
    const int per = fz_sub_chunks(S, warp, CH);
    for (int sub = 0; sub < S.nsub; ++sub) {
      // the staged vector of the sub-round
      const int t0 = sub * TB;
      const int pa = S.pa + sub * PB, np = min(PB, S.np - sub * PB);
      if (S.stage >= 0) {
        const int tag = S.stage == ST_EXP ? (0x40000 + si * 256 + sub) : (S.stage * 256 + sub);
        if (tag != staged) {
          __syncthreads();   // every warp is done with the previous vector
          if (S.stage == ST_EXP) {
            fz_stage_expert<PB>(S.kind == SK_UP ? A.up : A.dn, pa, np, xs4, sh->pid);
          } else {
            fz_stage_dense<TB>(A, S.stage == ST_X ? 0 : S.stage == ST_SH ? 1 : 2, t0, min(TB, T - t0), S.K,
                               xs4);
            __syncthreads();
          }
          staged = tag;
        }
      }
      if (si == 0) dstamp(2);
      // this warp's chunks of the sub-round
      float acc[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[t] = 0.f;
      for (int ci = 0; ci < per; ++ci) {
        const int sl = consumed % D;
        // (a copy that never lands only skips this warp's work: control flow
        // stays uniform, the status word records it)
        const bool wok = fz_mbar_wait(bar + sl, (consumed / D) & 1);
        if (si == 0) dstamp(3 + 2 * min(ci, 2));
        if (!wok && lane == 0) atomicOr(A.status, STATUS_TIMEOUT);
        const char* slot = ring + static_cast<size_t>(sl) * CH;
        const FzChunk C = fz_chunk(S, warp, ci, CH);
        if (ok && wok) {
          if (S.kind == SK_DENSE) {
            fz_dense_piece<TB>(A, S, slot, C.r, C.boff, C.nb, C.last, xs4, t0, min(TB, T - t0), acc);
          } else {
            const ExpertArgs& X = S.kind == SK_UP ? A.up : A.dn;
            const int ngr = X.K / X.G;
            const uint32_t qb = static_cast<uint32_t>(C.n) * (X.K / 2);
            const uint64_t sa = reinterpret_cast<uint64_t>(S.sb + static_cast<int64_t>(C.r) * ngr * 4);
            const uint32_t off = static_cast<uint32_t>(sa & 15);
            const uint32_t sbb = static_cast<uint32_t>((off + static_cast<uint64_t>(C.n) * ngr * 4 + 15) & ~uint64_t(15));
            const uint32_t* sbp = reinterpret_cast<const uint32_t*>(slot + qb + off);
            if (S.kind == SK_UP && S.q2) {
              const uint64_t sa2 = reinterpret_cast<uint64_t>(S.sb2 + static_cast<int64_t>(C.r) * ngr * 4);
              fz_expert_rows<PB, GATED>(X, slot, sbp, slot + qb + sbb,
                                        reinterpret_cast<const uint32_t*>(slot + 2 * qb + sbb + (sa2 & 15)),
                                        C.n, C.r, xs4, sh->pid, np);
            } else {
              fz_expert_rows<PB, false>(X, slot, sbp, nullptr, nullptr, C.n, C.r, xs4, sh->pid, np);
            }
          }
        }
        __syncwarp();   // every lane is done with the slot
        if (si == 0) dstamp(4 + 2 * min(ci, 2));
        ++consumed;
        produce();
      }
    }
    if (si == 0 && seg_limit == 1) {
      seg_limit = FZ_MAX_SEGS;
      produce();
    }
    if (S.sig >= 0) {
      __syncthreads();
      if (si == 0) dstamp(9);
      if (tid == 0) fz_post(sync + S.sig * FZ_SYNC_STRIDE);
      if (S.sig == FZ_DIN) stamp(3);
      if (S.sig == FZ_UP) stamp(5);
      if (S.sig == FZ_DN) stamp(8);
      if (S.sig == FZ_SD) stamp(9);
    }
  }
  stamp(10);

  // ---- tail: the combine (CTAs without fc2 rows) and the non-latent output ----
  if (A.L) {
    if (!comb_done) combine();
  } else {
    need(FZ_DN, G);
    if (A.Fs) need(FZ_SD, G);
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
__host__ __device__ constexpr int fused_pb(int tb) { return tb <= 1 ? 1 : (tb <= 4 ? 2 : 4); }

// Shared memory of k_fused<TB, PB>: warp rings, their barriers, the segment
// list, then the largest staged vector (or the routing block's scratch).
inline size_t fused_smem_bytes(int tb, int depth, int chunk_bytes, int H, int Fs, int L, int kin, int F,
                               size_t route_bytes) {
  const int pb = fused_pb(tb);
  const int mx = H > Fs ? (H > L ? H : L) : (Fs > L ? Fs : L);
  size_t st = static_cast<size_t>(tb) * 4 * static_cast<size_t>(mx);
  const size_t e1 = static_cast<size_t>(pb) * (4 * static_cast<size_t>(kin) + 4 * static_cast<size_t>(kin / 32));
  const size_t e2 = static_cast<size_t>(pb) * (4 * static_cast<size_t>(F) + 4 * static_cast<size_t>(F / 32));
  st = st > e1 ? st : e1;
  st = st > e2 ? st : e2;
  st = st > route_bytes ? st : route_bytes;
  return static_cast<size_t>(NW) * depth * chunk_bytes + NW * FZ_MAX_DEPTH * 8 +
         ((sizeof(FzShared) + 15) & ~size_t(15)) + st;
}

}  // namespace moe
