// Dense projections of the gemv path on warp-level tensor-core MMAs (sm_103a).
//
// The layer's bf16 matrices -- router, fc1_latent_proj and the shared expert's
// gate/up in the pass over x; fc2_latent_proj and the shared expert's down in
// the output pass -- contracted with the T token rows.  On the CUDA cores every
// weight costs a conversion and one fma per token row, and the staged rows are
// re-read from shared memory per fma; here a warp computes a 16-row tile with
// mma.sync m16n8k16 (bf16 operands, fp32 accumulators):
//
//   * A comes straight from the weights: create time re-lays each matrix
//     (k_tile_dense) so that a lane's four fragment registers of a 16-column
//     block are one 16-byte word (rows g, g + 8; columns 2t, 2t + 1, 2t + 8,
//     2t + 9, the fragment order of the instruction);
//   * B holds the token rows in the same k order: a 16-bit input as one bf16
//     column a token (exact), an fp32 input as two, hi = bf16(x) and
//     lo = bf16(x - hi) (about 2^-17 relative), summed after the MMAs;
//   * the products of bf16 values are exact in fp32, and each output element
//     depends on its own token's column only, so a row gives the same bits
//     whatever the batch.
//
// Weights stream through a private bulk-copy ring per warp, as in the expert
// kernel (moe_expert_mma.cuh): chunks of CK 64-column blocks of one 16-row tile,
// each 2 KB per block, complete on the stage's mbarrier (bounded waits).  The
// K range of a tile is split over KS warps by the matrix shape alone, and their
// partial sums are added in a fixed order through shared memory.
//
// The pass over x can carry the routing: CTA 0 holds no tiles; it warms the
// top-k code with a dry run while the CTAs holding the router rows compute
// them, waits (bounded) for their count, and routes.
#pragma once

#include <cuda_bf16.h>

#include "moe_kernels.cuh"
#include "moe_expert_bulk.cuh"   // eb_smem, eb_bulk, eb_wait
#include "moe_expert_mma.cuh"    // mma_16816, pack_bf16x2, em_ld16, EM_WARPS

namespace moe {

// Consecutive output rows of one matrix per part of the reduction axis.
struct DmSeg {
  const uint4* w[2];   // tiled weights of each part ([rows/16][K_p/16][32] words) or null
  int rows;            // output rows
  int col0;            // first output column (fp32 mode) / row (final mode)
};

// One input part of the reduction axis, for token row t:
//   mode 0: in[t * ld + off + k] (16-bit or fp32)
//   mode 1: act(gate, up) of the fp32 dense pass: gate at off_g, up at off + k
struct DmIn {
  const void* p;
  int dt, ld, off, off_g, mode, act;
  int K;   // columns (multiple of 64)
};

struct DmArgs {
  DmSeg seg[4];
  int nseg;
  int seg_t0[5];       // first tile of each segment (prefix over seg rows / 16), [nseg] = total
  DmIn in[2];
  int nparts;
  int T;
  // ring plan (host-chosen): chunks of ck 64-column blocks, ns stages a warp,
  // tokens per pass tp, warps per tile ks
  int ck, ns, tp, ks;
  int tile_ctas;       // CTAs that hold tiles (grid - 1 with a routing CTA)
  // output: fp32 columns (mode 0) or the layer output (mode 1)
  int out_mode;
  float* outf;         // mode 0: [T, out_ld]
  int out_ld;
  const void* x;       // mode 1: residual [T, H], act dtype
  int x_dt;
  void* out;           // mode 1: [T, H]
  float* delta;        // mode 1: [T, H] fp32 or null
  const float* y_add;  // mode 1: [T, H] routed output added directly, or null
  int H;
  int* status;
  // routing in CTA 0 (pass over x): its tiles' CTAs count themselves on route_counter
  int fuse_route;
  int route_ctas;      // CTAs 1..route_ctas hold the router rows (segment 0)
  int* route_counter;
  int debug_stall;
  RouteArgs route;
  int prefetch;        // issue the first copies before waiting for the previous kernel
  unsigned long long* trace;
};

struct DmPlan {
  int ck, ns, tp, ks, split;
  int stage_bytes, b_bytes, red_off, ring_off, bar_off;
  int smem;
};

__host__ __device__ inline int dm_ntp(int tp, int split) { return tp / (split ? 4 : 8); }

__host__ __device__ inline DmPlan dm_plan(int K, int ck, int ns, int tp, int ks, int split) {
  DmPlan p;
  p.ck = ck;
  p.ns = ns;
  p.tp = tp;
  p.ks = ks;
  p.split = split;
  p.stage_bytes = ck * 2048;
  p.b_bytes = dm_ntp(tp, split) * (K / 16) * 256;
  p.red_off = p.b_bytes;
  p.ring_off = p.red_off + (ks > 1 ? 2 * EM_WARPS * 4 * dm_ntp(tp, split) * 32 * 4 : 0);
  p.bar_off = p.ring_off + EM_WARPS * ns * p.stage_bytes;
  p.smem = p.bar_off + EM_WARPS * ns * 8;
  return p;
}

// Tiles [*tb, *te) of tile CTA c: with routing, CTAs 0 .. rc - 1 share the
// router's tiles [0, t1) (so that they finish early and the routing overlaps
// the rest of the pass) and the others share [t1, ntot); without, all share
// [0, ntot) evenly.
__host__ __device__ inline void dm_cta_tiles(int ntot, int t1, int rc, int ctas, int c, int* tb, int* te) {
  if (t1 > 0 && rc > 0 && rc < ctas) {
    if (c < rc) {
      *tb = static_cast<int>(static_cast<int64_t>(c) * t1 / rc);
      *te = static_cast<int>(static_cast<int64_t>(c + 1) * t1 / rc);
    } else {
      *tb = t1 + static_cast<int>(static_cast<int64_t>(c - rc) * (ntot - t1) / (ctas - rc));
      *te = t1 + static_cast<int>(static_cast<int64_t>(c - rc + 1) * (ntot - t1) / (ctas - rc));
    }
  } else {
    *tb = static_cast<int>(static_cast<int64_t>(c) * ntot / ctas);
    *te = static_cast<int>(static_cast<int64_t>(c + 1) * ntot / ctas);
  }
}

// The part holding 64-column block kc, and that part's end (in blocks).
__device__ __forceinline__ int dm_part(const DmArgs& A, int kc, int* pend) {
  const int k0 = A.in[0].K >> 6;
  if (A.nparts > 1 && kc >= k0) { *pend = k0 + (A.in[1].K >> 6); return 1; }
  *pend = k0;
  return 0;
}

// NTP: n-tiles of accumulators (tokens per pass: 4 NTP split, 8 NTP not).
// SPLIT: fp32 (or fp16) inputs as hi/lo bf16 column pairs; off: bf16 inputs.
template <int NTP, bool SPLIT>
__global__ void __launch_bounds__(EM_NT, NTP == 1 ? 2 : 1) k_dense_mma(const __grid_constant__ DmArgs A) {
  extern __shared__ __align__(128) unsigned char dm_smem[];
  constexpr int TPN = SPLIT ? 4 : 8;   // tokens an n-tile
  const int K0 = A.in[0].K, K = K0 + (A.nparts > 1 ? A.in[1].K : 0);
  const int nkc = K >> 6, nkb = K >> 4;
  const DmPlan P = dm_plan(K, A.ck, A.ns, A.tp, A.ks, SPLIT);
  const int CK = P.ck, NS = P.ns, KS = P.ks;
  uint2* bfrag = reinterpret_cast<uint2*>(dm_smem);
  float* red = reinterpret_cast<float*>(dm_smem + P.red_off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  unsigned char* ring = dm_smem + P.ring_off + warp * NS * P.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dm_smem + P.bar_off) + warp * NS;
  cta_stamp(A.trace, 0);

  const bool route_cta = A.fuse_route && blockIdx.x == 0;
  const int cta = A.fuse_route ? static_cast<int>(blockIdx.x) - 1 : static_cast<int>(blockIdx.x);
  int tb = 0, te = 0;
  dm_cta_tiles(A.seg_t0[A.nseg], A.fuse_route ? A.seg_t0[1] : 0, A.route_ctas, A.tile_ctas, cta, &tb, &te);
  if (route_cta) tb = te = 0;
  const bool holds_router = A.fuse_route && !route_cta && cta < A.route_ctas;
  const int npass = (A.T + P.tp - 1) / P.tp;

  // KS warps a tile (K split by the shape alone), EM_WARPS / KS tile slots
  const int nslot = EM_WARPS / KS, slot = warp / KS, ks = warp - slot * KS;
  const int kc_lo = ks * nkc / KS, kc_hi = (ks + 1) * nkc / KS;
  const int my_tiles = (te - tb > slot) ? (te - tb - slot + nslot - 1) / nslot : 0;
  // chunks of this warp's K range: at most CK blocks, never across the parts
  int nit = 0;
  for (int kc = kc_lo; kc < kc_hi;) {
    int pend;
    (void)dm_part(A, kc, &pend);
    kc = min(kc + CK, min(kc_hi, pend));
    ++nit;
  }
  const int total = route_cta ? 0 : my_tiles * nit * npass;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(eb_smem(bars + s)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  int iss_ti = 0, iss_kc = kc_lo, iss_s = 0, issued = 0;   // lane 0's issue position
  auto issue_next = [&]() {
    const int gt = tb + slot + nslot * iss_ti;
    int si = 0;
    while (si + 1 < A.nseg && gt >= A.seg_t0[si + 1]) ++si;
    const int lt = gt - A.seg_t0[si];
    int pend;
    const int p = dm_part(A, iss_kc, &pend);
    const int ckt = min(CK, min(kc_hi, pend) - iss_kc);
    const int kcp = iss_kc - (p ? (K0 >> 6) : 0);   // block within the part
    const int kbp = A.in[p].K >> 4;                  // 16-column blocks of the part
    const uint4* src = A.seg[si].w[p] + (static_cast<int64_t>(lt) * kbp + 4 * kcp) * 32;
    const uint32_t bar = eb_smem(bars + iss_s);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(ckt * 2048u) : "memory");
    eb_bulk(eb_smem(ring + iss_s * P.stage_bytes), src, ckt * 2048u, bar);
    ++issued;
    if (++iss_s == NS) iss_s = 0;
    iss_kc += ckt;
    if (iss_kc == kc_hi) { iss_kc = kc_lo; if (++iss_ti == my_tiles) iss_ti = 0; }
  };
  // the weights need nothing from the previous kernel: with `prefetch` their
  // first copies go out before the wait
  if (A.prefetch && lane == 0)
    while (issued < min(NS, total)) issue_next();
  if (route_cta) {
    // The first run of the top-k code is slow (its instructions come from a
    // cold L2), so the routing CTA runs its phases once, one per warp at once,
    // on whatever the buffers hold, writing nothing, before it waits for the
    // previous kernel: that run reads no value this launch depends on and
    // stores nothing.
    RouteArgs D = A.route;
    D.dry = 1;
    D.topk_only = D.T * D.k > 32;
    route_warm(D, reinterpret_cast<int*>(dm_smem));
    cta_stamp(A.trace, 4);
  }
  griddep_wait();
  griddep_launch();
  cta_stamp(A.trace, 1);
  if (!A.prefetch && lane == 0)
    while (issued < min(NS, total)) issue_next();

  if (route_cta) {
    // wait for the router rows, route
    __syncthreads();
    if (threadIdx.x == 0) {
      const bool ok = spin_until_geq(A.route_counter, A.route_ctas + (A.debug_stall ? 1 : 0));
      if (!ok) atomicOr(A.route.status, STATUS_TIMEOUT);
      __threadfence();
    }
    __syncthreads();
    cta_stamp(A.trace, 5);
    route_block(A.route, reinterpret_cast<int*>(dm_smem));
    __syncthreads();
    if (threadIdx.x == 0) *A.route_counter = 0;
    cta_stamp(A.trace, 3);
    return;
  }

  bool ok = true;
  int gi = 0, gi_fail = 0, cs = 0;   // items consumed; the next one's stage
  uint32_t phase = 0;
  for (int pass = 0; pass < npass; ++pass) {
    const int T0 = pass * P.tp, ntok = min(P.tp, A.T - T0), nnt = (ntok + TPN - 1) / TPN;
    if (pass) __syncthreads();   // every warp is done with the previous pass's B
    // ---- stage B: token tl -> n-tile tl / TPN, column tl % TPN (or the hi/lo
    // pair 2 (tl % 4), + 1); thread i takes block kb of token tl (kb fastest)
    // (the padding columns of the last n-tile are left as they are: an MMA
    // output column depends on its own B column only, and theirs are not stored)
    const int nblk = ntok * nkb;
#pragma unroll 2
    for (int i = threadIdx.x; i < nblk; i += EM_NT) {
      const int tl = i / nkb, kb = i - tl * nkb;
      float v[16];
      {
        const int tt = T0 + tl;
        const int p = (A.nparts > 1 && kb >= (K0 >> 4)) ? 1 : 0;
        const DmIn& I = A.in[p];
        const int kk = 16 * kb - (p ? K0 : 0);
        if (I.mode == 0) {
          const int64_t base = static_cast<int64_t>(tt) * I.ld + I.off + kk;
          const bool vec = I.dt == DT_FP32 ? ((I.ld | I.off) & 3) == 0 : ((I.ld | I.off) & 7) == 0;
          em_ld16(I.p, I.dt, base, vec, v);
        } else {
          const float* di = static_cast<const float*>(I.p) + static_cast<int64_t>(tt) * I.ld;
          float uv[16], gvv[16];
          const bool vec = ((I.ld | I.off | I.off_g) & 3) == 0;
          em_ld16(di, DT_FP32, I.off + kk, vec, uv);
          if (I.act == ACT_SWIGLU) em_ld16(di, DT_FP32, I.off_g + kk, vec, gvv);
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = act_fn(I.act, I.act == ACT_SWIGLU ? gvv[q] : 0.f, uv[q]);
        }
      }
      uint2* dst = bfrag + (static_cast<int64_t>(tl / TPN) * nkb + kb) * 32;
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        // lane (column, tt): k = 2 tt, 2 tt + 1 and 2 tt + 8, 2 tt + 9
        if (SPLIT) {
          float hi[4], lo[4];
          const int ks4[4] = {2 * tt, 2 * tt + 1, 2 * tt + 8, 2 * tt + 9};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hi[j] = __bfloat162float(__float2bfloat16_rn(v[ks4[j]]));
            lo[j] = v[ks4[j]] - hi[j];
          }
          const int c = 2 * (tl & 3);
          dst[c * 4 + tt] = make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]));
          dst[(c + 1) * 4 + tt] = make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
        } else {
          const int c = tl & 7;
          dst[c * 4 + tt] = make_uint2(pack_bf16x2(v[2 * tt], v[2 * tt + 1]),
                                       pack_bf16x2(v[2 * tt + 8], v[2 * tt + 9]));
        }
      }
    }
    __syncthreads();
    if (pass == 0) cta_stamp(A.trace, 6);

    // ---- this warp's tiles
    const uint2* bl = bfrag + lane;
    float acc[2][NTP][4], y[NTP][4];
    for (int ti = 0; ti < my_tiles; ++ti) {
      const int gt = tb + slot + nslot * ti;
#pragma unroll
      for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[0][nt][r] = acc[1][nt][r] = 0.f;
      int kc = kc_lo;
      for (int it = 0; it < nit; ++it, ++gi) {
        int pend;
        (void)dm_part(A, kc, &pend);
        const int ckt = min(CK, min(kc_hi, pend) - kc);
        if (ok && !eb_wait(eb_smem(bars + cs), phase)) {
          ok = false;
          gi_fail = gi;
          if (lane == 0) atomicOr(A.status, STATUS_TIMEOUT);
        }
        if (gi == 0) cta_stamp(A.trace, 7);
        if (ok) {
          const uint4* aw = reinterpret_cast<const uint4*>(ring + cs * P.stage_bytes) + lane;
#pragma unroll 1
          for (int c = 0; c < ckt; ++c) {
            const uint2* bk = bl + static_cast<int64_t>(kc + c) * 4 * 32;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 w = aw[(c * 4 + j) * 32];
              const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int nt = 0; nt < NTP; ++nt) {
                if (nt < nnt) {
                  const uint2 b = bk[(static_cast<int64_t>(nt) * nkb + j) * 32];
                  mma_16816(acc[j & 1][nt], a, b.x, b.y);
                }
              }
            }
          }
        }
        __syncwarp();   // every lane has read the stage
        if (lane == 0 && ok && issued < total) issue_next();
        if (++cs == NS) { cs = 0; phase ^= 1u; }
        kc += ckt;
      }
#pragma unroll
      for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) y[nt][r] = acc[0][nt][r] + acc[1][nt][r];
      // the tile's K parts: summed in the fixed order ks = 0, 1, ... (double
      // buffered by tile parity: one barrier a tile)
      if (KS > 1) {
        float* rb = red + (static_cast<size_t>((ti & 1) * EM_WARPS + warp) * (4 * NTP)) * 32 + lane;
#pragma unroll
        for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) rb[(4 * nt + r) * 32] = y[nt][r];
        asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(KS * 32) : "memory");
        if (ks == 0) {
          const float* r0 = red + (static_cast<size_t>((ti & 1) * EM_WARPS + slot * KS) * (4 * NTP)) * 32 + lane;
#pragma unroll
          for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) y[nt][r] = r0[(4 * nt + r) * 32];
          for (int k2 = 1; k2 < KS; ++k2) {
            const float* rk = r0 + static_cast<size_t>(k2) * (4 * NTP) * 32;
#pragma unroll
            for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
              for (int r = 0; r < 4; ++r) y[nt][r] += rk[(4 * nt + r) * 32];
          }
        }
      }
      if (ok && ks == 0) {
        int si = 0;
        while (si + 1 < A.nseg && gt >= A.seg_t0[si + 1]) ++si;
        const int r0 = (gt - A.seg_t0[si]) * 16 + g;   // rows r0 and r0 + 8 of the segment
#pragma unroll
        for (int nt = 0; nt < NTP; ++nt) {
          // (token, row, value) of this lane's accumulators
          float val[4];
          int tok[4];
          if (SPLIT) {
            val[0] = y[nt][0] + y[nt][1]; val[1] = y[nt][2] + y[nt][3];
            tok[0] = tok[1] = nt * 4 + t;
            tok[2] = tok[3] = -1;
          } else {
            val[0] = y[nt][0]; val[1] = y[nt][2]; val[2] = y[nt][1]; val[3] = y[nt][3];
            tok[0] = tok[1] = nt * 8 + 2 * t;
            tok[2] = tok[3] = nt * 8 + 2 * t + 1;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int row = r0 + 8 * (q & 1);
            if (nt >= nnt || tok[q] < 0 || tok[q] >= ntok || row >= A.seg[si].rows) continue;
            const int tt = T0 + tok[q];
            if (A.out_mode == 0) {
              A.outf[static_cast<int64_t>(tt) * A.out_ld + A.seg[si].col0 + row] = val[q];
            } else {
              const int64_t e = static_cast<int64_t>(tt) * A.H + A.seg[si].col0 + row;
              float sv = val[q];
              if (A.y_add) sv += __ldcg(A.y_add + e);
              if (A.delta) A.delta[e] = sv;
              reinterpret_cast<unsigned short*>(A.out)[e] = st16_bits(ld16(A.x, e, A.x_dt) + sv, A.x_dt);
            }
          }
        }
      }
    }
  }
  cta_stamp(A.trace, 2);
  if (!ok && lane == 0) {
    // after a wait ran out: let this warp's copies in flight land (bounded)
    for (int j = gi_fail; j < issued; ++j)
      (void)eb_wait(eb_smem(bars + j % NS), static_cast<uint32_t>(j / NS) & 1u);
  }
  if (holds_router) {
    // release this CTA's router logits to the routing CTA
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(A.route_counter, 1);
  }
  cta_stamp(A.trace, 3);
}

// A [rows, K] 16-bit matrix (row-major) -> [ceil(rows/16), K/16, 32 lanes, 8
// values]: lane (g, t) of tile rt, block kb holds rows 16 rt + g and + 8 at
// columns 16 kb + {2t, 2t + 1} and {2t + 8, 2t + 9}, in the order
// (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1), (g, 2t+8), (g, 2t+9), (g+8, 2t+8),
// (g+8, 2t+9); rows past the matrix are zeros.
static __global__ void k_tile_dense(const unsigned short* __restrict__ in, unsigned short* __restrict__ out,
                                    int rows, int K) {
  const int nkb = K >> 4;
  const int64_t n = static_cast<int64_t>((rows + 15) >> 4) * nkb * 32 * 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(i & 7), lane = static_cast<int>((i >> 3) & 31);
    const int64_t r = i >> 8;   // (tile, kb)
    const int kb = static_cast<int>(r % nkb);
    const int64_t rt = r / nkb;
    const int g = lane >> 2, t = lane & 3;
    const int64_t row = rt * 16 + g + ((v & 2) ? 8 : 0);
    const int col = kb * 16 + 2 * t + (v & 1) + ((v & 4) ? 8 : 0);
    out[i] = row < rows ? in[row * K + col] : static_cast<unsigned short>(0);
  }
}

}  // namespace moe
