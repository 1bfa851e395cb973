// Dense 16-bit gemv with its weight rows moved by bulk copies (sm_103a): the
// shared expert's gate/up and down projections and the layer's output
// projection on the gemv path.  Token rows go in passes of TB (one or two),
// the weights streamed once per pass; every pass reduces in the same order,
// so a row's result does not depend on the batch it is in.
//
// A CTA owns output rows [rb, re) and streams them in stages of SR rows: the
// rows of a stage that lie in one matrix are one contiguous range, so a stage
// is one bulk copy per (segment, part) run, issued by one thread and completing
// on the stage's mbarrier, through a ring of `nst` shared-memory stages (most
// of shared memory: the whole CTA's rows are requested in a few steps).
//
// The reduction axis is split over the warps: chunk c (8 elements, 16 bytes)
// belongs to warp (c / 32) % 8, lane c % 32, so a warp reads 512 contiguous
// bytes of a row per pass and each lane keeps the input elements of its chunks
// in registers for the whole launch (loaded once, TB token rows).  Per stage a
// warp accumulates SR x TB partial dot products, reduces them with one warp
// reduce-scatter, and the CTA sums the 8 warp partials of each (row, token)
// through shared memory before the epilogue.
#pragma once

#include "moe_kernels.cuh"
#include "moe_expert_bulk.cuh"   // eb_bulk, eb_wait, eb_smem

namespace moe {

constexpr int DB_SR = 8;          // rows per stage
constexpr int DB_MAX_STAGES = 6;
constexpr int DB_MAX_CPL = 3;     // chunks per lane: K up to 3 * 256 * 8 = 6144

enum : int { DB_SRC_X = 0, DB_SRC_OUT = 1 };     // input vector: x, or [y | act(shared)]
enum : int { DB_EPI_F32 = 0, DB_EPI_OUT = 1 };   // out_f32[t, r] = s, or the layer output

struct DbArgs {
  DenseSeg seg[4];        // row segments; every segment has the same parts (widths)
  int nseg;
  int total_rows;
  int K;                  // sum of the part widths (elements, multiple of 8)
  int T;
  int nst;                // ring stages
  int stage_bytes;        // SR rows of every part, 128-aligned
  // input vector
  int src;
  const void* x; int x_dt;                 // DB_SRC_X: [T, K] act dtype
  const float* staged; int staged_ld;      // DB_SRC_OUT: y [T, .] for k < latent
  int latent;
  const float* dense_in; int r_in, sh_g_off, sh_u_off, act;   //   act(gate, up) for k >= latent
  // epilogue
  int epi;
  float* out; int64_t out_ld; int out_col0;        // DB_EPI_F32: out[t * out_ld + out_col0 + r]
  const float* y_add; const float* add_f32;        // DB_EPI_OUT: s += y_add[t, r] + add_f32[t, r]
  const void* xres; void* outb; float* delta;      //   out = x + s (act dtype), delta = s
  int* status;
  int dep_tail;           // as DenseInArgs::dep_tail
  unsigned long long* trace;
};

// Byte offset of part p's block inside a stage (blocks are [SR, wk_p] rows).
__device__ __forceinline__ int db_part_off(const DenseSeg& S, int p) {
  return p == 0 ? 0 : DB_SR * S.part[0].wk * 2;
}

template <int TB, int CPL>
__global__ void __launch_bounds__(NT, 1) k_dense_bulk(const __grid_constant__ DbArgs A) {
  extern __shared__ __align__(128) unsigned char db_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nchunk = A.K >> 3;
  unsigned char* stages = db_smem;
  float* red = reinterpret_cast<float*>(db_smem + static_cast<size_t>(A.nst) * A.stage_bytes);   // [SR*TB][NW]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + DB_SR * TB * NW);
  const int nst = A.nst;
  const int64_t c0 = blockIdx.x, g0 = gridDim.x;
  const int rb = static_cast<int>(c0 * A.total_rows / g0), re = static_cast<int>((c0 + 1) * A.total_rows / g0);
  const int nstage = (re - rb + DB_SR - 1) / DB_SR;
  cta_stamp(A.trace, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(eb_smem(bars + s)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // token rows in passes of TB (the weights streamed once per pass)
  const int npass = (A.T + TB - 1) / TB;
  const int total = npass * nstage;
  // stage g (pass g / nstage): rows [rb + SR (g % nstage), ...), one copy per
  // (segment run, part)
  auto issue = [&](int g) {
    const int s = g % nst, i = g % nstage;
    const int r0 = rb + i * DB_SR, r1 = min(re, r0 + DB_SR);
    unsigned char* st = stages + static_cast<size_t>(s) * A.stage_bytes;
    const uint32_t bar = eb_smem(bars + s);
    uint32_t tot = 0;
    for (int r = r0; r < r1;) {
      int si = 0;
      while (r >= A.seg[si].row0 + A.seg[si].rows) ++si;
      const DenseSeg& S = A.seg[si];
      const int rr = min(r1, S.row0 + S.rows);
      for (int p = 0; p < S.nparts; ++p) tot += static_cast<uint32_t>(rr - r) * S.part[p].wk * 2;
      r = rr;
    }
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tot) : "memory");
    for (int r = r0; r < r1;) {
      int si = 0;
      while (r >= A.seg[si].row0 + A.seg[si].rows) ++si;
      const DenseSeg& S = A.seg[si];
      const int rr = min(r1, S.row0 + S.rows);
      for (int p = 0; p < S.nparts; ++p) {
        const DensePart& Pt = S.part[p];
        const char* src = static_cast<const char*>(Pt.w) + static_cast<int64_t>(r - S.row0) * Pt.wk * 2;
        unsigned char* dst = st + db_part_off(S, p) + (r - r0) * Pt.wk * 2;
        eb_bulk(eb_smem(dst), src, static_cast<uint32_t>(rr - r) * Pt.wk * 2, bar);
      }
      r = rr;
    }
  };
  // the weights depend on no earlier kernel: the first stages are requested
  // before waiting for the previous kernel (whose outputs are the input vector)
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < min(nst, total); ++issued) issue(issued);
  if (!A.dep_tail) griddep_wait();
  griddep_launch();
  cta_stamp(A.trace, 1);

  bool ok = true;
  for (int pass = 0; pass < npass; ++pass) {
  const int t0 = pass * TB, tb = min(TB, A.T - t0);
  // this lane's input elements: TB token rows x CPL chunks x 8, in registers
  float xr[TB][CPL][8];
#pragma unroll
  for (int tt = 0; tt < TB; ++tt)
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = (warp + NW * j) * 32 + lane;
      const int t = t0 + tt;
#pragma unroll
      for (int e = 0; e < 8; ++e) xr[tt][j][e] = 0.f;
      if (c < nchunk && tt < tb) {
        if (A.src == DB_SRC_X) {
          const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const char*>(A.x) +
                                                          (static_cast<int64_t>(t) * A.K + 8 * c) * 2);
          cvt8(v, A.x_dt, xr[tt][j]);
        } else if (8 * c < A.latent) {
          // y: 8 consecutive fp32 (latent widths are multiples of 8)
          const float4* y4 = reinterpret_cast<const float4*>(A.staged + static_cast<int64_t>(t) * A.staged_ld + 8 * c);
          const float4 a = __ldcg(y4), b = __ldcg(y4 + 1);
          xr[tt][j][0] = a.x; xr[tt][j][1] = a.y; xr[tt][j][2] = a.z; xr[tt][j][3] = a.w;
          xr[tt][j][4] = b.x; xr[tt][j][5] = b.y; xr[tt][j][6] = b.z; xr[tt][j][7] = b.w;
        } else {
          // act(shared gate, shared up) of 8 consecutive columns
          const float* di = A.dense_in + static_cast<int64_t>(t) * A.r_in;
          const int f = 8 * c - A.latent;
          float u[8], gg[8];
          if (((A.r_in | A.sh_u_off | A.sh_g_off) & 3) == 0) {
            const float4* u4 = reinterpret_cast<const float4*>(di + A.sh_u_off + f);
            const float4 u0 = __ldcg(u4), u1 = __ldcg(u4 + 1);
            u[0] = u0.x; u[1] = u0.y; u[2] = u0.z; u[3] = u0.w; u[4] = u1.x; u[5] = u1.y; u[6] = u1.z; u[7] = u1.w;
            if (A.act == ACT_SWIGLU) {
              const float4* g4 = reinterpret_cast<const float4*>(di + A.sh_g_off + f);
              const float4 g0 = __ldcg(g4), g1 = __ldcg(g4 + 1);
              gg[0] = g0.x; gg[1] = g0.y; gg[2] = g0.z; gg[3] = g0.w; gg[4] = g1.x; gg[5] = g1.y; gg[6] = g1.z; gg[7] = g1.w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              u[e] = __ldcg(di + A.sh_u_off + f + e);
              if (A.act == ACT_SWIGLU) gg[e] = __ldcg(di + A.sh_g_off + f + e);
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) xr[tt][j][e] = act_fn(A.act, A.act == ACT_SWIGLU ? gg[e] : 0.f, u[e]);
        }
      }
    }
  if (pass == 0) cta_stamp(A.trace, 4);

  for (int i = 0; i < nstage; ++i) {
    const int g = pass * nstage + i, s = g % nst;
    if (ok && !eb_wait(eb_smem(bars + s), static_cast<uint32_t>(g / nst) & 1u)) {
      ok = false;
      if (threadIdx.x == 0) atomicOr(A.status, STATUS_TIMEOUT);
    }
    if (g == 0) cta_stamp(A.trace, 5);
    const int r0 = rb + i * DB_SR, nr = min(DB_SR, re - r0);
    const unsigned char* st = stages + static_cast<size_t>(s) * A.stage_bytes;
    float acc[DB_SR][TB];
#pragma unroll
    for (int q = 0; q < DB_SR; ++q)
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[q][t] = 0.f;
    if (ok) {
      // every row of a stage has the parts of the stage's first segment
      int si = 0;
      while (r0 >= A.seg[si].row0 + A.seg[si].rows) ++si;
      const DenseSeg& S = A.seg[si];
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = (warp + NW * j) * 32 + lane;
        if (c >= nchunk) continue;
        // chunk c lies in part 0 or part 1
        const int k = 8 * c;
        const int p = (S.nparts > 1 && k >= S.part[0].wk) ? 1 : 0;
        const int wk = S.part[p].wk, kl = k - (p ? S.part[0].wk : 0);
        const unsigned char* blk = st + db_part_off(S, p) + kl * 2;
        const int dt = S.part[p].dt;
#pragma unroll
        for (int q = 0; q < DB_SR; ++q) {
          if (q < nr) {
            float wf[8];
            cvt8(*reinterpret_cast<const uint4*>(blk + q * wk * 2), dt, wf);
#pragma unroll
            for (int t = 0; t < TB; ++t) {
              float a = acc[q][t];
#pragma unroll
              for (int e = 0; e < 8; ++e) a = fmaf(wf[e], xr[t][j][e], a);
              acc[q][t] = a;
            }
          }
        }
      }
    }
    // warp reduce-scatter of the SR x TB partials, then the 8 warps through smem
    constexpr int NV = DB_SR * TB;
    float v[NV];
#pragma unroll
    for (int q = 0; q < DB_SR; ++q)
#pragma unroll
      for (int t = 0; t < TB; ++t) v[q * TB + t] = acc[q][t];
    const float tot = warp_reduce_scatter<NV>(v, lane);
    constexpr int LPV = 32 / NV;
    if ((lane & (LPV - 1)) == 0) red[(lane / LPV) * NW + warp] = tot;
    __syncthreads();   // stage s is free; red is complete
    if (threadIdx.x == 0 && ok && issued < total) issue(issued++);
    if (threadIdx.x < NV) {
      const int q = threadIdx.x / TB, tt = threadIdx.x % TB, t = t0 + tt;
      if (q < nr && tt < tb) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) sum += red[threadIdx.x * NW + w];
        const int r = r0 + q;
        if (A.epi == DB_EPI_F32) {
          A.out[static_cast<int64_t>(t) * A.out_ld + A.out_col0 + r] = sum;
        } else {
          const int64_t e = static_cast<int64_t>(t) * A.total_rows + r;
          if (A.y_add) sum += __ldcg(A.y_add + e);
          if (A.add_f32) sum += __ldcg(A.add_f32 + e);
          const float xv = ld16(A.xres, e, A.x_dt);
          reinterpret_cast<unsigned short*>(A.outb)[e] = st16_bits(xv + sum, A.x_dt);
          if (A.delta) A.delta[e] = sum;
        }
      }
    }
    __syncthreads();   // red is read before the next stage writes it
  }
  }
  if (!ok && threadIdx.x == 0) {
    // after a wait ran out: let the copies still in flight land (bounded)
    for (int i = 0; i < issued; ++i) (void)eb_wait(eb_smem(bars + i % nst), static_cast<uint32_t>(i / nst) & 1u);
  }
  if (A.dep_tail) griddep_wait();
  cta_stamp(A.trace, 3);
}

}  // namespace moe
