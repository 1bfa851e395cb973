// int4 affine expert gemv with its weights moved by bulk copies (sm_103a).
//
// The routed experts of a decode step are a few MB of packed codes, each byte
// read once.  A CTA owns rows [nb, ne) of one distinct selected expert and
// streams them in groups of 8 * R consecutive rows: the packed codes of a group
// and its interleaved scale/bias words (gate and up for SwiGLU) are each one
// contiguous range, so a group is two (four) bulk copies issued by one thread
// and completing on the stage's mbarrier, through a ring of `nst` shared-memory
// stages.  With the ring as deep as the CTA's groups every byte of the CTA's
// work is requested at once; the down projection issues its copies before it
// waits for the up projection (its experts are known once the routing is), so
// its weights arrive while the up projection finishes.
//
// Warp w computes rows w, w + 8, ..., w + 8 (R - 1) of a group, one row at a
// time, for every token pair of the expert (PB per pass over the weights), and
// finishes each row with one warp reduce-scatter of its PB (x 2 for SwiGLU) dot
// products.  The arithmetic is that of k_expert:
//   sum_k (s q_k + b) x_k = 16 s * sum_k (1 + q_k/16) x_k + (b - 16 s) * sum_k x_k
// per chunk, the chunk sums of x computed once when x is staged.  Every
// mbarrier wait is bounded; a wait that runs out sets the timeout bit of the
// status word and the CTA skips its remaining arithmetic.
#pragma once

#include "moe_kernels.cuh"

namespace moe {

constexpr int EB_WARPS = NT / 32;   // rows of a group per R
constexpr int EB_MAX_STAGES = 8;
constexpr uint32_t EB_SPIN_LIMIT = 1u << 22;

// Shared-memory plan of one k_expert_bulk launch (host and device agree on it).
struct EbPlan {
  int x_bytes;      // staged inputs: [PB][K] fp32 + [PB][K/32] chunk sums, 128-aligned
  int q_bytes;      // codes of one group of one matrix: 8 R rows x K/2
  int sb_bytes;     // scale/bias words of one group of one matrix, 16-byte rounded + 16 slack
  int st_bytes;     // one stage: (gate +) up, 128-aligned
};

__host__ __device__ inline EbPlan eb_plan(int K, int G, int pb, int r, bool gated) {
  EbPlan p;
  const int rows = EB_WARPS * r;
  p.x_bytes = ((pb * K * 4 + pb * (K / 32) * 4) + 127) & ~127;
  p.q_bytes = rows * (K / 2);
  p.sb_bytes = ((rows * (K / G) * 4 + 15) & ~15) + 16;
  p.st_bytes = ((gated ? 2 : 1) * (p.q_bytes + p.sb_bytes) + 127) & ~127;
  return p;
}

__device__ __forceinline__ uint32_t eb_smem(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void eb_bulk(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool eb_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < EB_SPIN_LIMIT; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Stage the input rows of pairs [pc, pc + np) swizzled for 32-element chunk
// readers (rows np..PB-1 zero), then their chunk sums.  Ends with a barrier.
template <int PB>
__device__ __forceinline__ void eb_stage_pairs(const ExpertArgs& A, const int* pairs, int pc, int np,
                                               float4* xs4, float* xsum) {
  const int K = A.K, K4 = K >> 2, nchunk = K >> 5;
  for (int i = threadIdx.x; i < PB * K4; i += NT) {
    const int pp = i / K4, f4 = i - pp * K4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (pp < np) {
      int pid = pairs[pc + pp];
      if (!idx_ok(A.status, CK_BULK_PAIR, pid, static_cast<long long>(A.T) * A.k)) pid = 0;
      const int64_t row = A.xin_by_pair ? pid : (pid / A.k);
      const int64_t base = A.xin_off + row * A.xin_stride + 4 * f4;
      if (A.xin_dt == DT_FP32) {
        const float* src = static_cast<const float*>(A.xin) + base;
        if (((A.xin_off | A.xin_stride) & 3) == 0) {
          v = __ldcg(reinterpret_cast<const float4*>(src));
        } else {
          v.x = __ldcg(src); v.y = __ldcg(src + 1); v.z = __ldcg(src + 2); v.w = __ldcg(src + 3);
        }
      } else {
        v.x = ld16(A.xin, base, A.xin_dt); v.y = ld16(A.xin, base + 1, A.xin_dt);
        v.z = ld16(A.xin, base + 2, A.xin_dt); v.w = ld16(A.xin, base + 3, A.xin_dt);
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

// sum over one 32-code chunk of (1 + q/16) * x, x in registers in chunk order:
// one accumulation chain in element order, exactly as k_expert's chunk_dot, so
// that both expert kernels give the same bits for a row (the forward picks
// either by batch size and a row must not depend on its batch)
__device__ __forceinline__ float eb_dot32(const uint4 w, const float (&x)[32]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = ws[i];
    s = fmaf(nib<0>(v), x[8 * i + 0], s); s = fmaf(nib<1>(v), x[8 * i + 1], s);
    s = fmaf(nib<2>(v), x[8 * i + 2], s); s = fmaf(nib<3>(v), x[8 * i + 3], s);
    s = fmaf(nib<4>(v), x[8 * i + 4], s); s = fmaf(nib<5>(v), x[8 * i + 5], s);
    s = fmaf(nib<6>(v), x[8 * i + 6], s); s = fmaf(nib<7>(v), x[8 * i + 7], s);
  }
  return s;
}

// The 32 codes of a chunk as the floats 1 + q/16 (element order).
__device__ __forceinline__ void eb_decode32(const uint4 w, float (&q)[32]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = ws[i];
    q[8 * i + 0] = nib<0>(v); q[8 * i + 1] = nib<1>(v); q[8 * i + 2] = nib<2>(v); q[8 * i + 3] = nib<3>(v);
    q[8 * i + 4] = nib<4>(v); q[8 * i + 5] = nib<5>(v); q[8 * i + 6] = nib<6>(v); q[8 * i + 7] = nib<7>(v);
  }
}

// eb_dot32 on decoded codes: the same single chain in element order.
__device__ __forceinline__ float eb_dot32f(const float (&q)[32], const float (&x)[32]) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) s = fmaf(q[i], x[i], s);
  return s;
}

template <int PB, int R, bool GATED>
__global__ void __launch_bounds__(NT, 2) k_expert_bulk(const __grid_constant__ ExpertArgs A) {
  extern __shared__ __align__(128) unsigned char eb_smem_raw[];
  const int cta = static_cast<int>(blockIdx.x);
  constexpr int NM = GATED ? 2 : 1;   // matrices: up (m 0) and gate (m 1)
  constexpr int GR = EB_WARPS * R;    // rows of a group
  const int K = A.K, K4 = K >> 2, nchunk = K >> 5, ngr = K / A.G, gsh = A.gsh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const EbPlan P = eb_plan(K, A.G, PB, R, GATED);
  float4* xs4 = reinterpret_cast<float4*>(eb_smem_raw);
  float* xsum = reinterpret_cast<float*>(xs4 + PB * K4);
  unsigned char* stages = eb_smem_raw + P.x_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + static_cast<size_t>(A.nst) * P.st_bytes);
  const int nst = A.nst;

  const int s_dt = A.s_dt;
  const int u = cta / A.cps, part = cta - u * A.cps;
  const int nb = static_cast<int>(static_cast<int64_t>(part) * A.n_rows / A.cps);
  const int ne = static_cast<int>(static_cast<int64_t>(part + 1) * A.n_rows / A.cps);
  const int* uniq_e = A.meta + 1;
  const int* uniq_p0 = A.meta + 1 + A.umax;
  const int* pairs = A.meta + 2 + 2 * A.umax;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(eb_smem(bars + s)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cta_stamp(A.trace, 0);
  if (!A.pre_wait_phase) griddep_wait();
  griddep_launch();
  if (!A.pre_wait_phase) cta_stamp(A.trace, 1);
  if (u >= A.meta[0]) { cta_stamp(A.trace, 3); return; }
  // a bad expert id (index checks) copies nothing and writes nothing
  const bool e_ok = idx_ok(A.status, CK_BULK_E, uniq_e[u], A.n_experts) &&
                    range_ok(A.status, uniq_p0[u], uniq_p0[u + 1], static_cast<long long>(A.T) * A.k);
  const int64_t e = e_ok ? uniq_e[u] : 0;
  const int pa = uniq_p0[u], pe = e_ok ? uniq_p0[u + 1] : pa;
  const int ngroups = e_ok ? (ne - nb + GR - 1) / GR : 0;
  const int nbatch = (pe - pa + PB - 1) / PB;
  // when the ring holds all of the CTA's groups they stay resident and every
  // pair batch reuses them (each weight byte read once); otherwise the groups
  // are streamed again per batch
  const bool resident = nst >= ngroups;
  const int total = resident ? ngroups : ngroups * nbatch;
  cta_stamp(A.trace, 4);

  // group g -> stage g % nst: per matrix the codes [rows, K/2], then the 16-byte
  // aligned range around the group's scale/bias words (which start sb_w0 words in)
  const uint32_t* qm[2] = {A.q, A.q_gate};
  const uint32_t* sm[2] = {A.sb, A.sb_gate};
  auto issue = [&](int g) {
    const int t = g % ngroups, s = g % nst;
    const int r0 = nb + t * GR, nr = min(GR, ne - r0);
    const uint32_t bar = eb_smem(bars + s);
    unsigned char* st = stages + static_cast<size_t>(s) * P.st_bytes;
    uint32_t bytes[2][2];
    const char* src[2][2];
    uint32_t tot = 0;
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      src[m][0] = reinterpret_cast<const char*>(qm[m] + (e * A.n_rows + r0) * (K >> 3));
      bytes[m][0] = static_cast<uint32_t>(nr) * (K >> 1);
      const uint64_t a = reinterpret_cast<uint64_t>(sm[m] + (e * A.n_rows + r0) * ngr);
      const uint64_t a0 = a & ~uint64_t(15), a1 = (a + static_cast<uint64_t>(nr) * ngr * 4 + 15) & ~uint64_t(15);
      src[m][1] = reinterpret_cast<const char*>(a0);
      bytes[m][1] = static_cast<uint32_t>(a1 - a0);
      tot += bytes[m][0] + bytes[m][1];
    }
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tot) : "memory");
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      unsigned char* d = st + m * (P.q_bytes + P.sb_bytes);
      eb_bulk(eb_smem(d), src[m][0], bytes[m][0], bar);
      eb_bulk(eb_smem(d + P.q_bytes), src[m][1], bytes[m][1], bar);
    }
  };
  int issued = 0;   // thread 0: groups whose copies were issued
  if (threadIdx.x == 0) {
    const int n0 = min(nst, total);
    for (; issued < n0; ++issued) issue(issued);
  }
  cta_stamp(A.trace, 5);
  if (A.pre_wait_phase) { griddep_wait(); cta_stamp(A.trace, 1); }

  bool ok = true;
  int g = 0, g_fail = 0;
  for (int b = 0; b < nbatch; ++b) {
    const int pc = pa + b * PB, np = min(PB, pe - pc);
    if (b) __syncthreads();
    eb_stage_pairs<PB>(A, pairs, pc, np, xs4, xsum);
    if (b == 0) cta_stamp(A.trace, 6);
    for (int t = 0; t < ngroups; ++t, ++g) {
      const int s = resident ? t : g % nst;
      if (ok && (!resident || b == 0) && !eb_wait(eb_smem(bars + s), static_cast<uint32_t>(g / nst) & 1u)) {
        ok = false;
        g_fail = g;
        if (threadIdx.x == 0) atomicOr(A.status, STATUS_TIMEOUT);
      }
      if (g == 0) cta_stamp(A.trace, 7);
      const int r0 = nb + t * GR, nr = min(GR, ne - r0);
      const unsigned char* st = stages + static_cast<size_t>(s) * P.st_bytes;
      const int sb_w0 = static_cast<int>((reinterpret_cast<uint64_t>(A.sb + (e * A.n_rows + r0) * ngr) & 15) >> 2);
      if (ok && warp < nr) {
        // rows warp + 8 j of the group, one at a time: a compact loop (code run
        // only a few times per launch is fetched from L2 as it runs, so a
        // body unrolled over rows stalls on instruction fetch)
        const int rows_w = (nr - warp + EB_WARPS - 1) / EB_WARPS;
#pragma unroll 1
        for (int j = 0; j < rows_w; ++j) {
          const int rl = warp + EB_WARPS * j;
          float acc[PB], accg[PB];
#pragma unroll
          for (int pp = 0; pp < PB; ++pp) { acc[pp] = 0.f; accg[pp] = 0.f; }
#pragma unroll 1
          for (int c = lane; c < nchunk; c += 32) {
            const int gi = c >> gsh;
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              const unsigned char* d = st + m * (P.q_bytes + P.sb_bytes);
              const uint4 w = reinterpret_cast<const uint4*>(d)[rl * (K >> 5) + c];
              float sc, bi;
              sb_decode(reinterpret_cast<const uint32_t*>(d + P.q_bytes)[sb_w0 + rl * ngr + gi], s_dt, sc, bi);
              const float s16 = 16.f * sc, bb = bi - s16;
              // the 32 codes as floats 1 + q/16, once for all the pairs
              float qf[32];
              eb_decode32(w, qf);
#pragma unroll
              for (int pp = 0; pp < PB; ++pp) {
                if (pp < np) {
                  // the input chunk in chunk order (staged swizzled)
                  const float4* x8 = xs4 + pp * K4 + 8 * c;
                  const int sw = c & 7;
                  float xr[32];
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    const float4 a4 = x8[i ^ sw];
                    xr[4 * i] = a4.x; xr[4 * i + 1] = a4.y; xr[4 * i + 2] = a4.z; xr[4 * i + 3] = a4.w;
                  }
                  float& dst = (m == 1) ? accg[pp] : acc[pp];
                  dst = fmaf(s16, eb_dot32f(qf, xr), fmaf(bb, xsum[pp * nchunk + c], dst));
                }
              }
            }
          }
          // warp reduce-scatter of the (pair, up|gate) partial sums
          constexpr int NV = PB * 2;
          float v[NV];
#pragma unroll
          for (int pp = 0; pp < PB; ++pp) { v[pp * 2] = acc[pp]; v[pp * 2 + 1] = accg[pp]; }
          const float tot = warp_reduce_scatter<NV>(v, lane);
          constexpr int LPV = 32 / NV;
          const int vi = lane / LPV;
          const float other = __shfl_down_sync(0xffffffffu, tot, LPV);   // gate partner
          if ((lane & (2 * LPV - 1)) == 0) {
            const int pp = vi >> 1;
            if (pp < np) {
              const int pid = pairs[pc + pp];
              const float val = (A.act >= 0) ? act_fn(A.act, other, tot) : tot;
              if (idx_ok(A.status, CK_BULK_PAIR, pid, static_cast<long long>(A.T) * A.k))
                A.out[static_cast<int64_t>(pid) * A.n_rows + r0 + rl] = val;
            }
          }
        }
      }
      if (g == 0) cta_stamp(A.trace, 8);
      __syncthreads();   // stage s is free
      if (threadIdx.x == 0 && ok && !resident && g + nst < total) issue(issued++);
    }
  }
  cta_stamp(A.trace, 2);
  if (!ok && threadIdx.x == 0) {
    // after a wait ran out: let the copies still in flight land (bounded)
    // before the CTA's shared memory is released
    for (int gg = g_fail; gg < issued; ++gg)
      (void)eb_wait(eb_smem(bars + gg % nst), static_cast<uint32_t>(gg / nst) & 1u);
  }
  __syncthreads();
  if (A.comb) expert_fused_combine(A, part, nb, ne);
  cta_stamp(A.trace, 3);
}

}  // namespace moe
