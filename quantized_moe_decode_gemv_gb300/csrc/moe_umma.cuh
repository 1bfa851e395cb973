// Row-grouped GEMM on the 5th-generation tensor cores (tcgen05, sm_103a) for
// many token rows per forward.
//
// When the batch holds enough token rows that several rows share an expert,
// the routed experts and the dense projections become real contractions, and
// CUDA-core FMAs can no longer keep up with HBM.  This kernel computes, per
// "group" (a distinct routed expert with the token rows routed to it, or all
// token rows for a dense matrix) and per 128-row tile of the weight matrix,
//
//     D[128 x N] = A[128 x K] . B[N x K]^T          (swap-AB: weights are M,
//                                                    tokens are N)
//
// with A = weights (int4 affine codes dequantised to 16-bit in shared memory,
// or 16-bit dense rows), B = the tokens' activations rounded to the same
// 16-bit type, fp32 accumulation in tensor memory (TMEM), and an epilogue that
// reads TMEM with tcgen05.ld.  One thread issues tcgen05.mma; operands are
// staged by all threads into the K-major, no-swizzle canonical layout
// (8-row x 16-byte core matrices) and handed to the tensor core through
// shared-memory descriptors; completion is signalled with tcgen05.commit on an
// mbarrier.  Two stage buffers let the staging of K-chunk c+1 overlap the MMAs
// of chunk c.  Every mbarrier wait is bounded: after the bound the kernel sets
// the timeout bit of the status word, frees its TMEM and returns.
#pragma once

#include "moe_kernels.cuh"

namespace moe {

constexpr int UM_M = 128;       // weight rows per tile (MMA M)
constexpr int UM_KC = 64;       // K elements per stage
constexpr int UM_NMAX = 256;    // tokens per MMA (MMA N, multiple of 16)
constexpr int UM_THREADS = 256;
constexpr uint32_t UM_SPIN_LIMIT = 1u << 22;

// canonical K-major no-swizzle layout of a [rows x 64] 16-bit tile:
// core matrix (row / 8, k / 8) at (row / 8) * 1024 + (k / 8) * 128 bytes,
// element (row % 8, k % 8) at (row % 8) * 16 + (k % 8) * 2 inside it.
constexpr uint32_t UM_LBO = 128;    // between core matrices along K
constexpr uint32_t UM_SBO = 1024;   // between 8-row groups along M / N
constexpr int UM_A_BYTES = UM_M * UM_KC * 2;        // 16 KB
constexpr int UM_B_BYTES = UM_NMAX * UM_KC * 2;     // 32 KB

enum : int { UA_INT4 = 0, UA_DENSE = 1 };                  // A source
enum : int { UE_ROWS = 0, UE_DENSE_IN = 1, UE_OUT = 2 };   // epilogue

struct UmmaArgs {
  // ---- groups ----
  int experts;              // 1: groups are the distinct routed experts (route metadata)
  const int* meta;          // route metadata (experts mode)
  int umax;
  int n_tokens;             // dense mode: tokens of the single group
  int n_rows;               // rows of A (per expert / total dense rows)
  int K;                    // reduction length (multiple of 64)
  // ---- A ----
  int a_mode;
  const uint32_t* q;        // int4: [E, n_rows, K/8]
  const uint32_t* sb;       // int4: [E, n_rows, K/G]
  const uint32_t* q2;       // int4 gate (SwiGLU up): second A, or null
  const uint32_t* sb2;
  int G;
  int s_dt;
  DenseSeg seg[4];          // dense: row segments (parts concatenated along K)
  int nseg;
  int mma_dt;               // DT_BF16 or DT_FP16: the 16-bit type of A and B
  // ---- B: token n's activation row ----
  // experts mode: pair p = pairs[p0 + n]; source row = by_pair ? p : p / k
  // dense mode: source row = n
  const void* b0; int b0_dt; int64_t b0_stride; int64_t b0_off; int b0_k;   // columns [0, b0_k)
  const void* b1; int b1_dt; int64_t b1_stride; int64_t b1_off;             // columns [b0_k, K)
  int by_pair;
  int k;                    // top_k
  // ---- epilogue ----
  int epi;
  int act;                  // UE_ROWS: activation applied (-1: none)
  float* out_f32;           // UE_ROWS: [P, n_rows]; UE_DENSE_IN: [T, ld]
  int64_t out_ld;
  int out_col0;             // UE_DENSE_IN: first output column
  // UE_OUT: out[t, n] = x[t, n] + acc (+ combine of pexp for non-latent)
  const void* x; int x_dt; void* out; float* delta;
  const float* pexp; const float* wts; int add_combine;
  int* status;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(UM_LBO >> 4) << 16) |
         (static_cast<uint64_t>(UM_SBO >> 4) << 32) |
         (1ull << 46);  // descriptor version for tcgen05; layout type 0 = no swizzle
}

// kind::f16 instruction descriptor: fp32 accumulate, A/B type, K-major both, N, M=128
__device__ __forceinline__ uint32_t umma_idesc(int n, int dt) {
  const uint32_t ab = (dt == DT_BF16) ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(UM_M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count) : "memory");
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
  for (uint32_t i = 0; i < UM_SPIN_LIMIT; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack16(float a, float b, int dt) {
  if (dt == DT_BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t core_off(int row, int k) {
  return static_cast<uint32_t>((row >> 3) * UM_SBO + (k >> 3) * UM_LBO + (row & 7) * 16 + (k & 7) * 2);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

struct UmmaGroup {
  int e;      // expert id (experts mode)
  int p0;     // first pair
  int n;      // tokens
};

__device__ __forceinline__ UmmaGroup umma_group(const UmmaArgs& A, int g) {
  UmmaGroup G;
  if (A.experts) {
    G.e = A.meta[1 + g];
    G.p0 = A.meta[1 + A.umax + g];
    G.n = A.meta[1 + A.umax + g + 1] - G.p0;
  } else {
    G.e = 0;
    G.p0 = 0;
    G.n = A.n_tokens;
  }
  return G;
}

// source row of token n of the group
__device__ __forceinline__ int64_t umma_token_row(const UmmaArgs& A, const UmmaGroup& G, int n,
                                                  int* pid_out) {
  if (!A.experts) {
    *pid_out = n;
    return n;
  }
  const int pid = A.meta[2 + 2 * A.umax + G.p0 + n];
  *pid_out = pid;
  return A.by_pair ? pid : pid / A.k;
}

// Stage A rows [m0, m0 + 128) x K-chunk kc of matrix (q, sb) or of the dense
// segments into sA.
__device__ __forceinline__ void umma_stage_a(const UmmaArgs& A, const UmmaGroup& G, int m0, int kc,
                                             const uint32_t* q, const uint32_t* sb, char* sA) {
  const int k0 = kc * UM_KC;
  if (A.a_mode == UA_INT4) {
    // 128 rows x 2 halves of 32 codes: one 16-byte load per thread
    const int t = threadIdx.x;
    const int r = t >> 1, h = t & 1;
    const int m = m0 + r;
    if (m < A.n_rows) {
      const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
      const uint4 w = ldg_stream(q + row * (A.K >> 3) + (k0 >> 3) + 4 * h);
      const int g = (k0 + 32 * h) / A.G;
      float s, b;
      sb_decode(ldg_u32(sb + row * (A.K / A.G) + g), A.s_dt, s, b);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // word i holds elements 32h + 8i .. +7 (one core-matrix row), nibble n -> element n
        uint32_t pr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = fmaf(s, static_cast<float>((ws[i] >> (8 * j)) & 0xFu), b);
          const float hi = fmaf(s, static_cast<float>((ws[i] >> (8 * j + 4)) & 0xFu), b);
          pr[j] = pack16(lo, hi, A.mma_dt);
        }
        *reinterpret_cast<uint4*>(sA + core_off(r, 32 * h + 8 * i)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(sA + core_off(r, 32 * h + 8 * i)) = make_uint4(0u, 0u, 0u, 0u);
    }
  } else {
    // dense 16-bit rows: 128 rows x 8 chunks of 16 bytes = 1024 chunks, 4 per thread
    for (int c = threadIdx.x; c < UM_M * (UM_KC / 8); c += UM_THREADS) {
      const int r = c >> 3, j = c & 7;
      const int m = m0 + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < A.n_rows) {
        int si = 0;
        while (m >= A.seg[si].row0 + A.seg[si].rows) ++si;
        const DenseSeg& S = A.seg[si];
        const int kk = k0 + 8 * j;
        for (int p = 0; p < S.nparts; ++p) {
          const DensePart& P = S.part[p];
          if (kk >= P.k0 && kk < P.k0 + P.wk) {
            const char* base = static_cast<const char*>(P.w) +
                               (static_cast<int64_t>(m - S.row0) * P.wk + (kk - P.k0)) * 2;
            v = ldg_stream(base);
          }
        }
      }
      *reinterpret_cast<uint4*>(sA + core_off(r, 8 * j)) = v;
    }
  }
}

// Stage B: tokens [n0, n0 + npad) of the group, K-chunk kc, as 16-bit.
__device__ __forceinline__ void umma_stage_b(const UmmaArgs& A, const UmmaGroup& G, int n0,
                                             int nvalid, int npad, int kc, char* sB) {
  const int k0 = kc * UM_KC;
  for (int c = threadIdx.x; c < npad * (UM_KC / 8); c += UM_THREADS) {
    const int n = c >> 3, j = c & 7;
    const int kk = k0 + 8 * j;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < nvalid) {
      int pid;
      const int64_t row = umma_token_row(A, G, n0 + n, &pid);
      const void* src;
      int dt;
      int64_t e;
      if (kk < A.b0_k) {
        src = A.b0; dt = A.b0_dt; e = A.b0_off + row * A.b0_stride + kk;
      } else {
        src = A.b1; dt = A.b1_dt; e = A.b1_off + row * A.b1_stride + (kk - A.b0_k);
      }
      if (dt == A.mma_dt) {
        v = *reinterpret_cast<const uint4*>(static_cast<const char*>(src) + e * 2);
      } else {
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = ld_any(src, e + i, dt);
        v.x = pack16(f[0], f[1], A.mma_dt); v.y = pack16(f[2], f[3], A.mma_dt);
        v.z = pack16(f[4], f[5], A.mma_dt); v.w = pack16(f[6], f[7], A.mma_dt);
      }
    }
    *reinterpret_cast<uint4*>(sB + core_off(n, 8 * j)) = v;
  }
}

constexpr size_t umma_smem_bytes() {
  return 2 * (2 * static_cast<size_t>(UM_A_BYTES) + UM_B_BYTES) + 64;
}

__global__ void __launch_bounds__(UM_THREADS, 1) k_umma(const UmmaArgs A) {
  extern __shared__ __align__(1024) char um_smem[];
  // layout: [2 stages][A (16 KB), A2 (16 KB), B (32 KB)] then 2 mbarriers + tmem holder
  constexpr int STAGE = 2 * UM_A_BYTES + UM_B_BYTES;
  char* base = um_smem;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(base + 2 * STAGE);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + 2 * STAGE + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool gated = (A.a_mode == UA_INT4) && A.q2 != nullptr;
  const int ncols = gated ? 512 : 256;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(smem_u32(&mbar[0]), 1);
    mbar_init(smem_u32(&mbar[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  uint32_t phase[2] = {0u, 0u};
  uint32_t pending[2] = {0u, 0u};   // a commit on this stage not yet waited for
  bool ok = true;

  const int n_groups = A.experts ? A.meta[0] : 1;
  const int mtiles = (A.n_rows + UM_M - 1) / UM_M;
  const int nkc = A.K / UM_KC;

  for (int unit = blockIdx.x; ok && unit < n_groups * mtiles; unit += gridDim.x) {
    const int g = unit / mtiles, mt = unit - g * mtiles;
    const UmmaGroup G = umma_group(A, g);
    const int m0 = mt * UM_M;
    for (int n0 = 0; ok && n0 < G.n; n0 += UM_NMAX) {
      const int nvalid = min(UM_NMAX, G.n - n0);
      const int npad = (nvalid + 15) & ~15;
      const uint32_t idesc = umma_idesc(npad, A.mma_dt);
      for (int kc = 0; kc < nkc; ++kc) {
        const int st = kc & 1;
        char* sA = base + st * STAGE;
        char* sA2 = sA + UM_A_BYTES;
        char* sB = sA + 2 * UM_A_BYTES;
        // the MMAs that last read this stage must be done before overwriting it;
        // thread 0 waits, the barrier makes the outcome uniform
        if (pending[st]) {
          bool w = true;
          if (tid == 0) w = mbar_wait(smem_u32(&mbar[st]), phase[st]);
          phase[st] ^= 1u;
          pending[st] = 0u;
          if (!__syncthreads_and(w)) { ok = false; break; }
        }
        umma_stage_a(A, G, m0, kc, A.q, A.sb, sA);
        if (gated) umma_stage_a(A, G, m0, kc, A.q2, A.sb2, sA2);
        umma_stage_b(A, G, n0, nvalid, npad, kc, sB);
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < UM_KC / 16; ++kk) {
            const uint64_t ad = umma_desc(smem_u32(sA) + kk * 2 * UM_LBO);
            const uint64_t bd = umma_desc(smem_u32(sB) + kk * 2 * UM_LBO);
            umma_f16(tmem, ad, bd, idesc, (kc | kk) ? 1u : 0u);
            if (gated) {
              const uint64_t a2 = umma_desc(smem_u32(sA2) + kk * 2 * UM_LBO);
              umma_f16(tmem + 256, a2, bd, idesc, (kc | kk) ? 1u : 0u);
            }
          }
          umma_commit(smem_u32(&mbar[st]));
        }
        pending[st] = 1u;
      }
      if (!ok) break;
      // wait for the last MMAs (both stages), then read the accumulators
      {
        bool w = true;
        for (int st = 0; st < 2; ++st) {
          if (pending[st]) {
            if (tid == 0 && w) w = mbar_wait(smem_u32(&mbar[st]), phase[st]);
            phase[st] ^= 1u;
            pending[st] = 0u;
          }
        }
        if (!__syncthreads_and(w)) { ok = false; break; }
      }
      tc_fence_after();
      // epilogue: warp w reads TMEM lanes 32*(w%4).. (rows), columns split by w/4
      const int q4 = warp & 3, half = warp >> 2;
      const int m = m0 + 32 * q4 + lane;
      for (int c0 = half * 16; c0 < npad; c0 += 32) {
        float acc[16], accg[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + c0, acc);
        if (gated) tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 256 + c0, accg);
        if (m >= A.n_rows) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          if (n >= nvalid) break;
          int pid;
          const int64_t trow = umma_token_row(A, G, n0 + n, &pid);
          (void)trow;
          float v = acc[i];
          if (A.epi == UE_ROWS) {
            // gate accumulates in the second TMEM block; act(g, u)
            // A (q) is the up projection, A2 (q2) the gate: act(gate, up)
            if (A.act >= 0) v = gated ? act_fn(A.act, accg[i], v) : act_fn(A.act, 0.f, v);
            A.out_f32[static_cast<int64_t>(pid) * A.n_rows + m] = v;
          } else if (A.epi == UE_DENSE_IN) {
            A.out_f32[static_cast<int64_t>(pid) * A.out_ld + A.out_col0 + m] = v;
          } else {
            const int t = pid;
            if (A.add_combine) {
              float y = 0.f;
              for (int p = 0; p < A.k; ++p)
                y = fmaf(A.wts[t * A.k + p], A.pexp[static_cast<int64_t>(t * A.k + p) * A.n_rows + m], y);
              v += y;
            }
            const int64_t e = static_cast<int64_t>(t) * A.n_rows + m;
            const float xv = ld16(A.x, e, A.x_dt);
            reinterpret_cast<unsigned short*>(A.out)[e] = st16_bits(xv + v, A.x_dt);
            if (A.delta) A.delta[e] = v;
          }
        }
      }
      // all TMEM reads done before the next unit's MMAs overwrite the accumulators
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  }
  if (!ok && tid == 0) {
    atomicOr(A.status, STATUS_TIMEOUT);
    // bounded wait for MMAs still in flight before releasing TMEM
    for (int st = 0; st < 2; ++st)
      if (pending[st]) mbar_wait(smem_u32(&mbar[st]), phase[st]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
  }
}

}  // namespace moe

namespace moe {

// Operand B of the grouped output projection: per token, [combined routed
// output y (latent layers) | shared-expert activation], rounded to the MMA type.
struct PrepOutArgs {
  int T, L, Fs, k, act, mma_dt;
  const float* pexp;       // [T*k, L]
  const float* wts;        // [T*k]
  const float* dense_in;   // [T, r_in]
  int r_in, sh_g_off, sh_u_off;
  unsigned short* bout;    // [T, L + Fs]
};

__global__ void k_prep_out(const PrepOutArgs A) {
  const int K = A.L + A.Fs;
  const int64_t n = static_cast<int64_t>(A.T) * K;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / K), c = static_cast<int>(i - static_cast<int64_t>(t) * K);
    float v;
    if (c < A.L) {
      v = 0.f;
      for (int p = 0; p < A.k; ++p)
        v = fmaf(A.wts[t * A.k + p], A.pexp[static_cast<int64_t>(t * A.k + p) * A.L + c], v);
    } else {
      const float* di = A.dense_in + static_cast<int64_t>(t) * A.r_in;
      const int f = c - A.L;
      const float u = di[A.sh_u_off + f];
      const float g = (A.act == ACT_SWIGLU) ? di[A.sh_g_off + f] : 0.f;
      v = act_fn(A.act, g, u);
    }
    A.bout[i] = st16_bits(v, A.mma_dt);
  }
}

}  // namespace moe
