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
// with fp32 accumulation in tensor memory (TMEM) and an epilogue that reads
// TMEM with tcgen05.ld.  A is either 16-bit dense rows or int4 affine codes,
// which are dequantised to 16 bits in shared memory; B is the tokens' 16-bit
// activations.  Both are moved by cp.async into a ring of `stages` shared-memory
// slots in the K-major, no-swizzle canonical layout (8-row x 16-byte core
// matrices), so several K-chunks are in flight while the tensor core works on
// an earlier one.  One thread issues tcgen05.mma through shared-memory
// descriptors and signals completion with tcgen05.commit on an mbarrier.  Every
// mbarrier wait is bounded: after the bound the kernel sets the timeout bit of
// the status word, frees its TMEM and returns.
#pragma once

#include <cuda.h>   // CUtensorMap (the layout only; maps are encoded on the host)

#include "moe_kernels.cuh"

namespace moe {

constexpr int UM_M = 128;       // weight rows per tile (MMA M)
constexpr int UM_KC = 64;       // K elements per stage
constexpr int UM_THREADS = 256;
constexpr int UM_MAX_STAGES = 8;
constexpr int UM_MAX_KSPLIT = 8;
constexpr int UM_MAX_ABUFS = 4;
constexpr uint32_t UM_SPIN_LIMIT = 1u << 22;
constexpr int UM_KSPLIT_MAX_T = 256;   // dense GEMMs split K only up to this many token rows

// canonical K-major no-swizzle layout of a [rows x 64] 16-bit tile:
// core matrix (row / 8, k / 8) at (row / 8) * 1024 + (k / 8) * 128 bytes,
// element (row % 8, k % 8) at (row % 8) * 16 + (k % 8) * 2 inside it.
constexpr uint32_t UM_LBO = 128;    // between core matrices along K
constexpr uint32_t UM_SBO = 1024;   // between 8-row groups along M / N
constexpr int UM_A_BYTES = UM_M * UM_KC * 2;        // 16 KB (a 16-bit A tile)
constexpr int UM_CODE_BYTES = UM_M * UM_KC / 2;     // 4 KB (int4 codes of an A tile)
constexpr int UM_SB_BYTES = UM_M * 8;               // 1 KB (<= 2 scale/bias words per row)

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
  DenseSeg seg[4];          // dense: row segments (16-bit parts concatenated along K)
  int nseg;
  int mma_dt;               // DT_BF16 or DT_FP16: the 16-bit type of A and B
  // ---- B: token n's activation row, 16-bit (mma_dt) ----
  // experts mode: pair p = pairs[p0 + n]; source row = by_pair ? p : p / k
  // dense mode: source row = n
  const void* b0; int64_t b0_stride; int64_t b0_off;
  int by_pair;
  int k;                    // top_k
  // ---- pipeline (host-chosen) ----
  int n_tile;               // tokens per MMA (multiple of 16, <= 256)
  int stages;               // ring depth, 3..UM_MAX_STAGES
  int abufs;                // int4 (k_umma2): dequantised A tiles in the ring, 2..UM_MAX_ABUFS (k_umma: 2)
  int ksplit;               // dense mode: K split over this many units (partials in `part`)
  float* part;              // [ksplit, n_tokens, n_rows] fp32 partial sums (ksplit > 1)
  // ---- epilogue ----
  int epi;
  int act;                  // UE_ROWS: activation applied (-1: none)
  float* out_f32;           // UE_ROWS: [P, n_rows] (if out16 null); UE_DENSE_IN: [T, ld]
  int64_t out_ld;
  int out_col0;             // UE_DENSE_IN: first output column
  unsigned short* out16;    // UE_ROWS: 16-bit [P, n_rows] instead of fp32;
                            // UE_DENSE_IN: 16-bit copy of columns [c16_0, c16_1)
  int64_t out16_ld;
  int c16_0, c16_1;
  // UE_OUT: out[t, n] = x[t, n] + acc (+ combine of pexp for non-latent)
  const void* x; int x_dt; void* out; float* delta;
  const float* pexp; const float* wts; int add_combine;
  int* status;
  int min_pairs;            // experts mode: groups with fewer token pairs are left to the gemv kernel
  int n_experts, n_pairs;   // experts mode: bounds of expert and pair ids (index checks)
  unsigned long long* trace;   // diagnostics: CTA 0's per-chunk role stamps (k_umma2), or null
  // ---- operands by tensor copies (k_umma2; host-encoded maps) ----
  // tma_a (else cp.async): dense: map [2 * seg + part] over that part's [rows, wk]
  //   16-bit matrix, 128 x 64 boxes with the 128-byte swizzle; int4: map [0] the
  //   codes [E, n_rows, K/8] words (128 x 8-word boxes), [1] the gate's codes,
  //   [2] / [3] the group-major scale/bias words [E, K/G, n_rows] (128 x
  //   words-per-chunk boxes).
  // tma_b (else cp.async): map [8] over the B rows [rows, K] 16-bit (dense
  //   tokens, or the pairs' hidden rows in sorted order), n_tile x 64 boxes with
  //   the 128-byte swizzle.
  int tma_a, tma_b;
  int wait_sleep_ns;        // k_umma2: sleep between mbarrier polls (0: poll back to back)
  int sub;                  // k_umma2: 64-column chunks per ring slot (2: int4 with every operand by tensor copies)
  int b_sorted;             // experts: B row of pair slot n is p0 + n (hidden rows in sorted order)
  int out_sorted;           // UE_ROWS: output row of pair slot n is p0 + n instead of the pair id
  const uint32_t* sbT;      // host: group-major scale/bias words (maps [2], [3])
  const uint32_t* sbT2;
  int b_rows;               // host: rows of the B matrix (map [8])
  CUtensorMap tm[9];
};

constexpr int UM_TRACE_CHUNKS = 128;                        // chunks stamped per launch
constexpr int UM_TRACE_STAMPS = 12;                         // stamps a chunk
constexpr int UM_TRACE_WORDS = UM_TRACE_CHUNKS * UM_TRACE_STAMPS + 8;   // then the start

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

// Descriptor of a K-major tile written with the 128-byte swizzle (8-row
// groups 1024 bytes apart; the tile starts on a 1024-byte boundary, and a
// K step inside the 128-byte row advances the start address).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (1ull << 16) |                                   // leading offset (unused when swizzled)
         (static_cast<uint64_t>(1024 >> 4) << 32) |       // 8-row group stride
         (1ull << 46) |                                   // descriptor version for tcgen05
         (2ull << 61);                                    // layout: 128-byte swizzle
}

// Tensor copies global -> shared, completing on an mbarrier (transaction bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// Arrive on the mbarrier once this thread's earlier cp.async copies have landed
// (the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(mbar) : "memory");
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

// Bounded wait that sleeps `ns` between polls (0: poll back to back), so that
// waiting warps leave the issue slots to the working ones; false on timeout.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t mbar, uint32_t parity, int ns) {
  if (ns <= 0) return mbar_wait(mbar, parity);
  for (uint32_t i = 0; i < UM_SPIN_LIMIT; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
    __nanosleep(static_cast<unsigned>(ns));
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

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most n of this thread's groups are pending (n = stages - 1)
__device__ __forceinline__ void cp_async_wait(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
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

// exact float of a 4-bit code: the bits of 2^23 + q, minus 2^23
__device__ __forceinline__ float code_f(uint32_t q) { return __uint_as_float(0x4B000000u | q) - 8388608.0f; }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

struct UmmaGroup {
  int e;      // expert id (experts mode)
  int p0;     // first pair
  int n;      // tokens
};

// pair id at sorted position i of the route metadata (index checks: 0 if bad)
__device__ __forceinline__ int umma_pair(const UmmaArgs& A, int i) {
  const int pid = A.meta[2 + 2 * A.umax + i];
  return idx_ok(A.status, CK_UMMA_PAIR, pid, A.n_pairs) ? pid : 0;
}

__device__ __forceinline__ UmmaGroup umma_group(const UmmaArgs& A, int g) {
  UmmaGroup G;
  if (A.experts) {
    G.e = A.meta[1 + g];
    if (!idx_ok(A.status, CK_UMMA_E, G.e, A.n_experts)) G.e = 0;
    G.p0 = A.meta[1 + A.umax + g];
    G.n = A.meta[1 + A.umax + g + 1] - G.p0;
    if (!range_ok(A.status, G.p0, G.p0 + G.n, A.n_pairs)) { G.p0 = 0; G.n = 0; }
    if (G.n < A.min_pairs) G.n = 0;   // served by the int4 gemv kernel
  } else {
    G.e = 0;
    G.p0 = 0;
    G.n = A.n_tokens;
  }
  return G;
}

// Work units of a launch.  A unit is one 128-row tile of A against one tile
// of up to n_tile tokens of one group (and one part of K when K is split), so
// that a group with many tokens -- a dense matrix, or an expert that takes a
// large share of a batch -- spreads over many CTAs instead of walking its
// token tiles inside one.  Units are numbered by group, then A tile, then
// token tile: CTAs running side by side read the same A tile.
constexpr int UM_MAX_GROUPS = 4 * UM_THREADS;
static_assert(UM_MAX_GROUPS >= MAX_E, "one prefix entry per routed expert");

// pref[g] = token tiles of the groups before g, for g = 0..n_groups (block
// scan: 4 groups per thread; wsum holds the 8 warp totals).  Ends with a CTA
// barrier; every thread of the CTA calls it.
__device__ __forceinline__ void umma_tile_prefix(const UmmaArgs& A, int n_groups, int* pref, int* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int cnt[4], sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int g = 4 * tid + i;
    cnt[i] = g < n_groups ? (umma_group(A, g).n + A.n_tile - 1) / A.n_tile : 0;
    sum += cnt[i];
  }
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int run = inc - sum;
  for (int w = 0; w < warp; ++w) run += wsum[w];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    pref[4 * tid + i] = run;
    run += cnt[i];
  }
  if (tid == UM_THREADS - 1) pref[UM_MAX_GROUPS] = run;
  __syncthreads();
}

struct UmmaUnit {
  int g, mt, nt, split;
};

// Unit u (< pref[n_groups] * mtiles * nsplit) -> its group, A tile, token tile and K part.
__device__ __forceinline__ UmmaUnit umma_unit(const int* pref, int n_groups, int mtiles, int nsplit, int u) {
  UmmaUnit U;
  U.split = u % nsplit;
  const int r = u / nsplit;
  // the last group whose first unit is at or before r (it has units: r is valid)
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] * mtiles <= r) lo = mid;
    else hi = mid - 1;
  }
  U.g = lo;
  const int ntg = pref[lo + 1] - pref[lo];
  const int local = r - pref[lo] * mtiles;
  U.mt = local / ntg;
  U.nt = local - U.mt * ntg;
  return U;
}

// Shared-memory plan of one launch: `stages` ring slots of
// [A (16-bit tile, or int4 codes + scale/bias words, x2 when gated) | B],
// then (int4 only) two 16-bit A tiles (x2 when gated), the token table (256
// ints), the mbarriers, the TMEM address and the unit prefix.
struct UmmaPlan {
  uint32_t code_bytes, sb_bytes, sb_box;   // int4, per matrix and slot: codes, scale/bias region, its copy
  uint32_t a_raw, b_tile, b_bytes, stage, abuf, tok, pref, total;
};

// A ring slot holds `sub` consecutive 64-column chunks (k_umma2 with every
// operand by tensor copies: 2 for int4; else 1), G the int4 group size.
__host__ __device__ inline UmmaPlan umma_plan(int a_mode, bool gated, int n_tile, int stages, int abufs = 2,
                                              int sub = 1, int G = 64) {
  UmmaPlan p;
  const uint32_t groups = static_cast<uint32_t>(sub * UM_KC / G > 0 ? sub * UM_KC / G : 1);
  p.code_bytes = static_cast<uint32_t>(UM_CODE_BYTES * sub);
  p.sb_box = 128u * 4u * groups;
  p.sb_bytes = p.sb_box > static_cast<uint32_t>(UM_SB_BYTES) ? p.sb_box : static_cast<uint32_t>(UM_SB_BYTES);
  p.a_raw = a_mode == UA_DENSE ? static_cast<uint32_t>(UM_A_BYTES) : (gated ? 2u : 1u) * (p.code_bytes + p.sb_bytes);
  p.b_tile = static_cast<uint32_t>(n_tile) * UM_KC * 2;
  p.b_bytes = p.b_tile * static_cast<uint32_t>(sub);
  p.stage = p.a_raw + p.b_bytes;
  p.abuf = static_cast<uint32_t>(stages) * p.stage;
  const uint32_t abuf_bytes =
      a_mode == UA_DENSE ? 0u : static_cast<uint32_t>(abufs) * (gated ? 2u : 1u) * UM_A_BYTES;
  p.tok = p.abuf + abuf_bytes;
  p.pref = p.tok + 2048;            // token table, mbarriers, TMEM address
  // unit prefix and warp totals, then room to put the plan on a 1024-byte
  // boundary (swizzled tiles)
  p.total = p.pref + (UM_MAX_GROUPS + 1 + 15) * 4 + 1024;
  return p;
}

// Final value of output row m for token/pair `pid` from its accumulator.
// `orow` is the output row of UE_ROWS (the pair id, or the pair's slot in the
// sorted lists).
__device__ __forceinline__ void umma_epilogue(const UmmaArgs& A, int pid, int m, float v, float vg,
                                              bool gated, int orow) {
  if (A.epi == UE_ROWS) {
    // A (q) is the up projection, A2 (q2) the gate: act(gate, up)
    if (A.act >= 0) v = gated ? act_fn(A.act, vg, v) : act_fn(A.act, 0.f, v);
    if (A.out16)
      A.out16[static_cast<int64_t>(orow) * A.n_rows + m] = st16_bits(v, A.mma_dt);
    else
      A.out_f32[static_cast<int64_t>(orow) * A.n_rows + m] = v;
  } else if (A.epi == UE_DENSE_IN) {
    const int col = A.out_col0 + m;
    A.out_f32[static_cast<int64_t>(pid) * A.out_ld + col] = v;
    if (A.out16 && col >= A.c16_0 && col < A.c16_1)
      A.out16[static_cast<int64_t>(pid) * A.out16_ld + (col - A.c16_0)] = st16_bits(v, A.mma_dt);
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

__global__ void __launch_bounds__(UM_THREADS, 2) k_umma(const __grid_constant__ UmmaArgs A) {
  extern __shared__ __align__(1024) char um_smem[];
  const bool gated = (A.a_mode == UA_INT4) && A.q2 != nullptr;
  const UmmaPlan P = umma_plan(A.a_mode, gated, A.n_tile, A.stages);
  char* base = um_smem;
  int* tok_row = reinterpret_cast<int*>(base + P.tok);        // [n_tile] source rows
  uint64_t* mbar = reinterpret_cast<uint64_t*>(base + P.tok + 256 * 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + P.tok + 256 * 4 + 32);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = gated ? 512 : 256;
  const int S = A.stages;

  griddep_wait();
  griddep_launch();
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
  // tcgen05.commit operations issued so far on each mbarrier; chunk c of a
  // tile commits on mbarrier c & 1, and every commit is waited for in order
  uint32_t commits[2] = {0u, 0u}, waited[2] = {0u, 0u};
  bool ok = true;

  const int n_groups = A.experts ? A.meta[0] : 1;
  const int mtiles = (A.n_rows + UM_M - 1) / UM_M;
  const int nkc = A.K / UM_KC;
  const int ngr = A.K / A.G;

  const int nsplit = A.ksplit > 1 ? A.ksplit : 1;
  int* pref = reinterpret_cast<int*>(base + P.pref);
  umma_tile_prefix(A, n_groups, pref, pref + UM_MAX_GROUPS + 1);
  const int nunits = pref[n_groups] * mtiles * nsplit;
  for (int unit = blockIdx.x; ok && unit < nunits; unit += gridDim.x) {
    const UmmaUnit U = umma_unit(pref, n_groups, mtiles, nsplit, unit);
    const int split = U.split;
    const int kc_begin = static_cast<int>(static_cast<int64_t>(split) * nkc / nsplit);
    const int nit = static_cast<int>(static_cast<int64_t>(split + 1) * nkc / nsplit) - kc_begin;
    const UmmaGroup G = umma_group(A, U.g);
    const int m0 = U.mt * UM_M;
    const int n_first = U.nt * A.n_tile, n_end = min(G.n, n_first + A.n_tile);
    for (int n0 = n_first; ok && n0 < n_end; n0 += A.n_tile) {
      const int nvalid = min(A.n_tile, G.n - n0);
      const int npad = (nvalid + 15) & ~15;
      const uint32_t idesc = umma_idesc(npad, A.mma_dt);
      // token table: source row of every token of this tile
      for (int n = tid; n < nvalid; n += UM_THREADS) {
        int row = n0 + n;
        if (A.experts) {
          const int pid = umma_pair(A, G.p0 + n0 + n);
          row = A.by_pair ? pid : pid / A.k;
        }
        tok_row[n] = row;
      }
      __syncthreads();

      // issue the copies of K-chunk kc (the tile's it-th) into ring slot it % S
      auto issue = [&](int kc, int it) {
        char* slot = base + static_cast<size_t>(it % S) * P.stage;
        const uint32_t sa = smem_u32(slot), sbb = smem_u32(slot + P.a_raw);
        const int k0 = kc * UM_KC;
        if (A.a_mode == UA_DENSE) {
          for (int c = tid; c < UM_M * 8; c += UM_THREADS) {
            const int r = c >> 3, j = c & 7;
            const int m = m0 + r, kk = k0 + 8 * j;
            const void* src = A.b0;
            uint32_t nbytes = 0;
            if (m < A.n_rows) {
              int si = 0;
              while (m >= A.seg[si].row0 + A.seg[si].rows) ++si;
              const DenseSeg& Sg = A.seg[si];
              for (int p = 0; p < Sg.nparts; ++p) {
                const DensePart& Pt = Sg.part[p];
                if (kk >= Pt.k0 && kk < Pt.k0 + Pt.wk) {
                  src = static_cast<const char*>(Pt.w) +
                        (static_cast<int64_t>(m - Sg.row0) * Pt.wk + (kk - Pt.k0)) * 2;
                  nbytes = 16;
                }
              }
            }
            cp_async16(sa + core_off(r, 8 * j), src, nbytes);
          }
        } else {
          // codes: row r = tid / 2, 32 codes (16 bytes) per half
          {
            const int r = tid >> 1, hh = tid & 1;
            const int m = min(m0 + r, A.n_rows - 1);
            const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
            const uint32_t nb = (m0 + r < A.n_rows) ? 16u : 0u;
            cp_async16(sa + r * 32 + hh * 16, A.q + row * (A.K >> 3) + (k0 >> 3) + 4 * hh, nb);
            if (gated)
              cp_async16(sa + UM_CODE_BYTES + UM_SB_BYTES + r * 32 + hh * 16,
                         A.q2 + row * (A.K >> 3) + (k0 >> 3) + 4 * hh, nb);
          }
          // scale/bias words of the chunk: one word per row (G >= 64), two (G = 32)
          if (tid < UM_M) {
            const int r = tid;
            const int m = min(m0 + r, A.n_rows - 1);
            const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
            const int gw = k0 / A.G;
            if (A.G == 32) {
              cp_async8(sa + UM_CODE_BYTES + r * 8, A.sb + row * ngr + gw);
              if (gated) cp_async8(sa + 2 * UM_CODE_BYTES + UM_SB_BYTES + r * 8, A.sb2 + row * ngr + gw);
            } else {
              cp_async4(sa + UM_CODE_BYTES + r * 8, A.sb + row * ngr + gw);
              if (gated) cp_async4(sa + 2 * UM_CODE_BYTES + UM_SB_BYTES + r * 8, A.sb2 + row * ngr + gw);
            }
          }
        }
        // B: npad tokens x 8 chunks of 16 bytes
        for (int c = tid; c < npad * 8; c += UM_THREADS) {
          const int n = c >> 3, j = c & 7;
          const void* src = A.b0;
          uint32_t nbytes = 0;
          if (n < nvalid) {
            src = static_cast<const char*>(A.b0) +
                  (A.b0_off + static_cast<int64_t>(tok_row[n]) * A.b0_stride + k0 + 8 * j) * 2;
            nbytes = 16;
          }
          cp_async16(sbb + core_off(n, 8 * j), src, nbytes);
        }
      };

      // dequantise the int4 codes of ring slot it % S into A tile buffer it & 1
      auto dequant = [&](int it) {
        const char* slot = base + static_cast<size_t>(it % S) * P.stage;
        const int r = tid >> 1, hh = tid & 1;
        for (int gsel = 0; gsel < (gated ? 2 : 1); ++gsel) {
          const char* raw = slot + gsel * (UM_CODE_BYTES + UM_SB_BYTES);
          char* dst = base + P.abuf + static_cast<size_t>((it & 1) + 2 * gsel) * UM_A_BYTES;
          const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 32 + hh * 16);
          const uint32_t sbw = *reinterpret_cast<const uint32_t*>(
              raw + UM_CODE_BYTES + r * 8 + ((A.G == 32) ? 4 * hh : 0));
          float s, b;
          sb_decode(sbw, A.s_dt, s, b);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t pr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = fmaf(s, code_f((ws[i] >> (8 * j)) & 0xFu), b);
              const float hi = fmaf(s, code_f((ws[i] >> (8 * j + 4)) & 0xFu), b);
              pr[j] = pack16(lo, hi, A.mma_dt);
            }
            *reinterpret_cast<uint4*>(dst + core_off(r, 32 * hh + 8 * i)) =
                make_uint4(pr[0], pr[1], pr[2], pr[3]);
          }
        }
      };

      // Ring protocol, chunk kc in slot kc % S: the copies of chunks up to
      // kc + S - 3 are in flight while chunk kc is computed.  Before a slot or
      // an A buffer is reused, the MMAs of chunk kc - 2 (which read them) must
      // be done -- two chunks back, so the tensor core's latency overlaps one
      // chunk of staging.
      auto wait_commit = [&](int b) -> bool {   // oldest unwaited commit on mbarrier b
        bool w = true;
        if (tid == 0) w = mbar_wait(smem_u32(&mbar[b]), waited[b] & 1u);
        ++waited[b];
        return w;
      };
      for (int s = 0; s < S - 2; ++s) {
        if (s < nit) issue(kc_begin + s, s);
        cp_async_commit();
      }
      for (int it = 0; it < nit; ++it) {
        const int kc = kc_begin + it;
        bool w = true;
        if (it >= 2) w = wait_commit(it & 1);       // chunk kc - 2 committed on mbarrier kc & 1
        cp_async_wait(S - 3);                        // this thread's copies of chunk kc
        if (!__syncthreads_and(w)) { ok = false; break; }
        if (it + S - 2 < nit) issue(kc + S - 2, it + S - 2);   // into slot (it - 2) % S
        cp_async_commit();
        if (A.a_mode == UA_INT4) dequant(it);
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
          const char* slot = base + static_cast<size_t>(it % S) * P.stage;
          const uint32_t a_addr = A.a_mode == UA_DENSE
                                      ? smem_u32(slot)
                                      : smem_u32(base + P.abuf + static_cast<size_t>(it & 1) * UM_A_BYTES);
          const uint32_t b_addr = smem_u32(slot + P.a_raw);
#pragma unroll
          for (int kk = 0; kk < UM_KC / 16; ++kk) {
            const uint64_t ad = umma_desc(a_addr + kk * 2 * UM_LBO);
            const uint64_t bd = umma_desc(b_addr + kk * 2 * UM_LBO);
            umma_f16(tmem, ad, bd, idesc, (it | kk) ? 1u : 0u);
            if (gated) {
              const uint32_t a2 = smem_u32(base + P.abuf + static_cast<size_t>((it & 1) + 2) * UM_A_BYTES);
              umma_f16(tmem + 256, umma_desc(a2 + kk * 2 * UM_LBO), bd, idesc, (it | kk) ? 1u : 0u);
            }
          }
          umma_commit(smem_u32(&mbar[it & 1]));
        }
        ++commits[it & 1];
      }
      if (!ok) break;
      cp_async_wait(0);
      {
        // the last (up to two) chunks' MMAs
        bool w = true;
        for (int b = 0; b < 2; ++b)
          while (waited[b] < commits[b]) w = wait_commit(b) && w;
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
          const int pid = A.experts ? umma_pair(A, G.p0 + n0 + n) : n0 + n;
          if (A.ksplit > 1) {
            A.part[(static_cast<int64_t>(split) * A.n_tokens + pid) * A.n_rows + m] = acc[i];
          } else {
            umma_epilogue(A, pid, m, acc[i], gated ? accg[i] : 0.f, gated, pid);
          }
        }
      }
      // all TMEM reads done before the next tile's MMAs overwrite the accumulators
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  }
  cp_async_wait(0);
  if (!ok && tid == 0) {
    atomicOr(A.status, STATUS_TIMEOUT);
    // bounded waits for MMAs still in flight before releasing TMEM
    for (int b = 0; b < 2; ++b)
      while (waited[b] < commits[b]) { mbar_wait(smem_u32(&mbar[b]), waited[b] & 1u); ++waited[b]; }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
  }
}

// Sums the split-K partials of a dense grouped launch and applies its epilogue.
__global__ void k_umma_reduce(const __grid_constant__ UmmaArgs A) {
  griddep_wait();
  griddep_launch();
  const int64_t n = static_cast<int64_t>(A.n_tokens) * A.n_rows;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / A.n_rows), m = static_cast<int>(i - static_cast<int64_t>(t) * A.n_rows);
    float v = 0.f;
    for (int sp = 0; sp < A.ksplit; ++sp) v += A.part[static_cast<int64_t>(sp) * n + i];
    umma_epilogue(A, t, m, v, 0.f, false, t);
  }
}

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

__global__ void k_prep_out(const __grid_constant__ PrepOutArgs A) {
  griddep_wait();
  griddep_launch();
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
