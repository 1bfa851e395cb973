// Device kernels of the quantized MoE decode layer (sm_103a).
//
// The layer (TensorFold PR #1038, Bolt latent MoE, "What's in it") is split
// into five launches, each an HBM-streaming pass over one set of weights:
//
//   k_dense_in   router gemv + fc1_latent_proj + shared-expert gate/up gemv:
//                every dense matrix that reads the layer input x, in one pass
//   k_route      sigmoid/softmax top-k per row, combine weights, and the list
//                of distinct selected experts with the rows routed to each
//   k_expert     int4 affine dequant gemv over the distinct experts; used for
//                the up(+gate) projection with the activation fused, and for
//                the down projection with the weighted combine (fp32, pick
//                order) fused into its last CTA per column range
//   k_dense_out  fc2_latent_proj, shared-expert down gemv and the residual,
//                rounded once to the activation dtype
//
// The shared expert does not depend on the routing: on its own stream its
// gate/up rows (k_dense_in) and down rows (k_dense_out, fp32 output) run while
// the routed chain runs, and the output kernel adds their result.
//
// Dense gemv design: a CTA owns a contiguous range of output rows (so every
// CTA streams the same number of bytes), its 256 threads stride the reduction
// axis of each row with 16-byte loads, every thread keeps partial sums for a
// batch of rows and all token rows of the pass, and the partials are reduced
// once per batch with a warp reduce-scatter and a cross-warp pass in shared
// memory.  The token rows are staged in shared memory as fp32 with an XOR
// swizzle so that the 16-byte reads of a warp phase hit distinct banks.
//
// Expert gemv design: one warp per weight row; a lane takes 32 packed codes
// (one 16-byte load, one quantisation group or part of one).  A code q becomes
// the float 1 + q/16 with one shift and one logic op (q placed in the top
// mantissa bits of 1.0f), so the inner product needs no integer conversion:
//   sum_k (s q_k + b) x_k = 16 s * sum_k (1 + q_k/16) x_k + (b - 16 s) * sum_k x_k
// per 32-element chunk, with the chunk sums of x computed once at staging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <cstdio>
#include <climits>

namespace moe {

constexpr int NT = 256;       // threads per CTA
constexpr int NW = NT / 32;   // warps per CTA
constexpr int RB = 4;         // dense rows per register batch
constexpr int MAXC = 2;       // 16-byte chunks per thread per row per round
constexpr int RED_ROWS = 64;  // dense rows per reduction round
constexpr int MAX_E = 1024;   // routed experts served
constexpr int MAX_K = 16;     // top-k served

enum : int { DT_BF16 = 0, DT_FP16 = 1, DT_FP32 = 2 };
enum : int { ACT_SWIGLU = 0, ACT_RELU2 = 1 };
enum : int { ROUTER_SOFTMAX = 0, ROUTER_SIGMOID = 1 };
enum : int { STATUS_NONFINITE = 1, STATUS_TIMEOUT = 2, STATUS_INDEX = 4 };

// ---------------------------------------------------------------------------
// index checks (builds with MOE_CHECKS=1)
// ---------------------------------------------------------------------------
// The indices a kernel reads from data -- an expert id or a token-pair id taken
// from the route metadata -- are checked against their bound before they
// address memory.  A violation sets STATUS_INDEX in status word 0 and the first
// one stores (site, index, bound) in words 1..3; the caller then skips the
// access or substitutes index 0, so the kernel neither traps nor reads outside
// a buffer.  Every other index of these kernels is a loop counter over launch
// sizes checked on the host.  In the default build a check is `true`.
#ifndef MOE_CHECKS
#define MOE_CHECKS 0
#endif
enum : int {
  CK_EXPERT_E = 1,     // k_expert: distinct expert id
  CK_EXPERT_PAIR = 2,  // k_expert: pair id of a staged input / output row
  CK_BULK_E = 3,       // k_expert_bulk: distinct expert id
  CK_BULK_PAIR = 4,    // k_expert_bulk: pair id
  CK_GATHER_PAIR = 5,  // k_gather_pairs: pair id
  CK_UMMA_E = 6,       // grouped GEMMs: expert id of a group
  CK_UMMA_PAIR = 7,    // grouped GEMMs: pair id of a token slot
  CK_PREFETCH_E = 8,   // routing CTA: expert id of an L2 prefetch
  CK_SLOT_RANGE = 9    // pair range [p0, p1) of a distinct expert outside [0, T*k]
};

#if MOE_CHECKS
static __device__ __noinline__ void check_fail(int* status, int site, long long idx, long long bound) {
  if (!status) return;
  atomicOr(status, STATUS_INDEX);
  if (atomicCAS(status + 1, 0, site) == 0) {
    status[2] = static_cast<int>(idx);
    status[3] = static_cast<int>(bound);
  }
}
#endif

__device__ __forceinline__ bool idx_ok(int* status, int site, long long idx, long long bound) {
#if MOE_CHECKS
  if (idx >= 0 && idx < bound) return true;
  check_fail(status, site, idx, bound);
  return false;
#else
  (void)status; (void)site; (void)idx; (void)bound;
  return true;
#endif
}

// a distinct expert's pair range: 0 <= p0 <= p1 <= n_pairs
__device__ __forceinline__ bool range_ok(int* status, long long p0, long long p1, long long n_pairs) {
#if MOE_CHECKS
  if (p0 >= 0 && p0 <= p1 && p1 <= n_pairs) return true;
  check_fail(status, CK_SLOT_RANGE, p0 < 0 || p0 > p1 ? p0 : p1, n_pairs + 1);
  return false;
#else
  (void)status; (void)p0; (void)p1; (void)n_pairs;
  return true;
#endif
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

// Streaming loads of read-only weights.  Volatile so that the compiler keeps
// them in program order and issues a batch of them before the first use
// (a plain asm statement may be sunk next to its use, which serialises the
// memory latency of every load).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Programmatic dependent launch: wait for the preceding kernel of the stream
// (a no-op when launched without the attribute) / let the next one launch.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// Asynchronous prefetch of [p, p + bytes) into L2 by the bulk-copy engine.
// The bulk prefetch needs a 16-byte aligned start and a size that is a
// multiple of 16, so the range is widened to 16-byte bounds (every buffer the
// library prefetches from is allocated with at least 256 bytes of padding).
__device__ __forceinline__ void prefetch_l2(const void* p, int64_t bytes) {
  if (bytes <= 0) return;
  uint64_t a = reinterpret_cast<uint64_t>(p) & ~uint64_t(15);
  const uint64_t e = (reinterpret_cast<uint64_t>(p) + static_cast<uint64_t>(bytes) + 15) &
                     ~uint64_t(15);
  for (; a < e; a += 65536) {
    const uint64_t rem = e - a;
    const uint32_t n = static_cast<uint32_t>(rem < 65536 ? rem : 65536);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(n) : "memory");
  }
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float f16lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xffffu)));
}
__device__ __forceinline__ float f16hi(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

// 16-bit scalar load (act / scale dtype) to fp32
__device__ __forceinline__ float ld16(const void* base, int64_t i, int dt) {
  const unsigned short u = reinterpret_cast<const unsigned short*>(base)[i];
  return dt == DT_BF16 ? __uint_as_float(static_cast<uint32_t>(u) << 16)
                       : __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ float ld_any(const void* base, int64_t i, int dt) {
  if (dt == DT_FP32) return reinterpret_cast<const float*>(base)[i];
  return ld16(base, i, dt);
}

__device__ __forceinline__ unsigned short st16_bits(float v, int dt) {
  return dt == DT_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                       : __half_as_ushort(__float2half_rn(v));
}

// 8 elements of a 16-bit chunk to fp32
__device__ __forceinline__ void cvt8(const uint4 v, int dt, float f[8]) {
  if (dt == DT_BF16) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
  } else {
    f[0] = f16lo(v.x); f[1] = f16hi(v.x); f[2] = f16lo(v.y); f[3] = f16hi(v.y);
    f[4] = f16lo(v.z); f[5] = f16hi(v.z); f[6] = f16lo(v.w); f[7] = f16hi(v.w);
  }
}

// code q (bits 4n..4n+3 of w) -> float 1 + q/16
template <int N>
__device__ __forceinline__ float nib(uint32_t w) {
  uint32_t t = (N <= 4) ? (w << (19 - 4 * N)) : (w >> (4 * N - 19));
  return __uint_as_float((t & 0x00780000u) | 0x3f800000u);
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ float act_fn(int act, float g, float u) {
  if (act == ACT_SWIGLU) return silu(g) * u;
  const float r = fmaxf(u, 0.0f);
  return r * r;
}

// Swizzled float4 slot of element-float4 index f4 for readers that take
// (nf4m1 + 1) consecutive float4 per 16-byte weight chunk.
__device__ __forceinline__ int swz(int f4, int nf4m1) { return f4 ^ ((f4 >> 3) & nf4m1); }

// Reduce NV values held by every lane of a warp.  Afterwards the lane with
// (lane & (32/NV - 1)) == 0 holds the warp total of value (lane / (32/NV)).
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV], int lane) {
  static_assert(NV == 1 || NV == 2 || NV == 4 || NV == 8 || NV == 16 || NV == 32, "NV");
  int n = NV;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (lane & o) != 0;
      const int half = n >> 1;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

// ---------------------------------------------------------------------------
// routing arguments
// ---------------------------------------------------------------------------

// Route metadata (int32 buffer):
//   [0]                      n_uniq
//   [1, 1 + umax)            uniq_e[u]   distinct selected experts, ascending
//   [1 + umax, 2 + 2 umax)   uniq_p0[u]  first position of u's pairs (u = n_uniq: total)
//   [2 + 2 umax, ...)        pairs[i]    pair ids t*k + j grouped by expert, t ascending
struct RouteArgs {
  const float* logits;   // dense_in, row stride r_in, experts at columns [0, E)
  int r_in;
  const float* bias;     // [E] or null
  int E, k, T;
  int router, renorm;
  float scale;
  int* ids;              // [T*k]
  float* w;              // [T*k]
  int* meta;
  int umax;
  int* ext_ids;          // optional copies for the caller
  float* ext_w;
  int* status;
  int mask_words;        // > 0: rank pairs with per-expert row bitmasks of this many
                         // words in dynamic shared memory (E * mask_words words)
  int debug_times;       // print per-phase timestamps (diagnostics only)
  int topk_only;         // 1: ids and weights only (the lists come from k_route_lists)
  int rows_per_cta;      // k_route_rows: rows of one CTA (fewer rows: more warps per row)
  int max_w;             // route_block: most warps sharing a row's keys (1..8)
  int dry;               // 1: run the top-k code without writing anything (warms the
                         // instruction cache and the bias lines before the logits exist)
  int debug_bad;         // MOE_CHECKS builds, few-pair lists only: plant an out-of-range
                         // index in the metadata (1: first expert id = E + 3, 2: first
                         // pair id = T*k + 5) for the consumers' checks to catch
};

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Diagnostics (MOE_CTA_TRACE): per-CTA global-timer stamps of a launch --
// 0 entry, 1 past the wait for the previous kernel, 2 main loop done, 3 exit;
// 4..15 kernel-specific intermediate points.
constexpr int CT_MAX_CTAS = 2048;
constexpr int CT_STAMPS = 16;
constexpr int CT_SLOTS = 12;   // launches stamped per forward
__device__ __forceinline__ void cta_stamp(unsigned long long* t, int i) {
  if (t != nullptr && threadIdx.x == 0 && blockIdx.x < CT_MAX_CTAS) {
    t[blockIdx.x * CT_STAMPS + i] = global_ns();
    // the SM clock at entry and exit (slots 14, 15): cycles per ns of the CTA
    if (i == 0 || i == 3) t[blockIdx.x * CT_STAMPS + (i == 0 ? 14 : 15)] = clock64();
  }
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded spin of one thread until *p >= target (false when the bound ran out).
constexpr uint32_t SPIN_LIMIT = 1u << 22;   // polls (~0.2 s with the sleeps)
__device__ __forceinline__ bool spin_until_geq(const int* p, int target, uint32_t limit = SPIN_LIMIT) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ld_acquire_gpu(p) >= target) return true;
    __nanosleep(40);
  }
  return false;
}

__device__ __forceinline__ bool key_better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Signed integers in the order of the floats (for keys without NaN and -0).
__device__ __forceinline__ int ordered_bits(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : (b ^ 0x7fffffff);
}
__device__ __forceinline__ float from_ordered_bits(int b) {
  return __int_as_float(b >= 0 ? b : (b ^ 0x7fffffff));
}

// Shared memory of route_block: two int arrays of MAX_E and 2 x 32 ints, plus
// E * mask_words words of row bitmasks when A.mask_words > 0.
constexpr int ROUTE_CAND_WORDS = 32 * MAX_K * 3;   // per-warp candidate lists (32 warps max)
constexpr int ROUTE_SMEM_BYTES = (2 * MAX_E + 64 + ROUTE_CAND_WORDS) * 4;

// Routing of all T rows by one CTA (any block size that is a multiple of 32):
// top-k per row by warp-shuffle selection, the combine weights, then the
// distinct selected experts (ascending) with their (row, pick) pairs in row
// order.  Logits are read with ld.global.cg, so this may run in the last CTA
// of the kernel that produced them.

// k rounds of selection over register-held keys.  Every round takes the
// lane's best remaining key with a pairwise tree (keys as order-preserving
// integers, ties to the smaller expert id, its weight input carried along),
// then the warp's largest key by a warp max and, among the lanes that hold
// it, the smallest expert id by a warp min: pick j.  The lane that holds it
// writes its key, id and weight input to ck/ci/cs[j] (ck and ci may be null;
// cs is the warp's scratch of MAX_K) and retires it.  Lane j ends with pick
// j (its expert id and its weight input).  The two warp reductions are the
// round's only collectives.
template <int NPL>
__device__ __forceinline__ void topk_rounds(float (&kv)[NPL], const int (&ev)[NPL], const float (&sv)[NPL],
                                            int k, int lane, int& my_id, float& my_z, float* ck,
                                            int* ci, float* cs) {
  int ik[NPL];   // keys carry no -0 and no NaN
#pragma unroll
  for (int i = 0; i < NPL; ++i) ik[i] = ordered_bits(kv[i]);
  for (int j = 0; j < k; ++j) {
    int tk[NPL], tix[NPL];
    float ts[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) { tk[i] = ik[i]; tix[i] = ev[i]; ts[i] = sv[i]; }
#pragma unroll
    for (int w = NPL / 2; w >= 1; w >>= 1) {
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const bool b1 = tk[i + w] > tk[i] || (tk[i + w] == tk[i] && tix[i + w] < tix[i]);
        tk[i] = b1 ? tk[i + w] : tk[i];
        tix[i] = b1 ? tix[i + w] : tix[i];
        ts[i] = b1 ? ts[i + w] : ts[i];
      }
    }
    const int mx = __reduce_max_sync(0xffffffffu, tk[0]);
    const int bi = static_cast<int>(__reduce_min_sync(
        0xffffffffu, tk[0] == mx ? static_cast<unsigned>(tix[0]) : 0xffffffffu));
    if (tk[0] == mx && tix[0] == bi) {
      cs[j] = ts[0];
      if (ck) { ck[j] = from_ordered_bits(mx); ci[j] = bi; }
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (ev[i] == bi) ik[i] = INT_MIN;
    if (lane == j) my_id = bi;
  }
  __syncwarp();
  my_z = lane < k ? cs[lane] : 0.f;
  __syncwarp();
}

// Keys of one member warp: experts lane + 32 * (g + W * i), i < NPL.
template <int NPL>
__device__ __forceinline__ void route_member(const RouteArgs& A, const float* z, int W, int g, int lane,
                                             int& my_id, float& my_z, float* ck, int* ci, float* cs,
                                             bool& bad) {
  float kv[NPL], sv[NPL];
  int ev[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * (g + W * i);
    const bool ok = e < A.E;
    ev[i] = ok ? e : 0x7fffffff;
    sv[i] = ok ? __ldcg(z + e) : 0.f;
    kv[i] = (ok && A.bias) ? __ldg(A.bias + e) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (ev[i] < A.E) {
      const float zz = sv[i];
      float key;
      if (A.router == ROUTER_SOFTMAX) {
        key = zz;                          // softmax weights use the logit
      } else {
        const float sg = 1.0f / (1.0f + expf(-zz));
        key = sg + kv[i];                  // selection key: score + bias
        sv[i] = sg;                        // weight: score without bias
      }
      if (!isfinite(key)) { bad = true; key = -INFINITY; }
      kv[i] = key + 0.0f;   // -0 -> +0: equal keys compare equal as integers too
    } else {
      kv[i] = -INFINITY;
    }
  }
  topk_rounds<NPL>(kv, ev, sv, A.k, lane, my_id, my_z, ck, ci, cs);
}

// The warp-level phases of route_block, each compiled as its own function (not
// inlined) so that a dry run can execute all of them at once, one per warp
// (route_warm): the first run of each fetches its instructions from a cold L2,
// and in parallel warps those fetches overlap instead of adding up.
struct RoutePick {
  int id;      // lane j < k: pick j's expert id
  float z;     // its weight input (logit or sigmoid score)
  int bad;     // a selection key of the warp's slice was not finite
};

// One member warp's top-k over its slice of the experts (route_member).
template <int NPL>
static __device__ __noinline__ RoutePick route_member_fn(const RouteArgs& A, const float* z, int W, int g,
                                                         float* ck, int* ci, float* cs) {
  RoutePick r{-1, 0.f, 0};
  bool bad = false;
  route_member<NPL>(A, z, W, g, threadIdx.x & 31, r.id, r.z, ck, ci, cs, bad);
  r.bad = bad ? 1 : 0;
  return r;
}

// The first warp of a row's group merges the W member lists of k picks.
static __device__ __noinline__ RoutePick route_merge_fn(const float* cand_k, const int* cand_i,
                                                        float* cand_s, int warp, int W, int k) {
  const int lane = threadIdx.x & 31;
  RoutePick r{-1, 0.f, 0};
  float kv[4], sv[4];
  int ev[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;            // candidate c of W * k
    const int wl = c / k, jl = c - wl * k;
    const bool ok = c < W * k;
    kv[i] = ok ? cand_k[(warp + wl) * MAX_K + jl] : -INFINITY;
    ev[i] = ok ? cand_i[(warp + wl) * MAX_K + jl] : 0x7fffffff;
    sv[i] = ok ? cand_s[(warp + wl) * MAX_K + jl] : 0.f;
  }
  topk_rounds<4>(kv, ev, sv, k, lane, r.id, r.z, nullptr, nullptr, cand_s + warp * MAX_K);
  return r;
}

// Combine weights of row t (lane j < k holds pick j; its z is the logit for
// softmax routing and the sigmoid score for sigmoid routing; zs[j] holds pick
// j's z for every lane), written unless dry.  Renormalising sums run over the
// picks in order j = 0..k-1.  With few pairs (T k <= 32) the ids also go to
// s_ids[t k + j] for the lists.
static __device__ __noinline__ void route_weights_fn(const RouteArgs& A, const float* z, int t, int my_id,
                                                     float my_z, const float* zs, int* s_ids) {
  // the arguments' fields, read once before any store
  const int lane = threadIdx.x & 31, k = A.k, E = A.E, T = A.T;
  const bool softmax = A.router == ROUTER_SOFTMAX, renorm = A.renorm != 0, dry = A.dry != 0;
  const float scale = A.scale;
  int* ids = A.ids;
  float* w = A.w;
  int* ext_ids = A.ext_ids;
  float* ext_w = A.ext_w;
  const float zj = (lane < k) ? my_z : 0.f;
  float wv = 0.f;
  if (softmax) {
    const float m = zs[0];   // the largest selected logit
    if (renorm) {
      float den = 0.f;
      for (int j = 0; j < k; ++j) den += expf(zs[j] - m);
      wv = (lane < k) ? expf(zj - m) / den : 0.f;
    } else {
      float mm = -INFINITY, den = 0.f;
      for (int i = lane; i < E; i += 32) mm = fmaxf(mm, __ldcg(z + i));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
      for (int i = lane; i < E; i += 32) den += expf(__ldcg(z + i) - mm);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      wv = (lane < k) ? expf(zj - mm) / den : 0.f;
    }
  } else {
    wv = zj;
    if (renorm) {
      float den = 0.f;
      for (int j = 0; j < k; ++j) den += zs[j];
      wv = zj / den;
    }
  }
  wv *= scale;
  if (lane < k && T * k <= 32) s_ids[t * k + lane] = my_id;
  if (lane < k && !dry) {
    ids[t * k + lane] = my_id;
    w[t * k + lane] = wv;
    if (ext_ids) ext_ids[t * k + lane] = my_id;
    if (ext_w) ext_w[t * k + lane] = wv;
  }
}

// Few pairs (T k <= 32): one warp sorts the pairs by (expert, pair): pair p's
// rank is the number of pairs with a smaller (expert, pair) key, and it goes
// to that place in s_ids[32..64); the first pair of each expert opens its
// group.  The pairs' ids come from s_ids[0..P) (written by route_weights_fn).
// Writes the route metadata unless dry.
static __device__ __noinline__ void route_lists_few_fn(const RouteArgs& A, int* s_ids) {
  const int lane = threadIdx.x & 31;
  const int P = A.T * A.k;
  int v = lane < P ? ((s_ids[lane] << 5) | lane) : 0x7fffffff;
  int rank = 0;
  for (int q = 0; q < P; ++q) rank += __shfl_sync(0xffffffffu, v, q) < v;
  int* s_sorted = s_ids + 32;
  if (lane < P) s_sorted[rank] = v;
  __syncwarp();
  v = lane < P ? s_sorted[lane] : 0x7fffffff;
  __syncwarp();
  const bool valid = lane < P;
  const int prev = __shfl_up_sync(0xffffffffu, v, 1);
  const bool open = valid && (lane == 0 || (prev >> 5) != (v >> 5));
  const unsigned om = __ballot_sync(0xffffffffu, open);
  const int u = __popc(om & ((2u << lane) - 1u)) - 1;
  int* uniq_e = A.meta + 1;
  int* uniq_p0 = A.meta + 1 + A.umax;
  int* pairs = A.meta + 2 + 2 * A.umax;
  if (!A.dry) {
    if (open) { uniq_e[u] = v >> 5; uniq_p0[u] = lane; }
    if (valid) pairs[lane] = v & 31;
    if (lane == 0) { A.meta[0] = __popc(om); uniq_p0[__popc(om)] = P; }
#if MOE_CHECKS
    if (lane == 0 && A.debug_bad == 1) uniq_e[0] = A.E + 3;
    if (lane == 0 && A.debug_bad == 2) pairs[0] = P + 5;
#endif
  }
}

// Warps per row of route_block and the keys a lane holds.
__device__ __forceinline__ void route_shape(const RouteArgs& A, int nwarp, int* W, int* npl) {
  int w = A.E > 16 * 32 ? 2 : 1;            // at most 16 keys per lane
  while (w < A.max_w && A.T * w * 2 <= nwarp) w *= 2;
  *W = w;
  *npl = (A.E + 32 * w - 1) / (32 * w);
}

template <int NPL>
__device__ __forceinline__ RoutePick route_member_call(const RouteArgs& A, const float* z, int W, int g, float* ck,
                                                       int* ci, float* cs) {
  return route_member_fn<NPL>(A, z, W, g, ck, ci, cs);
}
__device__ __forceinline__ RoutePick route_member_any(const RouteArgs& A, int npl, const float* z, int W, int g,
                                                      float* ck, int* ci, float* cs) {
  if (npl <= 1) return route_member_call<1>(A, z, W, g, ck, ci, cs);
  if (npl <= 2) return route_member_call<2>(A, z, W, g, ck, ci, cs);
  if (npl <= 4) return route_member_call<4>(A, z, W, g, ck, ci, cs);
  if (npl <= 8) return route_member_call<8>(A, z, W, g, ck, ci, cs);
  return route_member_call<16>(A, z, W, g, ck, ci, cs);
}

// A dry run of route_block's warp-level phases, one per warp at once (reads
// the buffers as they stand, writes no global memory; D.dry must be set).
static __device__ void route_warm(const RouteArgs& D, int* smem) {
  const int warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  float* cand_k = reinterpret_cast<float*>(smem + 2 * MAX_E + 64);
  int* cand_i = reinterpret_cast<int*>(cand_k + 32 * MAX_K);
  float* cand_s = reinterpret_cast<float*>(cand_i + 32 * MAX_K);
  int W, npl;
  route_shape(D, nwarp, &W, &npl);
  RoutePick r{-1, 0.f, 0};
  if (warp == 0) {
    r = route_member_any(D, npl, D.logits, W, 0, W > 1 ? cand_k + warp * MAX_K : nullptr,
                         cand_i + warp * MAX_K, cand_s + warp * MAX_K);
  } else if (warp == 1 % nwarp) {
    r = route_merge_fn(cand_k, cand_i, cand_s, 0, 1, D.k);
  } else if (warp == 2 % nwarp) {
    route_weights_fn(D, D.logits, 0, r.id, r.z, cand_s + warp * MAX_K, smem);
  } else if (warp == 3 % nwarp && D.T * D.k <= 32 && !D.topk_only) {
    route_lists_few_fn(D, smem + 32);
  }
  (void)r;
  __syncthreads();
}

static __device__ __noinline__ void route_block(const RouteArgs& A, int* smem) {
  int* s_cnt = smem;
  int* s_scan_c = smem + MAX_E;
  int* s_wsum_u = smem + 2 * MAX_E;
  int* s_wsum_c = s_wsum_u + 32;
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + 2 * MAX_E + 64 + ROUTE_CAND_WORDS);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  const int nthr = blockDim.x;
  const int E = A.E, k = A.k;
  unsigned long long tp[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (A.debug_times) tp[0] = global_ns();

  // W warps cooperate on one row (more when there are few rows), each with
  // its slice of the experts; the first warp of the group merges their lists
  float* cand_k = reinterpret_cast<float*>(smem + 2 * MAX_E + 64);
  int* cand_i = reinterpret_cast<int*>(cand_k + 32 * MAX_K);
  float* cand_s = reinterpret_cast<float*>(cand_i + 32 * MAX_K);
  int W, npl;
  route_shape(A, nwarp, &W, &npl);
  const int rows_per_pass = nwarp / W;
  for (int tb = 0; tb < A.T; tb += rows_per_pass) {
    const int t = tb + warp / W, g = warp % W;
    const bool active = t < A.T;
    const float* z = A.logits + static_cast<int64_t>(active ? t : 0) * A.r_in;
    RoutePick r{-1, 0.f, 0};
    float* ck = (W > 1) ? cand_k + warp * MAX_K : nullptr;
    int* ci = cand_i + warp * MAX_K;
    float* cs = cand_s + warp * MAX_K;
    if (active) {
      r = route_member_any(A, npl, z, W, g, ck, ci, cs);
      if (__any_sync(0xffffffffu, r.bad) && lane == 0 && !A.dry) atomicOr(A.status, STATUS_NONFINITE);
    }
    if (A.debug_times && tb == 0) tp[5] = global_ns();
    if (W > 1) {
      __syncthreads();
      if (A.debug_times && tb == 0) tp[6] = global_ns();
      if (active && g == 0) r = route_merge_fn(cand_k, cand_i, cand_s, warp, W, k);
    }
    if (A.debug_times && tb == 0) tp[7] = global_ns();
    if (active && g == 0) route_weights_fn(A, z, t, r.id, r.z, cand_s + warp * MAX_K, s_cnt);
    if (W > 1) __syncthreads();
  }
  if (A.topk_only) return;
  // ---- distinct experts and their pairs ----
  if (A.debug_times) tp[1] = global_ns();
  if (A.T * k <= 32) {
    // few pairs: one warp sorts them (route_lists_few_fn)
    __syncthreads();
    if (warp == 0) route_lists_few_fn(A, s_cnt);
    if (A.debug_times && tid == 0)
      printf("route phases (ns): topk %llu (member %llu sync %llu merge %llu weights %llu) list %llu\n",
             tp[1] - tp[0], tp[5] - tp[0], tp[6] - tp[5], tp[7] - tp[6], tp[1] - tp[7],
             global_ns() - tp[1]);
    return;
  }
  for (int e = tid; e < MAX_E; e += nthr) s_cnt[e] = 0;
  __syncthreads();
  if (A.debug_times) tp[2] = global_ns();
  const int P = A.T * k;
  for (int p = tid; p < P; p += nthr) atomicAdd(&s_cnt[A.ids[p]], 1);
  __syncthreads();
  if (A.debug_times) tp[3] = global_ns();
  // exclusive scans over experts of (cnt > 0) and cnt; thread tid owns the
  // experts [tid * ept, (tid + 1) * ept)
  {
    const int ept = MAX_E / nthr;
    int lu = 0, lc = 0;
    for (int i = 0; i < ept; ++i) {
      const int e = tid * ept + i;
      const int c = (e < E) ? s_cnt[e] : 0;
      lu += (c > 0);
      lc += c;
    }
    int iu = lu, ic = lc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, iu, o);
      const int b = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) { iu += a; ic += b; }
    }
    if (lane == 31) { s_wsum_u[warp] = iu; s_wsum_c[warp] = ic; }
    __syncthreads();
    if (warp == 0) {
      int a = (lane < nwarp) ? s_wsum_u[lane] : 0;
      int b = (lane < nwarp) ? s_wsum_c[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, a, o);
        const int y = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) { a += x; b += y; }
      }
      s_wsum_u[lane] = a;  // inclusive prefix over warps
      s_wsum_c[lane] = b;
    }
    __syncthreads();
    int pu = (warp ? s_wsum_u[warp - 1] : 0) + iu - lu;
    int pc = (warp ? s_wsum_c[warp - 1] : 0) + ic - lc;
    int* uniq_e = A.meta + 1;
    int* uniq_p0 = A.meta + 1 + A.umax;
    for (int i = 0; i < ept; ++i) {
      const int e = tid * ept + i;
      const int c = (e < E) ? s_cnt[e] : 0;
      s_scan_c[e] = pc;
      if (c > 0) { uniq_e[pu] = e; uniq_p0[pu] = pc; ++pu; }
      pc += c;
    }
    if (tid == nthr - 1) {
      A.meta[0] = pu;
      uniq_p0[pu] = pc;
    }
  }
  __syncthreads();
  if (A.debug_times) tp[4] = global_ns();
  int* pairs = A.meta + 2 + 2 * A.umax;
  if (A.mask_words > 0) {
    // rank of pair (t, j) among its expert's pairs = rows t' < t that chose
    // the same expert (a row picks an expert at most once)
    const int W = A.mask_words;
    for (int i = tid; i < E * W; i += nthr) s_mask[i] = 0u;
    __syncthreads();
    for (int p = tid; p < P; p += nthr) {
      const int t = p / k;
      atomicOr(&s_mask[A.ids[p] * W + (t >> 5)], 1u << (t & 31));
    }
    __syncthreads();
    for (int p = tid; p < P; p += nthr) {
      const int e = A.ids[p], t = p / k;
      const uint32_t* m = s_mask + e * W;
      int rank = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
      for (int w = 0; w < (t >> 5); ++w) rank += __popc(m[w]);
      pairs[s_scan_c[e] + rank] = p;
    }
  } else {
    for (int p = tid; p < P; p += nthr) {
      const int e = A.ids[p];
      int rank = 0;
      for (int q = 0; q < p; ++q) rank += (A.ids[q] == e);
      pairs[s_scan_c[e] + rank] = p;
    }
  }
  if (A.debug_times && tid == 0) {
    tp[5] = global_ns();
    printf("route phases (ns): topk %llu zero %llu count %llu scan %llu pairs %llu\n",
           tp[1] - tp[0], tp[2] - tp[1], tp[3] - tp[2], tp[4] - tp[3], tp[5] - tp[4]);
  }
}

// The routing kernel of the grouped path: one warp per row for up to 16 rows
// (route_block adapts to the block size; ~90 registers a thread).
constexpr int ROUTE_THREADS = 512;

// Routing of many rows (prefill): k_route_rows selects the top-k of
// ROUTE_ROWS_PER_CTA rows per CTA (ids and weights only), then one CTA of
// k_route_lists builds the distinct-expert lists.  A pair's place among its
// expert's pairs (row order) comes from per-expert row bitmasks: the number of
// earlier rows that chose the expert is a popcount prefix over the bitmask.
constexpr int ROUTE_ROWS_PER_CTA = 16;
constexpr int ROUTE_SMALL_T = 64;   // up to this many rows one k_route CTA does both
constexpr int LIST_THREADS = 1024;
static_assert(LIST_THREADS == MAX_E, "k_route_lists scans one expert per thread");

struct ListArgs {
  const int* ids;   // [T*k]
  int T, k, E, umax;
  int* meta;
  uint32_t* mask;   // [E][W] bit t of word t/32: row t chose the expert
  int* pref;        // [E][W] set bits in the expert's words before word w
  int W;            // (T + 31) / 32
};

static __global__ void __launch_bounds__(LIST_THREADS) k_route_lists(const __grid_constant__ ListArgs A) {
  __shared__ int s_cnt[MAX_E];
  __shared__ int s_base[MAX_E];
  __shared__ int s_wu[32], s_wc[32];
  griddep_wait();
  griddep_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int P = A.T * A.k, E = A.E, W = A.W;
  for (int64_t i = tid; i < static_cast<int64_t>(E) * W; i += nthr) A.mask[i] = 0u;
  __syncthreads();
  for (int p = tid; p < P; p += nthr) {
    const int e = A.ids[p], t = p / A.k;
    atomicOr(&A.mask[static_cast<int64_t>(e) * W + (t >> 5)], 1u << (t & 31));
  }
  __syncthreads();
  for (int e = tid; e < MAX_E; e += nthr) {
    int acc = 0;
    if (e < E) {
      for (int w = 0; w < W; ++w) {
        A.pref[static_cast<int64_t>(e) * W + w] = acc;
        acc += __popc(__ldcg(&A.mask[static_cast<int64_t>(e) * W + w]));
      }
    }
    s_cnt[e] = acc;
  }
  __syncthreads();
  // exclusive scans over experts (one expert per thread) of (count > 0) and count
  {
    const int e = tid;   // LIST_THREADS == MAX_E
    const int c = s_cnt[e];
    int iu = c > 0 ? 1 : 0, ic = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, iu, o);
      const int b = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) { iu += a; ic += b; }
    }
    if (lane == 31) { s_wu[warp] = iu; s_wc[warp] = ic; }
    __syncthreads();
    if (warp == 0) {
      int a = s_wu[lane], b = s_wc[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, a, o);
        const int y = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) { a += x; b += y; }
      }
      s_wu[lane] = a;
      s_wc[lane] = b;
    }
    __syncthreads();
    const int pu = (warp ? s_wu[warp - 1] : 0) + iu - (c > 0 ? 1 : 0);
    const int pc = (warp ? s_wc[warp - 1] : 0) + ic - c;
    s_base[e] = pc;
    int* uniq_e = A.meta + 1;
    int* uniq_p0 = A.meta + 1 + A.umax;
    if (c > 0) { uniq_e[pu] = e; uniq_p0[pu] = pc; }
    if (e == MAX_E - 1) {
      A.meta[0] = pu + (c > 0 ? 1 : 0);
      uniq_p0[pu + (c > 0 ? 1 : 0)] = P;
    }
  }
  __syncthreads();
  int* pairs = A.meta + 2 + 2 * A.umax;
  for (int p = tid; p < P; p += nthr) {
    const int e = A.ids[p], t = p / A.k, w = t >> 5;
    const int64_t o = static_cast<int64_t>(e) * W + w;
    const int r = __ldcg(&A.pref[o]) + __popc(__ldcg(&A.mask[o]) & ((1u << (t & 31)) - 1u));
    pairs[s_base[e] + r] = p;
  }
}

static __global__ void __launch_bounds__(ROUTE_THREADS) k_route_rows(const __grid_constant__ RouteArgs A) {
  extern __shared__ int route_smem[];
  griddep_wait();
  griddep_launch();
  RouteArgs B = A;
  const int rpc = A.rows_per_cta > 0 ? A.rows_per_cta : ROUTE_ROWS_PER_CTA;
  const int t0 = blockIdx.x * rpc;
  B.T = min(rpc, A.T - t0);
  B.logits = A.logits + static_cast<int64_t>(t0) * A.r_in;
  B.ids = A.ids + t0 * A.k;
  B.w = A.w + t0 * A.k;
  if (A.ext_ids) B.ext_ids = A.ext_ids + t0 * A.k;
  if (A.ext_w) B.ext_w = A.ext_w + t0 * A.k;
  B.topk_only = 1;
  B.mask_words = 0;
  route_block(B, route_smem);
}

static __global__ void __launch_bounds__(ROUTE_THREADS) k_route(const __grid_constant__ RouteArgs A) {
  extern __shared__ int route_smem[];
  unsigned long long t0 = 0, t1 = 0;
  if (A.debug_times) t0 = global_ns();
  griddep_wait();
  if (A.debug_times) t1 = global_ns();
  griddep_launch();
  route_block(A, route_smem);
  if (A.debug_times && threadIdx.x == 0)
    printf("route kernel: wait %llu ns, total %llu ns\n", t1 - t0, global_ns() - t0);
}

// ---------------------------------------------------------------------------
// dense gemv (k_dense_in / k_dense_out)
// ---------------------------------------------------------------------------

// One weight matrix of a row segment, reading the staged vector at
// [k0, k0 + wk).  Row r of the segment is at w + r * wk elements.
struct DensePart {
  const void* w;
  int dt;
  int k0;
  int wk;
};

// Consecutive output rows [row0, row0 + rows) computed from up to two parts
// (concatenated along the reduction axis).
struct DenseSeg {
  DensePart part[2];
  int nparts;
  int row0;
  int rows;
};

struct DenseInArgs {
  DenseSeg seg[4];
  int nseg;
  int total_rows;
  int K;             // staged vector length (hidden)
  const void* x;     // [T, K] act dtype
  int x_dt;
  float* out;        // [T, out_ld] fp32, rows [0, total_rows)
  int out_ld;
  int T;
  // routing fused into the CTA that finishes the router rows last
  int fuse_route;
  int route_ctas;    // CTAs whose row range meets the router rows [0, E)
  int* route_counter;
  int route_warm;    // 1: CTA 0 holds no rows; it warms the top-k code with a dry
                     // run, waits (bounded) for CTAs 1..route_ctas to write the
                     // router rows, then routes
  int debug_stall;   // tests only: CTA 0 waits for one router CTA more than exist
                     // (the bounded wait runs out and reports a timeout)
  RouteArgs route;
  // after routing, prefetch the distinct experts' up(+gate) weights into L2
  int prefetch_up;
  int64_t pf_budget;         // at most this many bytes
  const uint32_t* pf_q; const uint32_t* pf_sb; const uint32_t* pf_q2; const uint32_t* pf_sb2;
  int64_t pf_q_bytes, pf_sb_bytes;   // per expert
  unsigned long long* trace;   // diagnostics: CTA stamps or null
  int dep_tail;      // 1: rows that need nothing from the previous kernel: let the
                     // next kernel launch at once, run without waiting, and wait
                     // for the previous kernel only before exiting (so that this
                     // launch completes after it, and a kernel waiting on this
                     // one also waits on that one)
};

struct DenseOutArgs {
  DenseSeg seg[1];
  int nseg;
  int total_rows;    // hidden
  int K;             // staged vector length: latent + shared
  // staged vector [y (latent columns) | shared activation]
  int latent;        // L: columns [0, L) come from `staged` (0: none)
  int shared;        // shared_ffn columns computed from dense_in (0: none)
  const float* staged;  // [T, staged_ld] combined routed output y (latent layers)
  int staged_ld;
  const float* dense_in;  // [T, r_in]
  int r_in;          // dense_in row stride
  int sh_g_off, sh_u_off; // column offsets of shared gate/up logits in dense_in
  int act;
  // epilogue: s = dot + y_add + add_f32, then out = x + s (or out_f32 = s)
  const float* y_add;  // [T, total_rows] combined routed output (non-latent layers) or null
  const float* pexp;   // or, when y_add is null: unweighted per-pick outputs [T*k, total_rows]
  const float* wts;    // and their weights [T*k], combined here in pick order (or null)
  int k;
  const float* add_f32;  // [T, total_rows] e.g. the shared expert's output or null
  float* out_f32;    // [T, total_rows]: write s here and nothing else (null: residual output)
  const void* x;     // [T, H] residual, act dtype
  int x_dt;
  void* out;         // [T, H] act dtype
  float* delta;      // [T, H] fp32 or null
  int T;
  int prefetch;      // prefetch this CTA's weight rows into L2 before waiting
  unsigned long long* trace;   // diagnostics: CTA stamps or null
  int dep_tail;      // as DenseInArgs::dep_tail (its inputs are complete when it launches)
};

// Rows of the dense weights per register batch: every thread keeps partial sums
// for RB rows x TB token rows.
template <int TB>
__host__ __device__ constexpr int dense_rb() { return TB <= 2 ? 4 : 2; }

// One step of the dense streaming loop: rows [r, r + nb) of segment si, part
// p, 16-byte chunks [cbase, cbase + MAXC * NT).
struct DStep {
  int r, nb, si, p, cbase;
  bool valid;
};

__device__ __forceinline__ int dpart_chunks(const DensePart& P) {
  return P.wk / (P.dt == DT_FP32 ? 4 : 8);
}

template <int RBN>
__device__ __forceinline__ void dstep_first(const DenseSeg* segs, int r_begin, int r_end, DStep& st) {
  st.si = 0; st.r = r_begin; st.p = 0; st.cbase = 0; st.nb = 0;
  st.valid = r_begin < r_end;
  if (st.valid) {
    while (st.r >= segs[st.si].row0 + segs[st.si].rows) ++st.si;
    st.nb = min(RBN, min(r_end, segs[st.si].row0 + segs[st.si].rows) - st.r);
  }
}

template <int RBN>
__device__ __forceinline__ void dstep_next(const DenseSeg* segs, int r_end, DStep& st) {
  st.cbase += MAXC * NT;
  if (st.cbase < dpart_chunks(segs[st.si].part[st.p])) return;
  st.cbase = 0;
  if (++st.p < segs[st.si].nparts) return;
  st.p = 0;
  st.r += st.nb;
  if (st.r >= r_end) { st.valid = false; return; }
  while (st.r >= segs[st.si].row0 + segs[st.si].rows) ++st.si;
  st.nb = min(RBN, min(r_end, segs[st.si].row0 + segs[st.si].rows) - st.r);
}

template <int RBN>
__device__ __forceinline__ void dstep_load(const DenseSeg* segs, const DStep& st, uint4 (&wv)[RBN][MAXC]) {
  const DensePart& P = segs[st.si].part[st.p];
  const int esz = P.dt == DT_FP32 ? 4 : 2;
  const int nch = dpart_chunks(P);
  const int64_t rstride = static_cast<int64_t>(P.wk) * esz;
  const char* wbase = static_cast<const char*>(P.w) + static_cast<int64_t>(st.r - segs[st.si].row0) * rstride;
#pragma unroll
  for (int i = 0; i < RBN; ++i)
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
      const int ci = st.cbase + c * NT + static_cast<int>(threadIdx.x);
      if (i < st.nb && ci < nch)
        wv[i][c] = ldg_stream(wbase + i * rstride + static_cast<int64_t>(ci) * 16);
      else
        wv[i][c] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Streams the rows [r_begin, r_end) of the segments against xs (staged
// [TB][K] swizzled fp32) and leaves per-(row, t) warp partials in red.  The
// loads of step s + 1 are issued before step s is computed (two register
// buffers), so every warp keeps its next batch of weights in flight.
// `stage` is called once after the first loads are issued (it stages xs and
// ends with a barrier), so the first memory latency overlaps the staging.
template <int TB, typename StageFn>
__device__ __forceinline__ void dense_rows(const DenseSeg* segs, int r_begin, int r_end,
                                           const float4* xs4, int K4, float* red, StageFn stage) {
  constexpr int RBN = dense_rb<TB>();
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  float acc[RBN][TB];
#pragma unroll
  for (int i = 0; i < RBN; ++i)
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[i][t] = 0.0f;

  // compute one step from its loaded weights; reduce when its rows are done
  auto compute = [&](const DStep& cur, const uint4 (&w)[RBN][MAXC], const DStep& nxt) {
    const DensePart& P = segs[cur.si].part[cur.p];
    const int nch = dpart_chunks(P);
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
      const int ci = cur.cbase + c * NT + tid;
      if (ci >= nch) continue;
      if (P.dt != DT_FP32) {
        const int f4 = (P.k0 >> 2) + 2 * ci;
        const int s0 = swz(f4, 1), s1 = swz(f4 + 1, 1);
#pragma unroll
        for (int i = 0; i < RBN; ++i) {
          if (i >= cur.nb) continue;
          float wf[8];
          cvt8(w[i][c], P.dt, wf);
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            const float4 a = xs4[t * K4 + s0];
            const float4 b = xs4[t * K4 + s1];
            float sacc = acc[i][t];
            sacc = fmaf(wf[0], a.x, sacc); sacc = fmaf(wf[1], a.y, sacc);
            sacc = fmaf(wf[2], a.z, sacc); sacc = fmaf(wf[3], a.w, sacc);
            sacc = fmaf(wf[4], b.x, sacc); sacc = fmaf(wf[5], b.y, sacc);
            sacc = fmaf(wf[6], b.z, sacc); sacc = fmaf(wf[7], b.w, sacc);
            acc[i][t] = sacc;
          }
        }
      } else {
        const int s0 = swz((P.k0 >> 2) + ci, 1);
#pragma unroll
        for (int i = 0; i < RBN; ++i) {
          if (i >= cur.nb) continue;
          const uint4 v = w[i][c];
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            const float4 a = xs4[t * K4 + s0];
            float sacc = acc[i][t];
            sacc = fmaf(__uint_as_float(v.x), a.x, sacc); sacc = fmaf(__uint_as_float(v.y), a.y, sacc);
            sacc = fmaf(__uint_as_float(v.z), a.z, sacc); sacc = fmaf(__uint_as_float(v.w), a.w, sacc);
            acc[i][t] = sacc;
          }
        }
      }
    }
    if (!nxt.valid || nxt.r != cur.r) {
      // the rows of this batch are complete: warp reduce-scatter, one partial
      // per warp to shared memory
      constexpr int NV = RBN * TB;
      float v[NV];
#pragma unroll
      for (int i = 0; i < RBN; ++i)
#pragma unroll
        for (int t = 0; t < TB; ++t) { v[i * TB + t] = acc[i][t]; acc[i][t] = 0.0f; }
      const float tot = warp_reduce_scatter<NV>(v, lane);
      constexpr int LPV = 32 / NV;  // lanes per value
      if ((lane & (LPV - 1)) == 0) {
        const int vi = lane / LPV;
        const int i = vi / TB, t = vi % TB;
        if (i < cur.nb) red[((cur.r - r_begin + i) * TB + t) * NW + warp] = tot;
      }
    }
  };

  // two register buffers in ping-pong (no copies between them: a copy would
  // wait for the loads in flight)
  DStep sa, sb;
  uint4 wa[RBN][MAXC], wb[RBN][MAXC];
  dstep_first<RBN>(segs, r_begin, r_end, sa);
  if (sa.valid) dstep_load<RBN>(segs, sa, wa);
  stage();
  while (sa.valid) {
    sb = sa;
    dstep_next<RBN>(segs, r_end, sb);
    if (sb.valid) dstep_load<RBN>(segs, sb, wb);
    compute(sa, wa, sb);
    if (!sb.valid) break;
    sa = sb;
    dstep_next<RBN>(segs, r_end, sa);
    if (sa.valid) dstep_load<RBN>(segs, sa, wa);
    compute(sb, wb, sa);
  }
}

// Stage rows [t0, t0 + tb) of a [T, K] activation matrix (any dtype) as fp32,
// swizzled for 8-element chunk readers; rows tb..TB-1 are zero.
template <int TB>
__device__ __forceinline__ void stage_x(float* xs, const void* x, int x_dt, int K, int t0, int tb) {
  const int K4 = K >> 2;
  for (int i = threadIdx.x; i < TB * K4; i += NT) {
    const int t = i / K4, f4 = i - t * K4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < tb) {
      const int64_t e = static_cast<int64_t>(t0 + t) * K + 4 * f4;
      v.x = ld_any(x, e, x_dt); v.y = ld_any(x, e + 1, x_dt);
      v.z = ld_any(x, e + 2, x_dt); v.w = ld_any(x, e + 3, x_dt);
    }
    reinterpret_cast<float4*>(xs)[t * K4 + swz(f4, 1)] = v;
  }
}

// Rows per CTA for a dense launch of `rows` rows over `grid` CTAs.
__device__ __forceinline__ void cta_rows(int rows, int& b, int& e) {
  const int64_t c = blockIdx.x, g = gridDim.x;
  b = static_cast<int>(c * rows / g);
  e = static_cast<int>((c + 1) * rows / g);
}

// CTAs per SM the dense kernels are compiled for: more resident warps keep
// more weight loads in flight while other warps reduce.
template <int TB>
constexpr int dense_min_blocks() { return 2; }

// Rows [rb, re) of the dense matrices that read x, for all T token rows
// (staged TB at a time): out[t, r] = W_r . x_t in fp32.
template <int TB>
__device__ __forceinline__ void dense_in_rows(const DenseInArgs& A, int rb, int re, float4* smem4) {
  float* xs = reinterpret_cast<float*>(smem4);
  float* red = xs + TB * A.K;
  const int K4 = A.K >> 2;
  for (int t0 = 0; t0 < A.T; t0 += TB) {
    const int tb = min(TB, A.T - t0);
    if (t0) __syncthreads();
    for (int r0 = rb; r0 < re; r0 += RED_ROWS) {
      const int r1 = min(re, r0 + RED_ROWS);
      const bool first = r0 == rb;
      dense_rows<TB>(A.seg, r0, r1, smem4, K4, red, [&]() {
        if (first) stage_x<TB>(xs, A.x, A.x_dt, A.K, t0, tb);
        __syncthreads();
      });
      __syncthreads();
      for (int o = threadIdx.x; o < (r1 - r0) * TB; o += NT) {
        const int rl = o / TB, t = o % TB;
        if (t >= tb) continue;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += red[o * NW + w];
        A.out[static_cast<int64_t>(t0 + t) * A.out_ld + r0 + rl] = s;
      }
      __syncthreads();
    }
  }
}

template <int TB>
__global__ void __launch_bounds__(NT, dense_min_blocks<TB>()) k_dense_in(const __grid_constant__ DenseInArgs A) {
  extern __shared__ float4 smem4[];
  cta_stamp(A.trace, 0);
  if (A.fuse_route && A.route_warm && blockIdx.x == 0) {
    // The first run of the top-k code is slow (its instructions come from a
    // cold L2): the routing CTA runs its phases once, one per warp at once, on
    // whatever the buffers hold, writing nothing, before it waits for the
    // previous kernel (that run reads no value this launch depends on and
    // stores nothing).
    RouteArgs D = A.route;
    D.dry = 1;
    // the few-pairs list code (a warp's sort of the ids as they stand) runs
    // dry too; the counting path indexes shared memory by id, so not that
    D.topk_only = D.T * D.k > 32;
    route_warm(D, reinterpret_cast<int*>(smem4));
    cta_stamp(A.trace, 4);
  }
  if (!A.dep_tail) griddep_wait();
  griddep_launch();
  cta_stamp(A.trace, 1);
  int rb, re;
  if (A.fuse_route && A.route_warm) {
    // CTA 0 routes and holds no rows; CTAs 1..route_ctas take the router rows
    const int E = A.route.E, rc = A.route_ctas, c = blockIdx.x, g = gridDim.x;
    if (c == 0) {
      rb = re = 0;
    } else if (c <= rc) {
      rb = static_cast<int>(static_cast<int64_t>(c - 1) * E / rc);
      re = static_cast<int>(static_cast<int64_t>(c) * E / rc);
    } else {
      const int64_t rest = A.total_rows - E;
      rb = E + static_cast<int>(static_cast<int64_t>(c - 1 - rc) * rest / (g - 1 - rc));
      re = E + static_cast<int>(static_cast<int64_t>(c - rc) * rest / (g - 1 - rc));
    }
  } else if (A.fuse_route) {
    // the first route_ctas CTAs take the router rows [0, E) (fewer rows each,
    // so the routing starts early and overlaps the rest of the pass)
    const int E = A.route.E, rc = A.route_ctas, c = blockIdx.x, g = gridDim.x;
    if (c < rc) {
      rb = static_cast<int>(static_cast<int64_t>(c) * E / rc);
      re = static_cast<int>(static_cast<int64_t>(c + 1) * E / rc);
    } else {
      const int64_t rest = A.total_rows - E;
      rb = E + static_cast<int>(static_cast<int64_t>(c - rc) * rest / (g - rc));
      re = E + static_cast<int>(static_cast<int64_t>(c - rc + 1) * rest / (g - rc));
    }
  } else {
    cta_rows(A.total_rows, rb, re);
  }
  dense_in_rows<TB>(A, rb, re, smem4);
  cta_stamp(A.trace, 2);
  if (A.fuse_route && A.route_warm) {
    if (blockIdx.x == 0) {
      __shared__ int s_ok;
      __syncthreads();
      if (threadIdx.x == 0) {
        const bool ok = spin_until_geq(A.route_counter, A.route_ctas + (A.debug_stall ? 1 : 0));
        if (!ok) atomicOr(A.route.status, STATUS_TIMEOUT);
        s_ok = ok;
        __threadfence();
      }
      __syncthreads();
      cta_stamp(A.trace, 5);
      // on a timeout the routing still runs (on the logits as they stand), so
      // that the ids and lists stay well formed; the status reports it
      route_block(A.route, reinterpret_cast<int*>(smem4));
      cta_stamp(A.trace, 6);
      __syncthreads();
      if (threadIdx.x == 0) *A.route_counter = 0;
      (void)s_ok;
    } else if (static_cast<int>(blockIdx.x) <= A.route_ctas) {
      // release this CTA's router logits to the routing CTA
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) atomicAdd(A.route_counter, 1);
    }
  } else if (A.fuse_route && static_cast<int>(blockIdx.x) < A.route_ctas) {
    // the last CTA to finish router rows routes all T rows
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(A.route_counter, 1) == A.route_ctas - 1);
    __syncthreads();
    if (s_last) {
      __threadfence();
      route_block(A.route, reinterpret_cast<int*>(smem4));
      if (threadIdx.x == 0) *A.route_counter = 0;
      if (A.prefetch_up) {
        __syncthreads();
        const int nu = A.route.meta[0];
        const int64_t per = (A.pf_q_bytes + A.pf_sb_bytes) * (A.pf_q2 ? 2 : 1);
        const int64_t cap = A.pf_budget / (per > 0 ? per : 1);
        const int nmax = static_cast<int>(nu < cap ? nu : cap);
        for (int u = threadIdx.x; u < nmax; u += blockDim.x) {
          const int64_t e = A.route.meta[1 + u];
          if (!idx_ok(A.route.status, CK_PREFETCH_E, e, A.route.E)) continue;
          prefetch_l2(reinterpret_cast<const char*>(A.pf_q) + e * A.pf_q_bytes, A.pf_q_bytes);
          prefetch_l2(reinterpret_cast<const char*>(A.pf_sb) + e * A.pf_sb_bytes, A.pf_sb_bytes);
          if (A.pf_q2) {
            prefetch_l2(reinterpret_cast<const char*>(A.pf_q2) + e * A.pf_q_bytes, A.pf_q_bytes);
            prefetch_l2(reinterpret_cast<const char*>(A.pf_sb2) + e * A.pf_sb_bytes, A.pf_sb_bytes);
          }
        }
      }
    }
  }
  if (A.dep_tail) griddep_wait();
  cta_stamp(A.trace, 3);
}

// Output rows [rb, re) of the output projection for all T token rows (staged
// TB at a time): s = [fc2 | shared down] . [y | act(shared gate, up)] plus the
// routed and shared terms given, then out = x + s rounded once (or s in fp32).
template <int TB>
__device__ __forceinline__ void dense_out_rows(const DenseOutArgs& A, int rb, int re, float4* smem4) {
  float* red = reinterpret_cast<float*>(smem4) + TB * A.K;
  const int K4 = A.K >> 2;
  const int L = A.latent;
  for (int t0 = 0; t0 < A.T; t0 += TB) {
    const int tb = min(TB, A.T - t0);
    if (t0) __syncthreads();
    // staged vector: [combined routed output y (latent only) | shared activation]
    auto stage_body = [&]() {
      for (int i = threadIdx.x; i < TB * K4; i += NT) {
        const int t = i / K4, f4 = i - t * K4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < tb) {
          const int tt = t0 + t;
          if (4 * f4 < L) {
            v = __ldcg(reinterpret_cast<const float4*>(A.staged + static_cast<int64_t>(tt) * A.staged_ld) + f4);
          } else {
            const float* di = A.dense_in + static_cast<int64_t>(tt) * A.r_in;
            float r[4];
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int f = 4 * f4 + j - L;
              const float u = __ldcg(di + A.sh_u_off + f);
              const float g = (A.act == ACT_SWIGLU) ? __ldcg(di + A.sh_g_off + f) : 0.f;
              r[j] = act_fn(A.act, g, u);
            }
            v = make_float4(r[0], r[1], r[2], r[3]);
          }
        }
        smem4[t * K4 + swz(f4, 1)] = v;
      }
    };
    for (int r0 = rb; r0 < re; r0 += RED_ROWS) {
      const int r1 = min(re, r0 + RED_ROWS);
      const bool first = r0 == rb;
      if (A.nseg) dense_rows<TB>(A.seg, r0, r1, smem4, K4, red, [&]() {
        if (first) stage_body();
        __syncthreads();
      });
      __syncthreads();
      for (int o = threadIdx.x; o < (r1 - r0) * TB; o += NT) {
        const int rl = o / TB, t = o % TB;
        if (t >= tb) continue;
        const int tt = t0 + t, n = r0 + rl;
        float s = 0.f;
        if (A.nseg) {
#pragma unroll
          for (int w = 0; w < NW; ++w) s += red[o * NW + w];
        }
        const int64_t e = static_cast<int64_t>(tt) * A.total_rows + n;
        if (A.y_add) {
          s += __ldcg(A.y_add + e);                  // non-latent: routed output added directly
        } else if (A.pexp) {
          float y = 0.f;
          for (int p = 0; p < A.k; ++p)
            y = fmaf(A.wts[tt * A.k + p], A.pexp[static_cast<int64_t>(tt * A.k + p) * A.total_rows + n], y);
          s += y;
        }
        if (A.add_f32) s += __ldcg(A.add_f32 + e);   // the shared expert's output
        if (A.out_f32) {
          A.out_f32[e] = s;
          continue;
        }
        const float xv = ld16(A.x, e, A.x_dt);
        reinterpret_cast<unsigned short*>(A.out)[e] = st16_bits(xv + s, A.x_dt);
        if (A.delta) A.delta[e] = s;
      }
      __syncthreads();
    }
  }
}

template <int TB>
__global__ void __launch_bounds__(NT, dense_min_blocks<TB>()) k_dense_out(const __grid_constant__ DenseOutArgs A) {
  extern __shared__ float4 smem4[];
  int rb, re;
  cta_stamp(A.trace, 0);
  cta_rows(A.total_rows, rb, re);
  // the weights do not depend on this forward's earlier kernels: start them
  // towards L2 while those finish
  if (A.prefetch && A.nseg && threadIdx.x < A.seg[0].nparts && re > rb) {
    const DensePart& P = A.seg[0].part[threadIdx.x];
    const int esz = P.dt == DT_FP32 ? 4 : 2;
    prefetch_l2(static_cast<const char*>(P.w) + static_cast<int64_t>(rb) * P.wk * esz,
                static_cast<int64_t>(re - rb) * P.wk * esz);
  }
  if (!A.dep_tail) griddep_wait();
  griddep_launch();
  cta_stamp(A.trace, 1);
  dense_out_rows<TB>(A, rb, re, smem4);
  if (A.dep_tail) griddep_wait();
  cta_stamp(A.trace, 3);
}

// ---------------------------------------------------------------------------
// routing: top-k, weights, distinct-expert lists
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// int4 affine expert gemv (k_expert)
// ---------------------------------------------------------------------------

struct ExpertArgs {
  int n_rows;              // output rows per expert
  int K;                   // reduction length
  int G;                   // group size
  const uint32_t* q;       // [E, n_rows, K*bits/32] (bits: k_expert's code width)
  const uint32_t* sb;      // [E, n_rows, K/G]  (scale bits | bias bits << 16)
  const uint32_t* q_gate;  // SWIGLU up only: gate codes, else null
  const uint32_t* sb_gate;
  int s_dt;                // scale dtype
  int act;                 // activation applied to the output (-1: none)
  const int* meta;         // route metadata
  int umax;
  int k;                   // top_k
  // input row of pair p: by token (t = p / k) or by pair
  const void* xin;
  int xin_dt;
  int64_t xin_stride;      // elements between rows
  int64_t xin_off;         // element offset of the first row
  int xin_by_pair;
  float* out;              // [T*k, n_rows]
  int pre_wait_phase;      // 1: the route metadata is final at launch (the kernel
                           // before this one waited for it): let the next kernel
                           // launch, prefetch, then wait for the previous kernel.
                           // 0: wait first (the metadata may still be written).
  int prefetch;            // prefetch this CTA's weight rows into L2 (pre-wait phase)
  int cps;                 // CTAs per distinct-expert slot (grid = umax * cps)
  int max_pairs;           // > 0: slots with more token pairs are left to the grouped GEMM
  // weighted combine fused into the down projection: the last CTA to finish a
  // column range [nb, ne) (k_expert_mma: a 16-row tile) over all distinct
  // experts writes comb[t, n] = sum_j w[t, j] * out[t*k + j, n], picks in
  // order j = 0..k-1
  float* comb;             // [T, n_rows] or null
  const float* cwts;       // [T*k] combine weights
  int* ccnt;               // completion counters, one a range or tile (zero between launches)
  int T;
  int nst;                 // k_expert_bulk: shared-memory stages of the tile ring
  int* status;             // device status words (timeout bit; index checks)
  int gsh;                 // k_expert_bulk: log2(G) - 5 (chunk c lies in group c >> gsh)
  int n_experts;           // bound of expert ids (index checks)
  // k_expert_mma: codes and scale/bias words in its tiled layouts, chunks of
  // 64 columns per ring stage (ck; nst stages per warp), pairs per pass (pp)
  const uint32_t* qt;
  const uint32_t* sbt;
  const uint32_t* qt_gate;
  const uint32_t* sbt_gate;
  int ck, pp, ks;   // ks: warps sharing a tile's K range (1, 2 or 4)
  int one_pass;     // every slot has at most pp pairs (T <= pp): one segment a slot
  // k_expert_mma's weight format: 0 affine, 1 NVFP4 (sbt/sbt_gate hold the E4M3
  // block scales, four a word; gsc/gsc_gate the per-matrix fp32 scales [E]),
  // 2 MXFP4 (sbt/sbt_gate hold the E8M0 block scales, two a 16-bit entry)
  int wfmt;
  const float* gsc;
  const float* gsc_gate;
  unsigned long long* trace;   // diagnostics: CTA stamps or null
};

__device__ __forceinline__ void sb_decode(uint32_t v, int dt, float& s, float& b) {
  if (dt == DT_BF16) { s = bf16lo(v); b = bf16hi(v); }
  else { s = f16lo(v); b = f16hi(v); }
}

// one 32-code chunk (uint4) against one staged row; returns sum (1 + q/16) x
__device__ __forceinline__ float chunk_dot(const uint4 w, const float4* x8, int c) {
  const int sw = c & 7;
  float s = 0.f;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 a = x8[(2 * i) ^ sw];
    const float4 b = x8[(2 * i + 1) ^ sw];
    const uint32_t v = ws[i];
    s = fmaf(nib<0>(v), a.x, s); s = fmaf(nib<1>(v), a.y, s);
    s = fmaf(nib<2>(v), a.z, s); s = fmaf(nib<3>(v), a.w, s);
    s = fmaf(nib<4>(v), b.x, s); s = fmaf(nib<5>(v), b.y, s);
    s = fmaf(nib<6>(v), b.z, s); s = fmaf(nib<7>(v), b.w, s);
  }
  return s;
}

// 32 consecutive codes of a row: BITS words of its little-endian bit stream
// (code i in bits [i*BITS, i*BITS + BITS)); one 16-byte vector for 4-bit codes
template <int BITS>
struct CodeChunk { uint32_t w[BITS]; };
template <>
struct CodeChunk<4> { uint4 v; };

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// chunk c of a row starts at word c * BITS (16-byte aligned for 4 and 8 bits)
template <int BITS>
__device__ __forceinline__ CodeChunk<BITS> ld_chunk(const uint32_t* p) {
  CodeChunk<BITS> r;
  if constexpr (BITS == 4) {
    r.v = ldg_stream(p);
  } else if constexpr (BITS % 4 == 0) {
#pragma unroll
    for (int i = 0; i < BITS; i += 4) {
      const uint4 v = ldg_stream(p + i);
      r.w[i] = v.x; r.w[i + 1] = v.y; r.w[i + 2] = v.z; r.w[i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) r.w[i] = ldg_stream_u32(p + i);
  }
  return r;
}

// code I of a chunk -> float 1 + q / 2^BITS (the code placed under the
// mantissa of 1.0); a code that straddles two words is joined by a funnel shift
template <int BITS, int I>
__device__ __forceinline__ float code_f(const CodeChunk<BITS>& ch) {
  constexpr int p = I * BITS, wi = p >> 5, off = p & 31;
  uint32_t v;
  if constexpr (off + BITS <= 32) v = ch.w[wi] >> off;
  else v = __funnelshift_r(ch.w[wi], ch.w[wi + 1], off);
  return __uint_as_float(((v & ((1u << BITS) - 1u)) << (23 - BITS)) | 0x3f800000u);
}

template <int BITS, int I>
__device__ __forceinline__ float chunk_dot_part(const CodeChunk<BITS>& w, const float4* x8, int sw, float s) {
  const float4 a = x8[(2 * I) ^ sw];
  const float4 b = x8[(2 * I + 1) ^ sw];
  s = fmaf(code_f<BITS, 8 * I + 0>(w), a.x, s); s = fmaf(code_f<BITS, 8 * I + 1>(w), a.y, s);
  s = fmaf(code_f<BITS, 8 * I + 2>(w), a.z, s); s = fmaf(code_f<BITS, 8 * I + 3>(w), a.w, s);
  s = fmaf(code_f<BITS, 8 * I + 4>(w), b.x, s); s = fmaf(code_f<BITS, 8 * I + 5>(w), b.y, s);
  s = fmaf(code_f<BITS, 8 * I + 6>(w), b.z, s); s = fmaf(code_f<BITS, 8 * I + 7>(w), b.w, s);
  return s;
}

// chunk_dot for any code width: the same order of products (code 0 first)
template <int BITS>
__device__ __forceinline__ float chunk_dot_b(const CodeChunk<BITS>& w, const float4* x8, int c) {
  if constexpr (BITS == 4) {
    return chunk_dot(w.v, x8, c);
  } else {
    const int sw = c & 7;
    float s = chunk_dot_part<BITS, 0>(w, x8, sw, 0.f);
    s = chunk_dot_part<BITS, 1>(w, x8, sw, s);
    s = chunk_dot_part<BITS, 2>(w, x8, sw, s);
    return chunk_dot_part<BITS, 3>(w, x8, sw, s);
  }
}

// The weighted combine fused into the down projection's launch: every CTA of the
// column range [nb, ne) (counter `part`) counts itself done, and the last one
// writes comb[t, n] = sum_j w[t, j] * out[t*k + j, n], picks in order
// j = 0 .. k-1 (one fp32 fma chain).  All of an output's loads are issued before
// its chain, so they overlap instead of following one another.
// comb[tk, n] = sum_j w[tk, j] * out[tk*k + j, n], picks in order j = 0 .. k-1
// (one fp32 fma chain), every load issued before the chain
__device__ __forceinline__ void expert_combine_one(const ExpertArgs& A, int tk, int n) {
  const int k = A.k;
  const float* wr = A.cwts + tk * k;
  const float* xr = A.out + static_cast<int64_t>(tk * k) * A.n_rows + n;
  float wv[MAX_K], xv[MAX_K];
#pragma unroll
  for (int p = 0; p < MAX_K; ++p) {
    wv[p] = p < k ? __ldcg(wr + p) : 0.f;
    xv[p] = p < k ? __ldcg(xr + static_cast<int64_t>(p) * A.n_rows) : 0.f;
  }
  float yv = 0.f;
#pragma unroll
  for (int p = 0; p < MAX_K; ++p)
    if (p < k) yv = fmaf(wv[p], xv[p], yv);
  A.comb[static_cast<int64_t>(tk) * A.n_rows + n] = yv;
}

__device__ __forceinline__ void expert_fused_combine(const ExpertArgs& A, int part, int nb, int ne) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(A.ccnt + part, 1) == A.meta[0] - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int cols = ne - nb;
#pragma unroll 2
  for (int i = threadIdx.x; i < A.T * cols; i += blockDim.x) {
    const int tk = i / cols;
    expert_combine_one(A, tk, nb + (i - tk * cols));
  }
  if (threadIdx.x == 0) A.ccnt[part] = 0;
}

template <int PB, bool GATED>
constexpr int expert_min_blocks() { return PB <= 2 ? (GATED ? 2 : 3) : 2; }

// Expert rows as gemvs over the selected experts' b-bit codes:
//   sum_i (S q_i + B) x_i = 2^b S * sum_i (1 + q_i / 2^b) x_i + (B - 2^b S) * sum_i x_i
// per group (the code sum is exact in fp32: 1 + q / 2^b has b + 1 significant bits).
template <int PB, bool GATED, int BITS = 4>
__global__ void __launch_bounds__(NT, expert_min_blocks<PB, GATED>()) k_expert(const __grid_constant__ ExpertArgs A) {
  extern __shared__ float4 smem4[];
  const int K = A.K, K4 = K >> 2, nchunk = K >> 5;
  const int64_t rw = static_cast<int64_t>(nchunk) * BITS;   // code words a row
  float* xsum = reinterpret_cast<float*>(smem4 + PB * K4);   // [PB][nchunk]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ngr = K / A.G;
  constexpr bool gated = GATED;
  constexpr float QS = static_cast<float>(1 << BITS);
  // rows of a weight matrix in flight per warp (rows warp, warp + NW, ...);
  // halved for 8-bit codes (twice the registers a chunk)
  constexpr int RR0 = (PB <= 2) ? (GATED ? 2 : 4) : (PB <= 4 ? 2 : 1);
  constexpr int RR = (BITS > 4 && RR0 > 1) ? RR0 / 2 : RR0;
  constexpr int NV = RR * PB * 2;   // up and gate partial sums (gate 0 when not gated)
  // Static partition, independent of how many experts were selected: CTA
  // blockIdx.x serves slot u (the u-th distinct selected expert) and rows
  // [nb, ne) of its matrix; slots beyond the distinct count exit at once.
  const int u = blockIdx.x / A.cps, part = blockIdx.x - u * A.cps;
  const int nb = static_cast<int>(static_cast<int64_t>(part) * A.n_rows / A.cps);
  const int ne = static_cast<int>(static_cast<int64_t>(part + 1) * A.n_rows / A.cps);
  const int* uniq_e = A.meta + 1;
  const int* uniq_p0 = A.meta + 1 + A.umax;
  const int* pairs = A.meta + 2 + 2 * A.umax;
  cta_stamp(A.trace, 0);
  if (!A.pre_wait_phase) griddep_wait();
  griddep_launch();
  if (!A.pre_wait_phase) cta_stamp(A.trace, 1);
  if (u >= A.meta[0]) { cta_stamp(A.trace, 3); return; }
  if (A.max_pairs > 0 && uniq_p0[u + 1] - uniq_p0[u] > A.max_pairs) { cta_stamp(A.trace, 3); return; }
  const bool e_ok = idx_ok(A.status, CK_EXPERT_E, uniq_e[u], A.n_experts) &&
                    range_ok(A.status, uniq_p0[u], uniq_p0[u + 1], static_cast<long long>(A.T) * A.k);
  const int64_t e = e_ok ? uniq_e[u] : 0;   // a bad slot reads expert 0 and writes nothing
  if (A.pre_wait_phase && A.prefetch && threadIdx.x == 0) {
    // the route metadata was final before the previous kernel began
    prefetch_l2(A.q + (e * A.n_rows + nb) * rw, static_cast<int64_t>(ne - nb) * rw * 4);
    prefetch_l2(A.sb + (e * A.n_rows + nb) * ngr, static_cast<int64_t>(ne - nb) * ngr * 4);
  }
  if (A.pre_wait_phase) { griddep_wait(); cta_stamp(A.trace, 1); }
  const int pa = uniq_p0[u], pe = e_ok ? uniq_p0[u + 1] : pa;

  // first row batch: issue its weight loads before staging the inputs, so
  // their memory latency overlaps the staging
  CodeChunk<BITS> w0[RR], wg0[RR];
  uint32_t sb0[RR], sbg0[RR];
  {
    const int c = lane;
#pragma unroll
    for (int j = 0; j < RR; ++j) {
      const int n = nb + warp + NW * j;
      if (n < ne && c < nchunk) {
        const int64_t row = e * A.n_rows + n;
        w0[j] = ld_chunk<BITS>(A.q + row * rw + BITS * c);
        sb0[j] = ldg_u32(A.sb + row * ngr + (c << 5) / A.G);
        if (gated) {
          wg0[j] = ld_chunk<BITS>(A.q_gate + row * rw + BITS * c);
          sbg0[j] = ldg_u32(A.sb_gate + row * ngr + (c << 5) / A.G);
        }
      }
    }
  }
  for (int pc = pa; pc < pe; pc += PB) {
    const int np = min(PB, pe - pc);
    if (pc != pa) __syncthreads();
    // stage the input rows of pairs [pc, pc + np), swizzled for 32-element chunks
    for (int i = threadIdx.x; i < PB * K4; i += NT) {
      const int pp = i / K4, f4 = i - pp * K4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (pp < np) {
        int pid = pairs[pc + pp];
        if (!idx_ok(A.status, CK_EXPERT_PAIR, pid, static_cast<long long>(A.T) * A.k)) pid = 0;
        const int64_t row = A.xin_by_pair ? pid : (pid / A.k);
        const int64_t base = A.xin_off + row * A.xin_stride + 4 * f4;
        if (A.xin_dt == DT_FP32) {
          const float* src = static_cast<const float*>(A.xin) + base;
          if (((A.xin_off | A.xin_stride) & 3) == 0) {
            v = *reinterpret_cast<const float4*>(src);
          } else {   // latent columns of dense_in after a router width that is not a multiple of 4
            v.x = src[0]; v.y = src[1]; v.z = src[2]; v.w = src[3];
          }
        } else {
          v.x = ld16(A.xin, base, A.xin_dt); v.y = ld16(A.xin, base + 1, A.xin_dt);
          v.z = ld16(A.xin, base + 2, A.xin_dt); v.w = ld16(A.xin, base + 3, A.xin_dt);
        }
      }
      smem4[pp * K4 + swz(f4, 7)] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < PB * nchunk; i += NT) {
      const int pp = i / nchunk, c = i - pp * nchunk;
      const float4* x8 = smem4 + pp * K4 + 8 * c;
      float sx = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) { const float4 a = x8[j]; sx += (a.x + a.y) + (a.z + a.w); }
      xsum[pp * nchunk + c] = sx;
    }
    __syncthreads();
    for (int rbase = nb + warp; rbase < ne; rbase += NW * RR) {
      const bool first = (pc == pa) && (rbase == nb + warp);
      int nn[RR];
      int64_t rowq[RR], rows[RR];
      bool live[RR];
#pragma unroll
      for (int j = 0; j < RR; ++j) {
        const int n = rbase + NW * j;
        live[j] = n < ne;
        nn[j] = live[j] ? n : rbase;
        rowq[j] = (e * A.n_rows + nn[j]) * rw;
        rows[j] = (e * A.n_rows + nn[j]) * ngr;
      }
      float acc[RR][PB], accg[RR][PB];
#pragma unroll
      for (int j = 0; j < RR; ++j)
#pragma unroll
        for (int pp = 0; pp < PB; ++pp) { acc[j][pp] = 0.f; accg[j][pp] = 0.f; }
      for (int c = lane; c < nchunk; c += 32) {
        const int g = (c << 5) / A.G;
        CodeChunk<BITS> w[RR], wg[RR];
        uint32_t sbv[RR], sbg[RR];
        if (first && c == lane) {
#pragma unroll
          for (int j = 0; j < RR; ++j) { w[j] = w0[j]; sbv[j] = sb0[j]; wg[j] = wg0[j]; sbg[j] = sbg0[j]; }
        } else {
#pragma unroll
          for (int j = 0; j < RR; ++j) {
            if (live[j]) {
              w[j] = ld_chunk<BITS>(A.q + rowq[j] + BITS * c);
              sbv[j] = ldg_u32(A.sb + rows[j] + g);
              if (gated) {
                wg[j] = ld_chunk<BITS>(A.q_gate + rowq[j] + BITS * c);
                sbg[j] = ldg_u32(A.sb_gate + rows[j] + g);
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < RR; ++j) {
          if (!live[j]) continue;
          float sc, bi;
          sb_decode(sbv[j], A.s_dt, sc, bi);
          const float s16 = QS * sc, bb = bi - s16;
          float sg16 = 0.f, bbg = 0.f;
          if (gated) {
            float sg, bg;
            sb_decode(sbg[j], A.s_dt, sg, bg);
            sg16 = QS * sg; bbg = bg - sg16;
          }
#pragma unroll
          for (int pp = 0; pp < PB; ++pp) {
            if (pp < np) {
              const float4* x8 = smem4 + pp * K4 + 8 * c;
              const float xs = xsum[pp * nchunk + c];
              acc[j][pp] = fmaf(s16, chunk_dot_b<BITS>(w[j], x8, c), fmaf(bb, xs, acc[j][pp]));
              if (gated)
                accg[j][pp] = fmaf(sg16, chunk_dot_b<BITS>(wg[j], x8, c), fmaf(bbg, xs, accg[j][pp]));
            }
          }
        }
      }
      // warp reduce-scatter of all partial sums: value (j, pp, up|gate)
      float v[NV];
#pragma unroll
      for (int j = 0; j < RR; ++j)
#pragma unroll
        for (int pp = 0; pp < PB; ++pp) {
          v[(j * PB + pp) * 2] = acc[j][pp];
          v[(j * PB + pp) * 2 + 1] = accg[j][pp];
        }
      const float tot = warp_reduce_scatter<NV>(v, lane);
      constexpr int LPV = 32 / NV;
      const int vi = lane / LPV;
      const float other = __shfl_down_sync(0xffffffffu, tot, LPV);   // gate partner
      if ((lane & (2 * LPV - 1)) == 0) {
        const int j = (vi >> 1) / PB, pp = (vi >> 1) % PB;
        if (live[j] && pp < np) {
          const int pid = pairs[pc + pp];
          const float val = (A.act >= 0) ? act_fn(A.act, other, tot) : tot;
          if (idx_ok(A.status, CK_EXPERT_PAIR, pid, static_cast<long long>(A.T) * A.k))
            A.out[static_cast<int64_t>(pid) * A.n_rows + nn[j]] = val;
        }
      }
    }
  }
  cta_stamp(A.trace, 2);
  if (A.comb) expert_fused_combine(A, part, nb, ne);
  cta_stamp(A.trace, 3);
}

// ---------------------------------------------------------------------------
// create-time re-layout: interleave a group's scale and bias into one word
// ---------------------------------------------------------------------------
static __global__ void k_interleave_sb(const unsigned short* __restrict__ s,
                                const unsigned short* __restrict__ b, uint32_t* __restrict__ out,
                                int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = static_cast<uint32_t>(s[i]) | (static_cast<uint32_t>(b[i]) << 16);
}

// The up projection's B operand in the lists' sorted pair order: row p of
// `out` is the 16-bit input row of the pair at sorted position p (token pid / k),
// so that an expert's rows form one block for tensor copies.
struct GatherArgs {
  const int* meta;      // route metadata: pairs at meta[2 + 2 * umax + p]
  int umax, k, P, K;    // pairs, row length (multiple of 8)
  int* status;          // index checks (MOE_CHECKS builds)
  const unsigned short* in;
  int64_t in_stride;    // elements between input rows
  unsigned short* out;  // [P, K]
};

static __global__ void k_gather_pairs(const __grid_constant__ GatherArgs A) {
  griddep_wait();
  griddep_launch();
  const int v = A.K / 8;   // 16-byte pieces a row
  const int64_t n = static_cast<int64_t>(A.P) * v;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(i / v), j = static_cast<int>(i - static_cast<int64_t>(p) * v);
    int pid = A.meta[2 + 2 * A.umax + p];
    if (!idx_ok(A.status, CK_GATHER_PAIR, pid, A.P)) pid = 0;
    const int row = pid / A.k;
    reinterpret_cast<uint4*>(A.out)[i] =
        reinterpret_cast<const uint4*>(A.in + static_cast<int64_t>(row) * A.in_stride)[j];
  }
}

// Group-major copy of packed scale/bias words: out[e][g][r] = in[e][r][g], so
// that the words of one group for consecutive rows are contiguous (one tensor
// copy per chunk in the grouped GEMM).
static __global__ void k_sb_group_major(const uint32_t* __restrict__ in, uint32_t* __restrict__ out,
                                        int E, int rows, int ngr) {
  const int64_t n = static_cast<int64_t>(E) * rows * ngr;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i / (static_cast<int64_t>(rows) * ngr);
    const int64_t rem = i - e * rows * ngr;
    const int64_t g = rem / rows, r = rem - g * rows;
    out[i] = in[(e * rows + r) * ngr + g];
  }
}

}  // namespace moe
