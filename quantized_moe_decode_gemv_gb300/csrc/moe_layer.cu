// Host side of the quantized MoE decode layer: validation, create/destroy,
// forward orchestration and the C ABI declared in include/moe_layer.h.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>   // PFN_cuTensorMapEncodeTiled
#include <nvtx3/nvToolsExt.h>   // header-only NVTX v3

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "moe_layer.h"
#include "moe_kernels.cuh"
#include "moe_expert_bulk.cuh"
#include "moe_expert_mma.cuh"
#include "moe_dense_mma.cuh"
#include "moe_dense_bulk.cuh"
#include "moe_umma.cuh"
#include "moe_umma2.cuh"

using namespace moe;

namespace {

constexpr int kSmemMax = 227 * 1024;
constexpr int kCombineCounters = 4096;   // column ranges of the down projection's fused combine

std::atomic<int64_t> g_live_allocs{0};
std::atomic<int32_t> g_fail_countdown{0};
thread_local std::string g_create_error;

bool alloc_should_fail() {
  int32_t c = g_fail_countdown.load();
  while (c > 0) {
    if (g_fail_countdown.compare_exchange_weak(c, c - 1)) return c == 1;
  }
  return false;
}

int dt_size(int dt) { return dt == DT_FP32 ? 4 : 2; }

}  // namespace

struct moe_layer {
  moe_layer_config cfg{};
  int device = -1;
  int num_sms = 0;
  int path = MOE_PATH_AUTO;
  std::vector<void*> allocs;
  int64_t bytes = 0;
  std::string last_error;

  // library-owned weights
  void* router_w = nullptr;
  float* router_bias = nullptr;
  void* fc1 = nullptr;
  void* fc2 = nullptr;
  uint32_t *gate_q = nullptr, *up_q = nullptr, *down_q = nullptr;
  uint32_t *gate_sb = nullptr, *up_sb = nullptr, *down_sb = nullptr;
  // group-major copies of the scale/bias words ([E, K/G, rows]: the grouped GEMM's tensor copies)
  uint32_t *gate_sbT = nullptr, *up_sbT = nullptr, *down_sbT = nullptr;
  // the warp-MMA expert kernel's tiled copies (4-bit codes only)
  uint32_t *gate_qt = nullptr, *up_qt = nullptr, *down_qt = nullptr;
  uint32_t *gate_sbt = nullptr, *up_sbt = nullptr, *down_sbt = nullptr;
  // the warp-MMA dense kernel's tiled copies of the bf16 matrices
  void *router_t = nullptr, *fc1_t = nullptr, *fc2_t = nullptr;
  void *shg_t = nullptr, *shu_t = nullptr, *shd_t = nullptr;
  void *sh_gate = nullptr, *sh_up = nullptr, *sh_down = nullptr;

  // workspace
  float* dense_in = nullptr;  // [Tmax, r_in]
  int* ids = nullptr;         // [Tmax*k]
  float* wts = nullptr;       // [Tmax*k]
  int* meta = nullptr;
  float* hbuf = nullptr;      // [Tmax*k, F]
  float* pexp = nullptr;      // [Tmax*k, Kin]
  int* status = nullptr;
  int* route_counter = nullptr;
  float* comb = nullptr;      // [Tmax, L + F_sh] staged operand of the output projection
  void* xl16 = nullptr;       // [Tmax, L] 16-bit latent rows (grouped path B operand)
  void* h16 = nullptr;        // [Tmax*k, F] 16-bit expert activations (grouped path)
  void* xs = nullptr;         // [Tmax*k, K_in] 16-bit up-projection inputs in sorted pair order
  float* part = nullptr;      // split-K partial sums of the grouped dense GEMMs
  void* bout = nullptr;       // [Tmax, L + F_sh] 16-bit operand of the grouped output GEMM
  uint32_t* rmask = nullptr;  // [E, (Tmax+31)/32] routing row bitmasks (Tmax > route_small_t)
  int* rpref = nullptr;       // [E, (Tmax+31)/32] their popcount prefixes
  float* sdbuf = nullptr;     // [Tmax, H] shared-expert down output (fp32)
  void* x_stage = nullptr;    // [Tmax, H] act dtype (host-buffer forward)
  void* out_stage = nullptr;

  // per-stage timing
  bool profiling = false;
  // NVTX ranges around the forward and its stages (on by default in MOE_CHECKS
  // builds; MOE_NVTX=0/1 overrides)
  bool nvtx = MOE_CHECKS != 0;
  bool profiled = false;
  cudaEvent_t ev[MOE_NUM_STAGES + 1] = {};

  int r_in = 0, off_fc1 = 0, off_shg = 0, off_shu = 0;
  int umax = 0;
  int kin = 0;
  int bits = 4;           // code width of the routed experts (2, 3, 4, 5, 6 or 8)
  int fmt = 0;            // MOE_WFMT_AFFINE or MOE_WFMT_NVFP4
  float* up_gs = nullptr;     // NVFP4: per-matrix scales of the experts [E]
  float* gate_gs = nullptr;
  float* down_gs = nullptr;
  int grouped_min_t = 32;
  int expert_split = 0;   // AUTO's grouped path: light experts on the int4 gemv kernel
  int last_launches = 0;  // kernel launches of the last forward
  unsigned long long* um_trace = nullptr;   // diagnostics (MOE_UMMA_TRACE): grouped GEMM role stamps
  int um_trace_n = 0;                       // grouped launches stamped in this forward
  unsigned long long* ct_trace = nullptr;   // diagnostics (MOE_CTA_TRACE): gemv-path CTA stamps
  int ct_n = 0;                             // launches stamped in this forward
  const char* ct_names[CT_SLOTS] = {};
  int pdl_grouped = 1;    // programmatic dependent launch between the grouped-path kernels too
  int use_pdl = 1;        // programmatic dependent launch between the gemv-path kernels
  int expert_pb = 2;      // max token slots per pass of the gemv-path expert kernels
  int expert_target = 4;  // gemv-path expert kernels: CTAs per SM the grid is sized for
  int umma_ctas = 2;      // grouped path: resident CTAs per SM (2 when the TMEM columns allow)
  int umma_v = 0;         // grouped path GEMM: 1 = k_umma (CTA-synchronised K loop), 2 = k_umma2
                          // (warp-specialised roles, tensor copies), 0 = umma_is_v2's choice
  int gather_min_t = 1;     // grouped path: from this many rows the up GEMM's B rows are gathered
                             // into sorted pair order first (then read by tensor copies)
  int route_rpc = 2;         // rows per routing CTA up to route_rpc_max_t rows (else 16)
  int route_rpc_max_t = 256;
  int route_small_t = 8;   // up to this many rows one routing CTA does top-k and lists (at most
                            // ROUTE_SMALL_T); above, row blocks in parallel, then the list CTA
  int umma_sub = 2;            // grouped path (k_umma2, int4, all tensor copies): chunks per ring slot
  int umma_sleep_ns = 64;     // grouped path (k_umma2): sleep between mbarrier polls (waiting
                              // warps leave the issue slots to the working ones)
  int umma_abufs = 3;         // grouped path (k_umma2, int4): dequantised A tiles in the ring
  int umma_tma = 1;           // grouped path (k_umma2): A operand by tensor copies when the layout allows
  int umma_ntile_int4 = 128;  // grouped path: max tokens per MMA tile with int4 (dequantised) A
  int fuse_route = 1;     // routing in the last router CTA of the dense pass (0: own kernel)
  int route_warm = 1;     // fused routing: a dedicated CTA warms the top-k code, then waits
  int route_max_w = 8;    // routing block: most warps sharing a row's keys
  int debug_route = 0;    // diagnostics: print routing phase times
  int expert_bulk = 1;    // gemv path: expert kernels with bulk-copied weight tiles (k_expert_bulk)
  int expert_bulk_max_t = 2;   // the bulk expert kernel up to this many rows
  bool expert_mma = true;      // gemv path: warp-MMA expert kernel (4-bit codes)
  int expert_mma_max_t = 1 << 30;   // ... up to this many rows
  int expert_mma_pp = 8;       // its token pairs per pass (more pairs: more passes)
  bool dense_mma = true;       // gemv path: warp-MMA dense passes (bf16 layers)
  int expert_bulk_pb = 2;      // its token pairs per pass
  int dense_bulk = 1;     // gemv path: shared expert and output projection by k_dense_bulk
  int fill = 0;           // gemv path: the shared expert as launches of its own beside the routed chain
  int fill_ctas = 0;      // those CTAs per launch (0: one per SM)
  int side_stream = 0;    // gemv path: the shared expert on its own stream beside the routed chain
  int side_grid = 0;      // CTAs of the shared expert's launches (0: one per SM)
  cudaStream_t hi_s = nullptr;   // the routed chain (highest priority)
  cudaStream_t lo_s = nullptr;   // the shared expert (lowest priority)
  cudaEvent_t ev_fork = nullptr, ev_side = nullptr, ev_chain = nullptr;
  int* ccnt = nullptr;    // completion counters of the down projection's fused combine
  int prefetch = 6;       // bit 0: experts' up weights from the routing CTA (one SM's
                          // bulk engine: slow, off by default); bit 1: down weights;
                          // bit 2: output-projection weights

  cudaError_t alloc(void** p, size_t n) {
    *p = nullptr;
    if (alloc_should_fail()) return cudaErrorMemoryAllocation;
    // 256 bytes of padding: 16-byte-rounded bulk prefetches and vector loads
    // never leave the allocation
    cudaError_t e = cudaMalloc(p, n + 256);
    if (e == cudaSuccess) {
      allocs.push_back(*p);
      bytes += static_cast<int64_t>(n);
      g_live_allocs.fetch_add(1);
    }
    return e;
  }
  void free_events() {
    for (auto& e : ev) {
      if (e) cudaEventDestroy(e);
      e = nullptr;
    }
  }
  void free_streams() {
    for (cudaEvent_t* e : {&ev_fork, &ev_side, &ev_chain}) {
      if (*e) cudaEventDestroy(*e);
      *e = nullptr;
    }
    for (cudaStream_t* st : {&hi_s, &lo_s}) {
      if (*st) cudaStreamDestroy(*st);
      *st = nullptr;
    }
  }
  void free_all() {
    free_events();
    free_streams();
    for (void* p : allocs) {
      cudaFree(p);
      g_live_allocs.fetch_sub(1);
    }
    allocs.clear();
    bytes = 0;
  }
};

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------

static moe_status validate_impl(const moe_layer_config* c, const moe_layer_weights* w,
                                std::string* why) {
  auto fail = [&](moe_status s, const char* msg) {
    if (why) *why = msg;
    return s;
  };
  if (!c) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
  if (c->hidden <= 0 || c->n_experts <= 0 || c->expert_ffn <= 0 || c->max_tokens <= 0 ||
      c->latent < 0 || c->shared_ffn < 0)
    return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (latent/shared_ffn >= 0)");
  if (c->act != MOE_ACT_SWIGLU && c->act != MOE_ACT_RELU2)
    return fail(MOE_ERR_INVALID_ARG, "unknown activation");
  if (c->router != MOE_ROUTER_SOFTMAX && c->router != MOE_ROUTER_SIGMOID)
    return fail(MOE_ERR_INVALID_ARG, "unknown router");
  if (c->act_dtype < 0 || c->act_dtype > 2 || c->scale_dtype < 0 || c->scale_dtype > 2 ||
      c->router_dtype < 0 || c->router_dtype > 2)
    return fail(MOE_ERR_INVALID_ARG, "unknown dtype");
  if (c->top_k < 1 || c->top_k > c->n_experts)
    return fail(MOE_ERR_TOPK_GT_E, "top_k must be in 1..n_experts");
  if (c->latent > 0) {
    if (c->act_dtype == MOE_DTYPE_FP32)
      return fail(MOE_ERR_LATENT_PROJ, "latent projections must be bf16 or fp16");
    if (w && (!w->fc1_latent || !w->fc2_latent))
      return fail(MOE_ERR_LATENT_PROJ, "latent layer without fc1_latent_proj/fc2_latent_proj");
  } else if (w && (w->fc1_latent || w->fc2_latent)) {
    return fail(MOE_ERR_LATENT_PROJ, "latent projections given for a non-latent layer");
  }
  if (c->bits != 0 && (c->bits < 2 || c->bits > 8 || c->bits == 7))
    return fail(MOE_ERR_INVALID_ARG, "bits must be 0 (= 4), 2, 3, 4, 5, 6 or 8");
  if (c->weight_format != MOE_WFMT_AFFINE && c->weight_format != MOE_WFMT_NVFP4 &&
      c->weight_format != MOE_WFMT_MXFP4)
    return fail(MOE_ERR_INVALID_ARG, "unknown weight_format");
  const int G = c->group_size;
  const bool fp4_fmt = c->weight_format != MOE_WFMT_AFFINE;
  if (fp4_fmt && c->bits != 0 && c->bits != 4) return fail(MOE_ERR_INVALID_ARG, "fp4 codes are 4 bits");
  if (c->weight_format == MOE_WFMT_NVFP4) {
    if (G != 16) return fail(MOE_ERR_SHAPE, "NVFP4 blocks are 16 elements: group_size must be 16");
  } else if (c->weight_format == MOE_WFMT_MXFP4) {
    if (G != 32) return fail(MOE_ERR_SHAPE, "MXFP4 blocks are 32 elements: group_size must be 32");
  } else if (G != 32 && G != 64 && G != 128) {
    return fail(MOE_ERR_SHAPE, "group_size must be 32, 64 or 128");
  }
  const int kin = c->latent > 0 ? c->latent : c->hidden;
  if (c->hidden % 64 || c->expert_ffn % 64 || kin % 64 || (c->shared_ffn % 64))
    return fail(MOE_ERR_SHAPE, "hidden, expert_ffn, latent and shared_ffn must be multiples of 64");
  if (kin % G || c->expert_ffn % G)
    return fail(MOE_ERR_SHAPE, "expert input width and expert_ffn must be multiples of group_size");
  if (c->n_experts > MAX_E) return fail(MOE_ERR_UNSUPPORTED, "more than 1024 experts");
  if (c->top_k > MAX_K) return fail(MOE_ERR_UNSUPPORTED, "top_k above 16");
  if (c->act_dtype == MOE_DTYPE_FP32) return fail(MOE_ERR_UNSUPPORTED, "fp32 activations");
  if (c->scale_dtype == MOE_DTYPE_FP32 && c->weight_format == MOE_WFMT_AFFINE)
    return fail(MOE_ERR_UNSUPPORTED, "fp32 scales");
  if (c->has_router_bias && c->router != MOE_ROUTER_SIGMOID)
    return fail(MOE_ERR_UNSUPPORTED, "router bias is defined for sigmoid routing only");
  if (w) {
    if (!w->router_w) return fail(MOE_ERR_INVALID_ARG, "router weight missing");
    if (c->has_router_bias && !w->router_bias) return fail(MOE_ERR_INVALID_ARG, "router bias missing");
    // (MXFP4 has no per-matrix or bias term: its *_b pointers are unused)
    const bool need_b = c->weight_format != MOE_WFMT_MXFP4;
    if (!w->up_q || !w->up_s || (need_b && !w->up_b) || !w->down_q || !w->down_s || (need_b && !w->down_b))
      return fail(MOE_ERR_INVALID_ARG, "expert up/down weights missing");
    if (c->act == MOE_ACT_SWIGLU && (!w->gate_q || !w->gate_s || (need_b && !w->gate_b)))
      return fail(MOE_ERR_INVALID_ARG, "SwiGLU experts need gate weights");
    if (c->act == MOE_ACT_RELU2 && (w->gate_q || w->sh_gate))
      return fail(MOE_ERR_SHAPE, "squared-ReLU experts take no gate matrix");
    if (c->shared_ffn > 0) {
      if (!w->sh_up || !w->sh_down || (c->act == MOE_ACT_SWIGLU && !w->sh_gate))
        return fail(MOE_ERR_UNSUPPORTED, "shared expert weights missing");
    } else if (w->sh_up || w->sh_down || w->sh_gate) {
      return fail(MOE_ERR_SHAPE, "shared expert weights given with shared_ffn = 0");
    }
  }
  return MOE_OK;
}

// dense staging rows per pass that fit shared memory for a staged width K
static int dense_tb_cap(int K) {
  for (int tb = 8; tb >= 1; tb >>= 1)
    if (static_cast<int64_t>(tb) * (4LL * K + 4LL * RED_ROWS * NW) <= kSmemMax - 2048) return tb;
  return 0;
}
static int expert_pb_cap(int K) {
  for (int pb = 8; pb >= 1; pb >>= 1)
    if (static_cast<int64_t>(pb) * (4LL * K + 4LL * (K / 32)) <= kSmemMax - 2048) return pb;
  return 0;
}
static int pow2_at_least(int t, int cap) {
  int v = 1;
  while (v < t && v < cap) v <<= 1;
  return std::min(v, cap);
}

// ---------------------------------------------------------------------------
// launches
// ---------------------------------------------------------------------------

// Launch with the programmatic-stream-serialization attribute when pdl is set.
template <typename Arg>
static cudaError_t launch_ex(void (*kern)(Arg), int grid, int block, size_t smem, cudaStream_t s,
                             bool pdl, const Arg& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int TB>
static size_t dense_smem(int K) {
  return static_cast<size_t>(TB) * (4ull * K + 4ull * RED_ROWS * NW);
}

template <typename Args, int TB>
static cudaError_t launch_dense_in_t(const Args& a, int grid, cudaStream_t s) {
  size_t smem = dense_smem<TB>(a.K);
  if (a.fuse_route)
    smem = std::max<size_t>(smem, ROUTE_SMEM_BYTES + static_cast<size_t>(a.route.E) * a.route.mask_words * 4);
  k_dense_in<TB><<<grid, NT, smem, s>>>(a);
  return cudaGetLastError();
}
template <typename Args, int TB>
static cudaError_t launch_dense_out_t(const Args& a, int grid, cudaStream_t s, bool pdl) {
  return launch_ex<Args>(k_dense_out<TB>, grid, NT, dense_smem<TB>(a.K), s, pdl, a);
}
template <int PB, int BITS = 4>
static cudaError_t launch_expert_t(const ExpertArgs& a, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = static_cast<size_t>(PB) * (4ull * a.K + 4ull * (a.K / 32));
  if (a.q_gate) return launch_ex<ExpertArgs>(k_expert<PB, true, BITS>, grid, NT, smem, s, pdl, a);
  return launch_ex<ExpertArgs>(k_expert<PB, false, BITS>, grid, NT, smem, s, pdl, a);
}

// The gemv path's expert kernel with bulk-copied weight groups: token pairs
// per pass, rows per warp per group, ring stages, CTAs per SM and dynamic
// shared memory of one launch.
struct EbLaunch {
  int pb = 0, r = 0, nst = 0, per_sm = 0;
  size_t smem = 0;
};

// Largest pass of token pairs (up to pb_max); then two CTAs per SM before one;
// then groups of 8 rows per warp over the pass's pairs (R x PB = 8) before
// groups of one row per warp.  The ring holds a CTA's row groups, up to
// EB_MAX_STAGES, and at least two when the CTA has more than one (so that
// copies overlap the arithmetic).  `cps` is the CTAs per distinct expert of the
// chosen plan.  False when no plan fits shared memory (the caller falls back
// to k_expert).
static bool eb_choose(int K, int G, bool gated, int pb_max, int n_rows, int slots, int num_sms, EbLaunch* o,
                      int* cps_out) {
  for (int pb = pb_max; pb >= 1; pb >>= 1) {
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
      const int rs[2] = {8 / pb, 1};
      for (int ri = 0; ri < (rs[0] > 1 ? 2 : 1); ++ri) {
        const int budget = (per_sm == 2 ? kSmemMax / 2 : kSmemMax) - 2048;
        const EbPlan p = eb_plan(K, G, pb, rs[ri], gated);
        const int cps = std::max(1, std::min(std::max(1, n_rows / 8), num_sms * per_sm / std::max(1, slots)));
        const int rows = (n_rows + cps - 1) / cps;
        const int groups = (rows + EB_WARPS * rs[ri] - 1) / (EB_WARPS * rs[ri]);
        const int nst = std::min(std::min(EB_MAX_STAGES, groups), (budget - p.x_bytes) / (p.st_bytes + 8));
        if (nst >= std::min(groups, 2)) {
          o->pb = pb;
          o->r = rs[ri];
          o->nst = nst;
          o->per_sm = per_sm;
          o->smem = static_cast<size_t>(p.x_bytes) + static_cast<size_t>(nst) * (p.st_bytes + 8);
          *cps_out = cps;
          return true;
        }
      }
    }
  }
  return false;
}

// The bulk-copy dense gemv (one or two token rows): token rows per launch, input
// chunks per lane, ring stages, grid and dynamic shared memory.
struct DbLaunch {
  int tb = 0, cpl = 0, nst = 0, grid = 0, stage_bytes = 0;
  size_t smem = 0;
};

// A plan when every segment has the same 16-bit parts and the reduction width
// fits three chunks per lane; token rows in passes of two (one when T = 1);
// two CTAs per SM when their rings fit.
static bool db_choose(const DenseSeg* segs, int nseg, int total_rows, int T, int num_sms, DbLaunch* o) {
  if (nseg < 1 || total_rows < 1) return false;
  const DenseSeg& S0 = segs[0];
  int K = 0;
  for (int p = 0; p < S0.nparts; ++p) {
    if (S0.part[p].dt == DT_FP32 || S0.part[p].wk % 8 || S0.part[p].k0 != K) return false;
    if (reinterpret_cast<uintptr_t>(S0.part[p].w) % 16) return false;
    K += S0.part[p].wk;
  }
  for (int si = 1; si < nseg; ++si) {
    if (segs[si].nparts != S0.nparts) return false;
    for (int p = 0; p < S0.nparts; ++p)
      if (segs[si].part[p].wk != S0.part[p].wk || segs[si].part[p].dt != S0.part[p].dt ||
          reinterpret_cast<uintptr_t>(segs[si].part[p].w) % 16)
        return false;
  }
  const int cpl = (K / 8 + NT - 1) / NT;
  if (cpl > DB_MAX_CPL) return false;
  const int tb = T == 1 ? 1 : 2;
  const int stage_bytes = (DB_SR * K * 2 + 127) & ~127;
  const int fixed = DB_SR * tb * NW * 4 + DB_MAX_STAGES * 8 + 128;
  for (int per_sm = 2; per_sm >= 1; --per_sm) {
    const int budget = (per_sm == 2 ? kSmemMax / 2 : kSmemMax) - 2048;
    const int grid = std::min(num_sms * per_sm, (total_rows + DB_SR - 1) / DB_SR);
    const int rows = (total_rows + grid - 1) / grid;
    const int nstage = (rows + DB_SR - 1) / DB_SR * ((T + tb - 1) / tb);   // over all passes
    const int nst = std::min(std::min(DB_MAX_STAGES, nstage), (budget - fixed) / stage_bytes);
    if (nst >= std::min(2, nstage) && nst >= 1) {
      o->tb = tb;
      o->cpl = cpl;
      o->nst = nst;
      o->grid = grid;
      o->stage_bytes = stage_bytes;
      o->smem = static_cast<size_t>(nst) * stage_bytes + fixed;
      return true;
    }
  }
  return false;
}

template <int TB, int CPL>
static cudaError_t launch_dense_bulk_t(const DbArgs& a, const DbLaunch& d, cudaStream_t s, bool pdl) {
  return launch_ex<DbArgs>(k_dense_bulk<TB, CPL>, d.grid, NT, d.smem, s, pdl, a);
}
static cudaError_t launch_dense_bulk(DbArgs a, const DbLaunch& d, cudaStream_t s, bool pdl) {
  a.nst = d.nst;
  a.stage_bytes = d.stage_bytes;
  if (d.tb == 1) {
    if (d.cpl == 1) return launch_dense_bulk_t<1, 1>(a, d, s, pdl);
    if (d.cpl == 2) return launch_dense_bulk_t<1, 2>(a, d, s, pdl);
    return launch_dense_bulk_t<1, 3>(a, d, s, pdl);
  }
  if (d.cpl == 1) return launch_dense_bulk_t<2, 1>(a, d, s, pdl);
  if (d.cpl == 2) return launch_dense_bulk_t<2, 2>(a, d, s, pdl);
  return launch_dense_bulk_t<2, 3>(a, d, s, pdl);
}

// The bulk dense gemv over a DenseInArgs' rows (input x; fp32 rows out).
static DbArgs db_from_in(const DenseInArgs& a, float* out, int64_t out_ld, int out_col0, int* status) {
  DbArgs d{};
  for (int i = 0; i < a.nseg; ++i) d.seg[i] = a.seg[i];
  d.nseg = a.nseg;
  d.total_rows = a.total_rows;
  d.K = a.K;
  d.T = a.T;
  d.src = DB_SRC_X;
  d.x = a.x;
  d.x_dt = a.x_dt;
  d.epi = DB_EPI_F32;
  d.out = out;
  d.out_ld = out_ld;
  d.out_col0 = out_col0;
  d.status = status;
  d.dep_tail = a.dep_tail;
  return d;
}

// The bulk dense gemv over a DenseOutArgs' rows (input [y | act(shared)]).
static DbArgs db_from_out(const DenseOutArgs& a, int* status) {
  DbArgs d{};
  d.seg[0] = a.seg[0];
  d.nseg = a.nseg;
  d.total_rows = a.total_rows;
  d.K = a.K;
  d.T = a.T;
  d.src = DB_SRC_OUT;
  d.staged = a.staged;
  d.staged_ld = a.staged_ld;
  d.latent = a.latent;
  d.dense_in = a.dense_in;
  d.r_in = a.r_in;
  d.sh_g_off = a.sh_g_off;
  d.sh_u_off = a.sh_u_off;
  d.act = a.act;
  if (a.out_f32) {
    d.epi = DB_EPI_F32;
    d.out = a.out_f32;
    d.out_ld = a.total_rows;
    d.out_col0 = 0;
  } else {
    d.epi = DB_EPI_OUT;
    d.y_add = a.y_add;
    d.add_f32 = a.add_f32;
    d.xres = a.x;
    d.x_dt = a.x_dt;
    d.outb = a.out;
    d.delta = a.delta;
  }
  d.status = status;
  d.dep_tail = a.dep_tail;
  return d;
}

template <int PB, int R>
static cudaError_t launch_expert_bulk_t(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  if (a.q_gate) return launch_ex<ExpertArgs>(k_expert_bulk<PB, R, true>, grid, NT, smem, s, pdl, a);
  return launch_ex<ExpertArgs>(k_expert_bulk<PB, R, false>, grid, NT, smem, s, pdl, a);
}
static cudaError_t launch_expert_bulk(const ExpertArgs& a, const EbLaunch& eb, int grid, cudaStream_t s,
                                      bool pdl) {
  const size_t m = eb.smem;
  if (eb.r == 1) {
    switch (eb.pb) {
      case 1: return launch_expert_bulk_t<1, 1>(a, grid, m, s, pdl);
      case 2: return launch_expert_bulk_t<2, 1>(a, grid, m, s, pdl);
      case 4: return launch_expert_bulk_t<4, 1>(a, grid, m, s, pdl);
      default: return launch_expert_bulk_t<8, 1>(a, grid, m, s, pdl);
    }
  }
  switch (eb.pb) {
    case 1: return launch_expert_bulk_t<1, 8>(a, grid, m, s, pdl);
    case 2: return launch_expert_bulk_t<2, 4>(a, grid, m, s, pdl);
    case 4: return launch_expert_bulk_t<4, 2>(a, grid, m, s, pdl);
    default: return launch_expert_bulk_t<8, 1>(a, grid, m, s, pdl);
  }
}

// The warp-MMA expert kernel's plan: pairs per pass (a multiple of 4, up to
// the T rows' worth, at most EM_MAX_PAIRS), then two CTAs per SM before one,
// then the deepest ring (4 chunks of 64 columns a stage before 2; 4 stages a
// warp before fewer).  `cps` puts one wave of CTAs over the distinct-expert
// slots.  False when no plan fits shared memory.
struct EmLaunch {
  EmPlan plan{};
  int per_sm = 0, cps = 1;
};
static bool em_choose(int K, int G, bool gated, int T, int pp_cap, int n_rows, int slots, int num_sms,
                      EmLaunch* o, int gx = 0) {
  const int pp_want = std::min(std::min(EM_MAX_PAIRS, std::max(4, pp_cap & ~3)), std::max(4, (T + 3) & ~3));
  // warps per tile: a function of K alone, so that a row's sums do not depend
  // on the batch (about 6 to 12 chunks of 64 columns a warp)
  const int nkc = K / 64, nu = nkc / (G > 64 ? G / 64 : 1);   // group-aligned K units
  const int ks = (nkc >= 24 && nu >= 4) ? 4 : ((nkc >= 12 && nu >= 2) ? 2 : 1);
  static const int kCkNs[][2] = {{4, 4}, {4, 3}, {2, 4}, {2, 3}, {2, 2}};
  for (int pp = pp_want; pp >= 4; pp -= 4) {
    // two CTAs per SM only with up to two n-tiles of accumulators (registers)
    for (int per_sm = pp <= 8 ? 2 : 1; per_sm >= 1; --per_sm) {
      const int budget = per_sm == 2 ? 110 * 1024 : kSmemMax - 2048;
      for (const auto& cn : kCkNs) {
        if (G == 128 && cn[0] % 2) continue;
        const EmPlan p = em_plan(K, G, gated, cn[0], cn[1], pp, ks, gx);
        if (p.smem > budget) continue;
        o->plan = p;
        o->per_sm = per_sm;
        o->cps = std::max(1, std::min(n_rows / 16, num_sms * per_sm / std::max(1, slots)));
        return true;
      }
    }
  }
  return false;
}
// The warp-MMA dense kernel's plan and grid: tokens per pass (all T rows up to
// four n-tiles), warps per tile by K alone, then the ring with the most bytes
// in flight on an SM (chunks of 1 or 2 64-column blocks, 2 to 4 stages a warp,
// one or two CTAs an SM); one wave of CTAs over the 16-row tiles, plus the
// routing CTA.  False when no plan fits shared memory.
struct DmLaunch {
  DmPlan plan{};
  int tile_ctas = 1, grid = 1, route_ctas = 0;
};
static bool dm_choose(int K, int T, bool split, int ntiles, int t_router, int num_sms, bool fuse,
                      size_t min_smem, DmLaunch* o) {
  const int tpn = split ? 4 : 8;
  const int nkc = K / 64;
  const int ks = nkc >= 64 ? 8 : (nkc >= 32 ? 4 : (nkc >= 16 ? 2 : 1));
  int ntp = 1;
  while (ntp < 4 && ntp * tpn < T) ntp *= 2;
  static const int kCkNs[][2] = {{2, 4}, {2, 3}, {1, 4}, {2, 2}, {1, 3}, {1, 2}};
  for (; ntp >= 1; ntp >>= 1) {
    long best = -1;
    for (int per_sm = 1; per_sm <= (ntp == 1 ? 2 : 1); ++per_sm) {   // registers: two CTAs with one n-tile
      const int budget = per_sm == 2 ? 110 * 1024 : kSmemMax - 2048;
      for (const auto& cn : kCkNs) {
        const DmPlan p = dm_plan(K, cn[0], cn[1], ntp * tpn, ks, split);
        if (static_cast<size_t>(p.smem) > static_cast<size_t>(budget) || min_smem > static_cast<size_t>(budget)) continue;
        const long inflight = static_cast<long>(per_sm) * cn[0] * cn[1];
        if (inflight > best) {
          best = inflight;
          o->plan = p;
          o->tile_ctas = std::max(1, std::min(ntiles, num_sms * per_sm - (fuse ? 1 : 0)));
        }
      }
    }
    if (best > 0) break;
  }
  if (ntp < 1) return false;
  o->grid = o->tile_ctas + (fuse ? 1 : 0);
  // router tiles first, about one a CTA on a quarter of the CTAs at most
  // (dm_cta_tiles); a single tile CTA holds everything
  o->route_ctas = fuse ? std::min(o->tile_ctas, std::min(t_router, std::max(1, o->tile_ctas / 4))) : 0;
  return true;
}
template <int NTP, bool SPLIT>
static cudaError_t launch_dense_mma_t(const DmArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  return launch_ex<DmArgs>(k_dense_mma<NTP, SPLIT>, grid, EM_NT, smem, s, pdl, a);
}
static cudaError_t launch_dense_mma(DmArgs a, const DmLaunch& dl, size_t smem, cudaStream_t s, bool pdl) {
  a.ck = dl.plan.ck;
  a.ns = dl.plan.ns;
  a.tp = dl.plan.tp;
  a.ks = dl.plan.ks;
  a.tile_ctas = dl.tile_ctas;
  a.route_ctas = dl.route_ctas;
  const int ntp = dm_ntp(dl.plan.tp, dl.plan.split);
  if (dl.plan.split) {
    if (ntp == 1) return launch_dense_mma_t<1, true>(a, dl.grid, smem, s, pdl);
    if (ntp == 2) return launch_dense_mma_t<2, true>(a, dl.grid, smem, s, pdl);
    return launch_dense_mma_t<4, true>(a, dl.grid, smem, s, pdl);
  }
  if (ntp == 1) return launch_dense_mma_t<1, false>(a, dl.grid, smem, s, pdl);
  if (ntp == 2) return launch_dense_mma_t<2, false>(a, dl.grid, smem, s, pdl);
  return launch_dense_mma_t<4, false>(a, dl.grid, smem, s, pdl);
}

template <int NTP, int GB, int FMT>
static cudaError_t launch_expert_mma_t(const ExpertArgs& a, bool gated, int grid, size_t smem, cudaStream_t s,
                                       bool pdl) {
  if (gated) return launch_ex<ExpertArgs>(k_expert_mma<true, NTP, GB, FMT>, grid, EM_NT, smem, s, pdl, a);
  return launch_ex<ExpertArgs>(k_expert_mma<false, NTP, GB, FMT>, grid, EM_NT, smem, s, pdl, a);
}
template <int GB, int FMT = 0>
static cudaError_t launch_expert_mma_g(const ExpertArgs& a, bool gated, int pp, int grid, size_t smem,
                                       cudaStream_t s, bool pdl) {
  if (pp <= 4) return launch_expert_mma_t<1, GB, FMT>(a, gated, grid, smem, s, pdl);
  if (pp <= 8) return launch_expert_mma_t<2, GB, FMT>(a, gated, grid, smem, s, pdl);
  return launch_expert_mma_t<4, GB, FMT>(a, gated, grid, smem, s, pdl);
}
// (a.G: the columns a scale word covers -- 64 for the fp4 formats)
static cudaError_t launch_expert_mma(ExpertArgs a, const EmLaunch& el, int T, int grid, cudaStream_t s,
                                     bool pdl) {
  a.ck = el.plan.ck;
  a.nst = el.plan.ns;
  a.pp = el.plan.pp;
  a.ks = el.plan.ks;
  a.cps = el.cps;
  // a slot holds at most T pairs (a token picks an expert once)
  a.one_pass = T <= a.pp && (a.max_pairs <= 0 || a.max_pairs >= T);
  const size_t smem = static_cast<size_t>(el.plan.smem);
  const bool gated = a.qt_gate != nullptr;
  if (a.wfmt == MOE_WFMT_NVFP4) return launch_expert_mma_g<4, 1>(a, gated, el.plan.pp, grid, smem, s, pdl);
  if (a.wfmt == MOE_WFMT_MXFP4) return launch_expert_mma_g<4, 2>(a, gated, el.plan.pp, grid, smem, s, pdl);
  switch (a.G) {
    case 32: return launch_expert_mma_g<2>(a, gated, el.plan.pp, grid, smem, s, pdl);
    case 64: return launch_expert_mma_g<4>(a, gated, el.plan.pp, grid, smem, s, pdl);
    default: return launch_expert_mma_g<8>(a, gated, el.plan.pp, grid, smem, s, pdl);
  }
}

template <int TB>
static cudaError_t launch_dense_in_pdl_t(const DenseInArgs& a, int grid, cudaStream_t s) {
  return launch_ex<DenseInArgs>(k_dense_in<TB>, grid, NT, dense_smem<TB>(a.K), s, true, a);
}
// A dense_in launch (no fused routing) that may start before its predecessor ends.
static cudaError_t launch_dense_in_pdl(const DenseInArgs& a, int tb, int grid, cudaStream_t s) {
  switch (tb) {
    case 1: return launch_dense_in_pdl_t<1>(a, grid, s);
    case 2: return launch_dense_in_pdl_t<2>(a, grid, s);
    case 4: return launch_dense_in_pdl_t<4>(a, grid, s);
    default: return launch_dense_in_pdl_t<8>(a, grid, s);
  }
}

static cudaError_t launch_dense_in(const DenseInArgs& a, int tb, int grid, cudaStream_t s) {
  switch (tb) {
    case 1: return launch_dense_in_t<DenseInArgs, 1>(a, grid, s);
    case 2: return launch_dense_in_t<DenseInArgs, 2>(a, grid, s);
    case 4: return launch_dense_in_t<DenseInArgs, 4>(a, grid, s);
    default: return launch_dense_in_t<DenseInArgs, 8>(a, grid, s);
  }
}
static cudaError_t launch_dense_out(const DenseOutArgs& a, int tb, int grid, cudaStream_t s,
                                    bool pdl) {
  switch (tb) {
    case 1: return launch_dense_out_t<DenseOutArgs, 1>(a, grid, s, pdl);
    case 2: return launch_dense_out_t<DenseOutArgs, 2>(a, grid, s, pdl);
    case 4: return launch_dense_out_t<DenseOutArgs, 4>(a, grid, s, pdl);
    default: return launch_dense_out_t<DenseOutArgs, 8>(a, grid, s, pdl);
  }
}
// 2-, 3-, 5-, 6- and 8-bit codes: passes of one or two token pairs (pb above 2
// is clamped)
template <int B>
static cudaError_t launch_expert_b(const ExpertArgs& a, int pb, int grid, cudaStream_t s, bool pdl) {
  return pb <= 1 ? launch_expert_t<1, B>(a, grid, s, pdl) : launch_expert_t<2, B>(a, grid, s, pdl);
}
static cudaError_t launch_expert(const ExpertArgs& a, int pb, int grid, cudaStream_t s, bool pdl,
                                 int bits = 4) {
  switch (bits) {
    case 2: return launch_expert_b<2>(a, pb, grid, s, pdl);
    case 3: return launch_expert_b<3>(a, pb, grid, s, pdl);
    case 5: return launch_expert_b<5>(a, pb, grid, s, pdl);
    case 6: return launch_expert_b<6>(a, pb, grid, s, pdl);
    case 8: return launch_expert_b<8>(a, pb, grid, s, pdl);
    default: break;
  }
  switch (pb) {
    case 1: return launch_expert_t<1>(a, grid, s, pdl);
    case 2: return launch_expert_t<2>(a, grid, s, pdl);
    case 4: return launch_expert_t<4>(a, grid, s, pdl);
    default: return launch_expert_t<8>(a, grid, s, pdl);
  }
}

// Allow each kernel the dynamic shared memory left beside its static shared
// memory (227 KB per block in total).
template <typename F>
static cudaError_t set_smem_attr(F* fn) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(fn));
  if (e != cudaSuccess) return e;
  const int dyn = kSmemMax - static_cast<int>(fa.sharedSizeBytes);
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

static cudaError_t set_smem_attrs() {
  cudaError_t e = cudaSuccess;
#define MOE_SMEM_ATTR(fn) \
  if (e == cudaSuccess) e = set_smem_attr(fn);
  MOE_SMEM_ATTR(k_dense_in<1>) MOE_SMEM_ATTR(k_dense_in<2>) MOE_SMEM_ATTR(k_dense_in<4>)
  MOE_SMEM_ATTR(k_dense_in<8>) MOE_SMEM_ATTR(k_dense_out<1>) MOE_SMEM_ATTR(k_dense_out<2>)
  MOE_SMEM_ATTR(k_dense_out<4>) MOE_SMEM_ATTR(k_dense_out<8>)
  MOE_SMEM_ATTR((k_expert<1, false>)) MOE_SMEM_ATTR((k_expert<2, false>))
  MOE_SMEM_ATTR((k_expert<4, false>)) MOE_SMEM_ATTR((k_expert<8, false>))
  MOE_SMEM_ATTR((k_expert<1, true>)) MOE_SMEM_ATTR((k_expert<2, true>))
  MOE_SMEM_ATTR((k_expert<4, true>)) MOE_SMEM_ATTR((k_expert<8, true>))
#define MOE_SMEM_ATTR_EM(GB)                                                               \
  MOE_SMEM_ATTR((k_expert_mma<false, 1, GB>)) MOE_SMEM_ATTR((k_expert_mma<true, 1, GB>)) \
  MOE_SMEM_ATTR((k_expert_mma<false, 2, GB>)) MOE_SMEM_ATTR((k_expert_mma<true, 2, GB>)) \
  MOE_SMEM_ATTR((k_expert_mma<false, 4, GB>)) MOE_SMEM_ATTR((k_expert_mma<true, 4, GB>))
  MOE_SMEM_ATTR_EM(2) MOE_SMEM_ATTR_EM(4) MOE_SMEM_ATTR_EM(8)
#define MOE_SMEM_ATTR_FP4(F)                                                                   \
  MOE_SMEM_ATTR((k_expert_mma<false, 1, 4, F>)) MOE_SMEM_ATTR((k_expert_mma<true, 1, 4, F>)) \
  MOE_SMEM_ATTR((k_expert_mma<false, 2, 4, F>)) MOE_SMEM_ATTR((k_expert_mma<true, 2, 4, F>)) \
  MOE_SMEM_ATTR((k_expert_mma<false, 4, 4, F>)) MOE_SMEM_ATTR((k_expert_mma<true, 4, 4, F>))
  MOE_SMEM_ATTR_FP4(1) MOE_SMEM_ATTR_FP4(2)
#undef MOE_SMEM_ATTR_FP4
  MOE_SMEM_ATTR((k_dense_mma<1, false>)) MOE_SMEM_ATTR((k_dense_mma<2, false>))
  MOE_SMEM_ATTR((k_dense_mma<4, false>)) MOE_SMEM_ATTR((k_dense_mma<1, true>))
  MOE_SMEM_ATTR((k_dense_mma<2, true>)) MOE_SMEM_ATTR((k_dense_mma<4, true>))
#undef MOE_SMEM_ATTR_EM
#define MOE_SMEM_ATTR_BITS(B)                                                         \
  MOE_SMEM_ATTR((k_expert<1, false, B>)) MOE_SMEM_ATTR((k_expert<2, false, B>)) \
  MOE_SMEM_ATTR((k_expert<1, true, B>)) MOE_SMEM_ATTR((k_expert<2, true, B>))
  MOE_SMEM_ATTR_BITS(2) MOE_SMEM_ATTR_BITS(3) MOE_SMEM_ATTR_BITS(5) MOE_SMEM_ATTR_BITS(6)
  MOE_SMEM_ATTR_BITS(8)
#undef MOE_SMEM_ATTR_BITS
  MOE_SMEM_ATTR((k_expert_bulk<1, 8, false>)) MOE_SMEM_ATTR((k_expert_bulk<2, 4, false>))
  MOE_SMEM_ATTR((k_expert_bulk<4, 2, false>)) MOE_SMEM_ATTR((k_expert_bulk<8, 1, false>))
  MOE_SMEM_ATTR((k_expert_bulk<1, 1, false>)) MOE_SMEM_ATTR((k_expert_bulk<2, 1, false>))
  MOE_SMEM_ATTR((k_expert_bulk<4, 1, false>))
  MOE_SMEM_ATTR((k_expert_bulk<1, 8, true>)) MOE_SMEM_ATTR((k_expert_bulk<2, 4, true>))
  MOE_SMEM_ATTR((k_expert_bulk<4, 2, true>)) MOE_SMEM_ATTR((k_expert_bulk<8, 1, true>))
  MOE_SMEM_ATTR((k_expert_bulk<1, 1, true>)) MOE_SMEM_ATTR((k_expert_bulk<2, 1, true>))
  MOE_SMEM_ATTR((k_expert_bulk<4, 1, true>))
  MOE_SMEM_ATTR((k_dense_bulk<1, 1>)) MOE_SMEM_ATTR((k_dense_bulk<1, 2>)) MOE_SMEM_ATTR((k_dense_bulk<1, 3>))
  MOE_SMEM_ATTR((k_dense_bulk<2, 1>)) MOE_SMEM_ATTR((k_dense_bulk<2, 2>)) MOE_SMEM_ATTR((k_dense_bulk<2, 3>))
  MOE_SMEM_ATTR(k_umma) MOE_SMEM_ATTR(k_umma2) MOE_SMEM_ATTR(k_route) MOE_SMEM_ATTR(k_route_rows)
#undef MOE_SMEM_ATTR
  return e;
}

// ---------------------------------------------------------------------------
// create / destroy
// ---------------------------------------------------------------------------

#define MOE_TRY_CUDA(call, msg)                                              \
  do {                                                                       \
    cudaError_t _e = (call);                                                 \
    if (_e != cudaSuccess) {                                                 \
      why = std::string(msg) + ": " + cudaGetErrorString(_e);                \
      st = (_e == cudaErrorMemoryAllocation) ? MOE_ERR_OOM : MOE_ERR_CUDA;   \
      goto fail;                                                             \
    }                                                                        \
  } while (0)

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

int32_t moe_build_flags(void) {
  return MOE_CHECKS ? (MOE_BUILD_CHECKS | MOE_BUILD_NVTX_DEFAULT) : 0;
}

moe_status moe_layer_validate(const moe_layer_config* cfg, const moe_layer_weights* w) {
  std::string why;
  moe_status s = validate_impl(cfg, w, &why);
  if (s != MOE_OK) g_create_error = why;
  return s;
}

moe_status moe_layer_create(const moe_layer_config* cfg, const moe_layer_weights* w, void* stream,
                            moe_layer** out) {
  std::string why;
  moe_status st = MOE_OK;
  moe_layer* L = nullptr;
  if (out) *out = nullptr;
  if (!out || !w) {
    g_create_error = "out and weights must not be NULL";
    return MOE_ERR_INVALID_ARG;
  }
  st = validate_impl(cfg, w, &why);
  if (st != MOE_OK) {
    g_create_error = why;
    return st;
  }
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    g_create_error = "no CUDA device";
    return MOE_ERR_DEVICE;
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    g_create_error = std::string("device ") + prop.name + " is not compute capability 10.3";
    return MOE_ERR_DEVICE;
  }
  const moe_layer_config& c = *cfg;
  const int H = c.hidden, E = c.n_experts, k = c.top_k, F = c.expert_ffn, G = c.group_size;
  const int Lt = c.latent, Fs = c.shared_ffn, T = c.max_tokens;
  const int kin = Lt ? Lt : H;
  const bool gated = c.act == MOE_ACT_SWIGLU;
  const int kout = (Lt ? Lt : 0) + Fs;
  if (!dense_tb_cap(H) || (kout && !dense_tb_cap(kout)) || !expert_pb_cap(kin) ||
      !expert_pb_cap(F)) {
    g_create_error = "a reduction width exceeds the shared-memory staging limit";
    return MOE_ERR_UNSUPPORTED;
  }
  if (c.weight_format != MOE_WFMT_AFFINE) {
    // the fp4 expert kernel at four pairs a pass, which every batch can use
    EmLaunch p_up, p_dn;
    const int gx = c.weight_format == MOE_WFMT_NVFP4 ? 16 : 32;
    if (!em_choose(kin, 64, gated, 1, 4, F, 1, prop.multiProcessorCount, &p_up, gx) ||
        !em_choose(F, 64, false, 1, 4, kin, 1, prop.multiProcessorCount, &p_dn, gx)) {
      g_create_error = "no shared-memory plan of the fp4 expert kernel fits this shape";
      return MOE_ERR_UNSUPPORTED;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  L = new moe_layer();
  L->cfg = c;
  L->device = dev;
  L->num_sms = prop.multiProcessorCount;
  L->kin = kin;
  L->bits = c.bits == 0 ? 4 : c.bits;
  L->cfg.bits = L->bits;
  L->fmt = c.weight_format;
  L->off_fc1 = E;
  L->off_shg = E + Lt;
  L->off_shu = E + Lt + (gated ? Fs : 0);
  L->r_in = L->off_shu + Fs;
  L->umax = std::min(E, T * k);
  if (const char* env = std::getenv("MOE_GROUPED_MIN_T")) L->grouped_min_t = std::max(1, std::atoi(env));
  if (const char* env = std::getenv("MOE_EXPERT_SPLIT")) L->expert_split = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_PDL")) L->use_pdl = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_PDL_GROUPED")) L->pdl_grouped = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_PREFETCH")) L->prefetch = std::atoi(env);
  if (const char* env = std::getenv("MOE_EXPERT_PB")) L->expert_pb = std::max(1, std::min(8, std::atoi(env)));
  if (const char* env = std::getenv("MOE_EXPERT_TARGET")) L->expert_target = std::max(1, std::min(16, std::atoi(env)));
  if (const char* env = std::getenv("MOE_UMMA_CTAS")) L->umma_ctas = std::max(1, std::min(2, std::atoi(env)));
  if (const char* env = std::getenv("MOE_UMMA_V")) L->umma_v = std::max(0, std::min(2, std::atoi(env)));
  if (const char* env = std::getenv("MOE_GATHER_MIN_T")) L->gather_min_t = std::max(1, std::atoi(env));
  if (const char* env = std::getenv("MOE_ROUTE_RPC"))
    L->route_rpc = std::max(1, std::min(ROUTE_ROWS_PER_CTA, std::atoi(env)));
  if (const char* env = std::getenv("MOE_ROUTE_SMALL_T"))
    L->route_small_t = std::max(1, std::min(ROUTE_SMALL_T, std::atoi(env)));
  if (const char* env = std::getenv("MOE_UMMA_SUB")) L->umma_sub = std::max(1, std::min(2, std::atoi(env)));
  if (const char* env = std::getenv("MOE_UMMA_SLEEP")) L->umma_sleep_ns = std::max(0, std::min(2000, std::atoi(env)));
  if (const char* env = std::getenv("MOE_UMMA_ABUFS"))
    L->umma_abufs = std::max(2, std::min(UM_MAX_ABUFS, std::atoi(env)));
  if (const char* env = std::getenv("MOE_UMMA_TMA")) L->umma_tma = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_UMMA_NTILE"))
    L->umma_ntile_int4 = std::max(16, std::min(128, std::atoi(env))) & ~15;
  if (const char* env = std::getenv("MOE_FUSE_ROUTE")) L->fuse_route = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_SIDE_STREAM")) L->side_stream = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_EXPERT_BULK")) L->expert_bulk = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_DENSE_BULK")) L->dense_bulk = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_EXPERT_BULK_MAX_T")) L->expert_bulk_max_t = std::max(0, std::atoi(env));
  if (const char* env = std::getenv("MOE_EXPERT_MMA")) L->expert_mma = std::atoi(env) != 0;
  if (L->fmt != MOE_WFMT_AFFINE) L->expert_mma = true;   // the only kernel that decodes fp4
  if (const char* env = std::getenv("MOE_EXPERT_MMA_MAX_T")) L->expert_mma_max_t = std::max(0, std::atoi(env));
  if (const char* env = std::getenv("MOE_DENSE_MMA")) L->dense_mma = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_EXPERT_MMA_PP"))
    L->expert_mma_pp = std::max(4, std::min(EM_MAX_PAIRS, std::atoi(env)));
  if (const char* env = std::getenv("MOE_EXPERT_BULK_PB"))
    L->expert_bulk_pb = std::max(1, std::min(8, pow2_at_least(std::atoi(env), 8)));
  if (const char* env = std::getenv("MOE_FILL")) L->fill = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_FILL_CTAS")) L->fill_ctas = std::max(0, std::atoi(env));
  if (const char* env = std::getenv("MOE_ROUTE_WARM")) L->route_warm = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_ROUTE_MAXW")) L->route_max_w = std::max(1, std::min(8, std::atoi(env)));
  if (const char* env = std::getenv("MOE_SIDE_GRID")) L->side_grid = std::max(0, std::atoi(env));
  if (const char* env = std::getenv("MOE_DEBUG_ROUTE")) L->debug_route = std::atoi(env) != 0;
  if (const char* env = std::getenv("MOE_NVTX")) L->nvtx = std::atoi(env) != 0;
  {
    const size_t adt = dt_size(c.act_dtype), rdt = dt_size(c.router_dtype);
    const size_t sdt = dt_size(c.scale_dtype);
    const size_t nq_in = static_cast<size_t>(E) * F * (kin / 32) * L->bits;
    const size_t ng_in = static_cast<size_t>(E) * F * (kin / G);
    const size_t nq_dn = static_cast<size_t>(E) * kin * (F / 32) * L->bits;
    const size_t ng_dn = static_cast<size_t>(E) * kin * (F / G);
    (void)sdt;
    MOE_TRY_CUDA(set_smem_attrs(), "kernel attributes");
    MOE_TRY_CUDA(L->alloc(&L->router_w, static_cast<size_t>(E) * H * rdt), "router weight");
    MOE_TRY_CUDA(cudaMemcpyAsync(L->router_w, w->router_w, static_cast<size_t>(E) * H * rdt,
                                 cudaMemcpyDeviceToDevice, s), "router weight copy");
    if (c.has_router_bias) {
      MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->router_bias), E * sizeof(float)), "router bias");
      MOE_TRY_CUDA(cudaMemcpyAsync(L->router_bias, w->router_bias, E * sizeof(float),
                                   cudaMemcpyDeviceToDevice, s), "router bias copy");
    }
    if (Lt) {
      const size_t n = static_cast<size_t>(Lt) * H * adt;
      MOE_TRY_CUDA(L->alloc(&L->fc1, n), "fc1");
      MOE_TRY_CUDA(cudaMemcpyAsync(L->fc1, w->fc1_latent, n, cudaMemcpyDeviceToDevice, s), "fc1 copy");
      MOE_TRY_CUDA(L->alloc(&L->fc2, n), "fc2");
      MOE_TRY_CUDA(cudaMemcpyAsync(L->fc2, w->fc2_latent, n, cudaMemcpyDeviceToDevice, s), "fc2 copy");
    }
    auto copy_q = [&](uint32_t** dst, const uint32_t* src, size_t n) -> cudaError_t {
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), n * 4);
      if (e != cudaSuccess) return e;
      return cudaMemcpyAsync(*dst, src, n * 4, cudaMemcpyDeviceToDevice, s);
    };
    auto copy_sb = [&](uint32_t** dst, const void* sc, const void* bi, size_t n) -> cudaError_t {
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), n * 4);
      if (e != cudaSuccess) return e;
      const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
      k_interleave_sb<<<blocks, 256, 0, s>>>(static_cast<const unsigned short*>(sc),
                                             static_cast<const unsigned short*>(bi), *dst,
                                             static_cast<int64_t>(n));
      return cudaGetLastError();
    };
    const bool fp4 = L->fmt != MOE_WFMT_AFFINE, mx = L->fmt == MOE_WFMT_MXFP4;
    // the fp4 block scales as they are -- NVFP4: four E4M3 bytes a word (one
    // word per row and 64 columns) and the per-matrix fp32 scales; MXFP4: two
    // E8M0 bytes per row and 64 columns
    auto copy_fp4 = [&](uint32_t** dst, float** gdst, const void* sc, const void* gs, int rows,
                        int K) -> cudaError_t {
      const size_t nb = static_cast<size_t>(E) * rows * (K / 64) * (mx ? 2 : 4);
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), nb);
      if (e == cudaSuccess) e = cudaMemcpyAsync(*dst, sc, nb, cudaMemcpyDeviceToDevice, s);
      if (!mx) {
        if (e == cudaSuccess) e = L->alloc(reinterpret_cast<void**>(gdst), E * sizeof(float));
        if (e == cudaSuccess) e = cudaMemcpyAsync(*gdst, gs, E * sizeof(float), cudaMemcpyDeviceToDevice, s);
      }
      return e;
    };
    if (gated) {
      MOE_TRY_CUDA(copy_q(&L->gate_q, w->gate_q, nq_in), "gate codes");
      MOE_TRY_CUDA(fp4 ? copy_fp4(&L->gate_sb, &L->gate_gs, w->gate_s, w->gate_b, F, kin)
                       : copy_sb(&L->gate_sb, w->gate_s, w->gate_b, ng_in), "gate scales");
    }
    MOE_TRY_CUDA(copy_q(&L->up_q, w->up_q, nq_in), "up codes");
    MOE_TRY_CUDA(fp4 ? copy_fp4(&L->up_sb, &L->up_gs, w->up_s, w->up_b, F, kin)
                     : copy_sb(&L->up_sb, w->up_s, w->up_b, ng_in), "up scales");
    MOE_TRY_CUDA(copy_q(&L->down_q, w->down_q, nq_dn), "down codes");
    MOE_TRY_CUDA(fp4 ? copy_fp4(&L->down_sb, &L->down_gs, w->down_s, w->down_b, kin, F)
                     : copy_sb(&L->down_sb, w->down_s, w->down_b, ng_dn), "down scales");
    auto group_major = [&](uint32_t** dst, const uint32_t* src, int rows, int ngr) -> cudaError_t {
      const size_t n = static_cast<size_t>(E) * rows * ngr;
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), n * 4);
      if (e != cudaSuccess) return e;
      const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
      k_sb_group_major<<<blocks, 256, 0, s>>>(src, *dst, E, rows, ngr);
      return cudaGetLastError();
    };
    if (L->bits == 4 && !fp4) {   // the grouped GEMM's scale layout (4-bit affine codes only)
      if (gated) MOE_TRY_CUDA(group_major(&L->gate_sbT, L->gate_sb, F, kin / G), "gate scales");
      MOE_TRY_CUDA(group_major(&L->up_sbT, L->up_sb, F, kin / G), "up scales");
      MOE_TRY_CUDA(group_major(&L->down_sbT, L->down_sb, kin, F / G), "down scales");
    }
    // the warp-MMA expert kernel's tiled codes and scale/bias words (4-bit codes)
    auto tile_q = [&](uint32_t** dst, const uint32_t* src, int rows, int K) -> cudaError_t {
      const size_t n = static_cast<size_t>(E) * rows * (K / 8);
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), n * 4);
      if (e != cudaSuccess) return e;
      const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 8192));
      k_tile_codes<<<blocks, 256, 0, s>>>(src, *dst, E, rows, K);
      return cudaGetLastError();
    };
    auto tile_sb = [&](uint32_t** dst, const uint32_t* src, int rows, int ngr) -> cudaError_t {
      const size_t n = static_cast<size_t>(E) * rows * ngr;
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), n * 4);
      if (e != cudaSuccess) return e;
      const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 8192));
      k_tile_sb<<<blocks, 256, 0, s>>>(src, *dst, E, rows, ngr);
      return cudaGetLastError();
    };
    // MXFP4: 16-bit scale entries (two E8M0 bytes) per row and 64 columns
    auto tile_sb16 = [&](uint32_t** dst, const uint32_t* src, int rows, int nch) -> cudaError_t {
      const size_t n = static_cast<size_t>(E) * rows * nch;
      cudaError_t e = L->alloc(reinterpret_cast<void**>(dst), n * 2);
      if (e != cudaSuccess) return e;
      const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 8192));
      k_tile_sb16<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(src), reinterpret_cast<uint16_t*>(*dst),
                                         E, rows, nch);
      return cudaGetLastError();
    };
    if (L->bits == 4 && L->expert_mma) {
      const int Gs = fp4 ? 64 : G;   // columns a scale word (MXFP4: entry) covers
      auto tile_s = [&](uint32_t** dst, const uint32_t* src, int rows, int ngr) {
        return mx ? tile_sb16(dst, src, rows, ngr) : tile_sb(dst, src, rows, ngr);
      };
      if (gated) {
        MOE_TRY_CUDA(tile_q(&L->gate_qt, L->gate_q, F, kin), "gate tiles");
        MOE_TRY_CUDA(tile_s(&L->gate_sbt, L->gate_sb, F, kin / Gs), "gate tiles");
      }
      MOE_TRY_CUDA(tile_q(&L->up_qt, L->up_q, F, kin), "up tiles");
      MOE_TRY_CUDA(tile_s(&L->up_sbt, L->up_sb, F, kin / Gs), "up tiles");
      MOE_TRY_CUDA(tile_q(&L->down_qt, L->down_q, kin, F), "down tiles");
      MOE_TRY_CUDA(tile_s(&L->down_sbt, L->down_sb, kin, F / Gs), "down tiles");
    }
    if (Fs) {
      const size_t n = static_cast<size_t>(Fs) * H * adt;
      if (gated) {
        MOE_TRY_CUDA(L->alloc(&L->sh_gate, n), "shared gate");
        MOE_TRY_CUDA(cudaMemcpyAsync(L->sh_gate, w->sh_gate, n, cudaMemcpyDeviceToDevice, s), "shared gate copy");
      }
      MOE_TRY_CUDA(L->alloc(&L->sh_up, n), "shared up");
      MOE_TRY_CUDA(cudaMemcpyAsync(L->sh_up, w->sh_up, n, cudaMemcpyDeviceToDevice, s), "shared up copy");
      MOE_TRY_CUDA(L->alloc(&L->sh_down, n), "shared down");
      MOE_TRY_CUDA(cudaMemcpyAsync(L->sh_down, w->sh_down, n, cudaMemcpyDeviceToDevice, s), "shared down copy");
    }
    // the warp-MMA dense kernel's tiled bf16 matrices
    if (L->dense_mma && c.act_dtype == MOE_DTYPE_BF16 && c.router_dtype == MOE_DTYPE_BF16) {
      auto tile_d = [&](void** dst, const void* src, int rows, int K) -> cudaError_t {
        const size_t n = static_cast<size_t>((rows + 15) / 16) * 16 * K;
        cudaError_t e = L->alloc(dst, n * 2);
        if (e != cudaSuccess) return e;
        const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 8192));
        k_tile_dense<<<blocks, 256, 0, s>>>(static_cast<const unsigned short*>(src),
                                            static_cast<unsigned short*>(*dst), rows, K);
        return cudaGetLastError();
      };
      MOE_TRY_CUDA(tile_d(&L->router_t, L->router_w, E, H), "router tiles");
      if (Lt) {
        MOE_TRY_CUDA(tile_d(&L->fc1_t, L->fc1, Lt, H), "fc1 tiles");
        MOE_TRY_CUDA(tile_d(&L->fc2_t, L->fc2, H, Lt), "fc2 tiles");
      }
      if (Fs) {
        if (gated) MOE_TRY_CUDA(tile_d(&L->shg_t, L->sh_gate, Fs, H), "shared gate tiles");
        MOE_TRY_CUDA(tile_d(&L->shu_t, L->sh_up, Fs, H), "shared up tiles");
        MOE_TRY_CUDA(tile_d(&L->shd_t, L->sh_down, H, Fs), "shared down tiles");
      }
    }
    // workspace
    const size_t P = static_cast<size_t>(T) * k;
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->dense_in), static_cast<size_t>(T) * L->r_in * 4), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->ids), P * 4), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->wts), P * 4), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->meta), (2 + 2 * static_cast<size_t>(L->umax) + P) * 4), "workspace");
    MOE_TRY_CUDA(cudaMemsetAsync(L->meta, 0, (2 + 2 * static_cast<size_t>(L->umax) + P) * 4, s), "workspace clear");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->hbuf), P * F * 4), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->pexp), P * kin * 4), "workspace");
    // status words: flags, then the first index-check violation (site, index, bound)
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->status), 16), "workspace");
    MOE_TRY_CUDA(cudaMemsetAsync(L->status, 0, 16, s), "status clear");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->route_counter), 4), "workspace");
    MOE_TRY_CUDA(cudaMemsetAsync(L->route_counter, 0, 4, s), "counter clear");
    MOE_TRY_CUDA(L->alloc(&L->bout, static_cast<size_t>(T) * (Lt + Fs + 64) * 2), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->comb),
                          static_cast<size_t>(T) * (std::max(kin, Lt + Fs) + 64) * 4), "workspace");
    MOE_TRY_CUDA(L->alloc(&L->xl16, static_cast<size_t>(T) * (Lt + 64) * 2), "workspace");
    MOE_TRY_CUDA(L->alloc(&L->h16, P * F * 2), "workspace");
    if (T >= L->gather_min_t) MOE_TRY_CUDA(L->alloc(&L->xs, P * L->kin * 2), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->part),
                          static_cast<size_t>(UM_MAX_KSPLIT) * std::min(T, UM_KSPLIT_MAX_T) *
                              std::max(L->r_in, H) * 4), "workspace");
    if (T > L->route_small_t) {
      const size_t nw = static_cast<size_t>(E) * ((T + 31) / 32);
      MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->rmask), nw * 4), "workspace");
      MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->rpref), nw * 4), "workspace");
    }
    if (std::getenv("MOE_CTA_TRACE") && std::atoi(std::getenv("MOE_CTA_TRACE"))) {
      const size_t n = static_cast<size_t>(CT_SLOTS) * CT_MAX_CTAS * CT_STAMPS * 8;
      MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->ct_trace), n), "trace");
      MOE_TRY_CUDA(cudaMemsetAsync(L->ct_trace, 0, n, s), "trace");
    }
    if (std::getenv("MOE_UMMA_TRACE") && std::atoi(std::getenv("MOE_UMMA_TRACE"))) {
      MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->um_trace), 4 * UM_TRACE_WORDS * 8), "trace");
      MOE_TRY_CUDA(cudaMemsetAsync(L->um_trace, 0, 4 * UM_TRACE_WORDS * 8, s), "trace");
    }
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->sdbuf), static_cast<size_t>(T) * H * 4), "workspace");
    MOE_TRY_CUDA(L->alloc(reinterpret_cast<void**>(&L->ccnt), kCombineCounters * 4), "workspace");
    MOE_TRY_CUDA(cudaMemsetAsync(L->ccnt, 0, kCombineCounters * 4, s), "counter clear");
    if (Fs && L->side_stream) {
      // the routed chain and the shared expert each on a stream of their own,
      // forked from and joined back into the caller's stream every forward
      int least = 0, greatest = 0;
      MOE_TRY_CUDA(cudaDeviceGetStreamPriorityRange(&least, &greatest), "stream priorities");
      MOE_TRY_CUDA(cudaStreamCreateWithPriority(&L->hi_s, cudaStreamNonBlocking, greatest), "stream");
      MOE_TRY_CUDA(cudaStreamCreateWithPriority(&L->lo_s, cudaStreamNonBlocking, least), "stream");
      for (cudaEvent_t* ev : {&L->ev_fork, &L->ev_side, &L->ev_chain})
        MOE_TRY_CUDA(cudaEventCreateWithFlags(ev, cudaEventDisableTiming), "event");
    }
    MOE_TRY_CUDA(L->alloc(&L->x_stage, static_cast<size_t>(T) * H * adt), "workspace");
    MOE_TRY_CUDA(L->alloc(&L->out_stage, static_cast<size_t>(T) * H * adt), "workspace");
    MOE_TRY_CUDA(cudaStreamSynchronize(s), "create synchronise");
  }
  *out = L;
  return MOE_OK;
fail:
  if (L) {
    cudaStreamSynchronize(s);
    L->free_all();
    delete L;
  }
  g_create_error = why;
  return st;
}

moe_status moe_layer_destroy(moe_layer* h) {
  if (!h) return MOE_OK;
  cudaDeviceSynchronize();
  h->free_all();
  delete h;
  return MOE_OK;
}

// The CUDA driver API's tensor-map encoder (looked up once through the runtime).
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor maps of a grouped launch's A operand (layouts in UmmaArgs::tm).
// False -- A then goes by cp.async -- when the encoder is missing or a matrix
// breaks the copy engine's rules: 16-byte aligned bases and row strides,
// dense parts in whole 64-column chunks.
static bool umma_tensor_maps(UmmaArgs& a, int n_experts) {
  const auto enc = tmap_encoder();
  if (!enc) return false;
  const cuuint32_t unit[3] = {1, 1, 1};
  if (a.a_mode == UA_DENSE) {
    if (a.nseg < 1 || a.nseg > 4) return false;
    for (int si = 0; si < a.nseg; ++si) {
      const DenseSeg& S = a.seg[si];
      if (S.nparts < 1 || S.nparts > 2) return false;
      if (S.part[0].k0 != 0 || (S.nparts == 2 && S.part[1].k0 != S.part[0].wk)) return false;
      for (int p = 0; p < S.nparts; ++p) {
        const DensePart& Pt = S.part[p];
        if (Pt.wk % UM_KC || reinterpret_cast<uintptr_t>(Pt.w) % 16) return false;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Pt.wk), static_cast<cuuint64_t>(S.rows)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Pt.wk) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(UM_M)};
        if (enc(&a.tm[2 * si + p], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(Pt.w), dims, strides,
                box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return false;
      }
    }
    return true;
  }
  const cuuint64_t words = static_cast<cuuint64_t>(a.K / 8);
  const cuuint64_t rows = static_cast<cuuint64_t>(a.n_rows), ngr = static_cast<cuuint64_t>(a.K / a.G);
  const cuuint64_t dims[3] = {words, rows, static_cast<cuuint64_t>(n_experts)};
  const cuuint64_t strides[2] = {words * 4, words * 4 * rows};
  const int sub = a.sub > 1 ? 2 : 1;   // 64-column chunks per ring slot
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(8 * sub), 128, 1};
  // scale/bias words, group-major: 128 rows x the slot's groups
  const cuuint64_t sdims[3] = {rows, ngr, static_cast<cuuint64_t>(n_experts)};
  const cuuint64_t sstrides[2] = {rows * 4, rows * 4 * ngr};
  const cuuint32_t sbox[3] = {128, static_cast<cuuint32_t>(std::max(1, sub * UM_KC / a.G)), 1};
  if (a.n_rows % 4) return false;
  const uint32_t* qs[2] = {a.q, a.q2};
  const uint32_t* ss[2] = {a.sbT, a.sbT2};
  for (int i = 0; i < (a.q2 ? 2 : 1); ++i) {
    if (!qs[i] || !ss[i] || reinterpret_cast<uintptr_t>(qs[i]) % 16 || reinterpret_cast<uintptr_t>(ss[i]) % 16)
      return false;
    if (enc(&a.tm[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(qs[i]), dims, strides, box, unit,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
    if (enc(&a.tm[2 + i], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(ss[i]), sdims, sstrides, sbox,
            unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// Tensor map of a grouped launch's B operand (map [8]) when its rows form a
// plain matrix: the tokens of a dense launch, or the pairs' hidden rows in
// sorted order.  False (B then goes by cp.async) for gathered rows or when the
// base or the row stride breaks the 16-byte rule.
static bool umma_b_map(UmmaArgs& a) {
  const auto enc = tmap_encoder();
  if (!enc || (a.experts && !a.b_sorted)) return false;
  const char* base = static_cast<const char*>(a.b0) + a.b0_off * 2;
  const int64_t nrows = a.experts ? a.b_rows : a.n_tokens;
  if (reinterpret_cast<uintptr_t>(base) % 16 || (a.b0_stride * 2) % 16 || nrows < 1) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(nrows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.b0_stride) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(a.n_tile)};
  const cuuint32_t unit[2] = {1, 1};
  return enc(&a.tm[8], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<char*>(base), dims, strides, box, unit,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Which grouped GEMM a launch takes: k_umma2 for the dense projections at any
// T and for the experts up to 128 rows; above that the experts' wide token
// tiles run faster in k_umma (measured), unless MOE_UMMA_V forces one.
static bool umma_is_v2(const moe_layer* h, bool dense, int T) {
  if (h->umma_v == 1) return false;
  if (h->umma_v == 2) return true;
  return dense || T <= 128;
}

// Tokens per MMA and ring depth for a grouped launch, and its shared memory.
static size_t umma_config(UmmaArgs& a, int T, size_t budget, int int4_cap) {
  const bool gated = a.a_mode == UA_INT4 && a.q2 != nullptr;
  const int cap = a.a_mode == UA_DENSE ? 256 : int4_cap;
  a.n_tile = std::min(cap, (std::max(1, T) + 15) & ~15);
  const int sub = a.sub > 1 ? 2 : 1;
  int st = UM_MAX_STAGES;
  while (st > 3 && umma_plan(a.a_mode, gated, a.n_tile, st, a.abufs, sub, a.G).total > budget) --st;
  a.stages = st;
  return umma_plan(a.a_mode, gated, a.n_tile, st, a.abufs, sub, a.G).total;
}

// A grouped launch; a dense matrix with fewer 128-row tiles than SMs splits K
// over several CTAs and sums the partials in a second, deterministic pass.
static cudaError_t launch_umma(moe_layer* h, UmmaArgs& a, int T, cudaStream_t s, int* nl, bool pdl) {
  // two CTAs per SM when the accumulators fit twice in TMEM (256 columns each:
  // not gated), so that one CTA's copies and dequantisation overlap the other's
  const bool gated = a.a_mode == UA_INT4 && a.q2 != nullptr;
  const bool v2 = umma_is_v2(h, a.a_mode == UA_DENSE, T);
  int per_sm = 1;
  size_t smem = 0;
  // tokens per tile, ring depth, A tiles and CTAs per SM for `sub` chunks per slot
  auto configure = [&](int sub) {
    a.sub = sub;
    per_sm = (h->umma_ctas >= 2 && !gated) ? 2 : 1;
    a.abufs = 2;
    smem = umma_config(a, T, per_sm == 2 ? 110 * 1024 : 220 * 1024, h->umma_ntile_int4);
    if (per_sm == 2 && smem > 110 * 1024) {   // a wide token tile: one CTA per SM
      per_sm = 1;
      smem = umma_config(a, T, 220 * 1024, h->umma_ntile_int4);
    }
    if (v2 && a.a_mode == UA_INT4 && h->umma_abufs > 2) {
      // more dequantised A tiles in the ring, while it keeps at least 4 stages
      const int keep = a.stages;
      a.abufs = h->umma_abufs;
      const size_t sm = umma_config(a, T, per_sm == 2 ? 110 * 1024 : 220 * 1024, h->umma_ntile_int4);
      if (a.stages >= 4 && sm <= static_cast<size_t>(per_sm == 2 ? 110 * 1024 : 220 * 1024)) {
        smem = sm;
      } else {
        a.abufs = 2;
        a.stages = keep;
      }
    }
  };
  // two chunks per ring slot for int4 when every operand can go by tensor
  // copies (half the copy issues and slot handshakes per byte), unless the
  // wider slots would cost the second CTA per SM (measured: slower)
  const bool want2 = v2 && a.a_mode == UA_INT4 && h->umma_tma && h->umma_sub > 1;
  configure(want2 ? 2 : 1);
  if (want2 && per_sm == 1 && h->umma_ctas >= 2 && !gated) configure(1);
  a.ksplit = 1;
  if (!a.experts && T <= UM_KSPLIT_MAX_T) {
    // as many K parts as keep every unit in one wave of CTAs (k_umma2 tiles
    // each dense segment on its own)
    int mtiles = (a.n_rows + UM_M - 1) / UM_M;
    if (v2) {
      mtiles = 0;
      for (int si = 0; si < a.nseg; ++si) mtiles += (a.seg[si].rows + UM_M - 1) / UM_M;
    }
    const int nkc = a.K / UM_KC;
    int ks = std::max(1, h->num_sms * per_sm / std::max(1, mtiles));
    ks = std::min(ks, std::min(std::max(1, nkc / 4), UM_MAX_KSPLIT));
    a.ksplit = std::max(1, ks);
    a.part = h->part;
  }
  a.trace = nullptr;
  if (v2) {
    a.tma_a = (h->umma_tma && umma_tensor_maps(a, h->cfg.n_experts)) ? 1 : 0;
    a.tma_b = (h->umma_tma && umma_b_map(a)) ? 1 : 0;
    if (a.sub > 1 && !(a.tma_a && a.tma_b)) {   // a map was ruled out: one chunk per slot
      configure(1);
      a.tma_a = (h->umma_tma && umma_tensor_maps(a, h->cfg.n_experts)) ? 1 : 0;
      a.tma_b = (h->umma_tma && umma_b_map(a)) ? 1 : 0;
    }
    a.wait_sleep_ns = h->umma_sleep_ns;
    if (h->um_trace && h->um_trace_n < 4) a.trace = h->um_trace + static_cast<size_t>(h->um_trace_n++) * UM_TRACE_WORDS;
  } else {
    a.tma_a = a.tma_b = 0;
    if (a.b_sorted || a.out_sorted) return cudaErrorInvalidValue;   // sorted rows are k_umma2's
  }
  cudaError_t e = launch_ex<UmmaArgs>(v2 ? k_umma2 : k_umma, h->num_sms * per_sm, UM_THREADS, smem, s, pdl, a);
  if (e == cudaSuccess) ++*nl;
  if (e == cudaSuccess && a.ksplit > 1) {
    const int64_t n = static_cast<int64_t>(T) * a.n_rows;
    e = launch_ex<UmmaArgs>(k_umma_reduce, static_cast<int>(std::min<int64_t>((n + 255) / 256, h->num_sms * 8)),
                            256, 0, s, pdl, a);
    if (e == cudaSuccess) ++*nl;
  }
  return e;
}

}  // extern "C"

// Plan of a persistent-kernel launch: staged token rows per pass, per-warp
// ring depth and slot size, and the shared memory of one CTA.
// Diagnostics: CTA 0's role stamps per chunk of each grouped launch of the last
// forward, in microseconds since the CTA started (SM cycles at 2070 MHz).
static void print_umma_trace(moe_layer* h, cudaStream_t s) {
  std::vector<unsigned long long> t(static_cast<size_t>(4) * UM_TRACE_WORDS);
  const bool got = cudaMemcpyAsync(t.data(), h->um_trace, t.size() * 8, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
                   cudaStreamSynchronize(s) == cudaSuccess;
  cudaMemsetAsync(h->um_trace, 0, t.size() * 8, s);
  const int n = h->um_trace_n;
  h->um_trace_n = 0;
  if (!got) return;
  for (int l = 0; l < n; ++l) {
    const unsigned long long* L = t.data() + static_cast<size_t>(l) * UM_TRACE_WORDS;
    const unsigned long long t0 = L[UM_TRACE_CHUNKS * UM_TRACE_STAMPS];
    std::fprintf(stderr,
                 "umma trace launch %d: chunk: p_begin p_slot p_tx p_tma1 p_tma p_landed d_buf d_done m_start "
                 "m_issued p_arrived p_cpasync\n",
                 l);
    for (int c = 0; c < UM_TRACE_CHUNKS; ++c) {
      const unsigned long long* R = L + static_cast<size_t>(c) * UM_TRACE_STAMPS;
      if (!R[0] && !R[8]) continue;
      std::fprintf(stderr, "  %3d:", c);
      for (int k = 0; k < UM_TRACE_STAMPS; ++k)
        std::fprintf(stderr, " %7.3f", R[k] ? (static_cast<double>(R[k]) - static_cast<double>(t0)) / 2070.0 : -1.0);
      std::fprintf(stderr, "\n");
    }
  }
}

// Diagnostics: per launch of the last forward, the CTA count and the min /
// median / max over its CTAs of each stamp, in microseconds since the earliest
// stamp of the forward (one JSON line per launch on stderr).
static void print_cta_trace(moe_layer* h, cudaStream_t s) {
  const size_t per = static_cast<size_t>(CT_MAX_CTAS) * CT_STAMPS;
  std::vector<unsigned long long> t(per * CT_SLOTS);
  const bool got = cudaMemcpyAsync(t.data(), h->ct_trace, t.size() * 8, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
                   cudaStreamSynchronize(s) == cudaSuccess;
  cudaMemsetAsync(h->ct_trace, 0, t.size() * 8, s);
  const int n = h->ct_n;
  h->ct_n = 0;
  if (!got) return;
  unsigned long long t0 = ~0ull;
  for (size_t i = 0; i < per * n; ++i)
    if (t[i] && t[i] < t0 && (i % CT_STAMPS) < 14) t0 = t[i];
  for (int l = 0; l < n; ++l) {
    std::string line = std::string("cta_trace {\"launch\": ") + std::to_string(l) + ", \"kernel\": \"" +
                       h->ct_names[l] + "\"";
    int ctas = 0;
    for (int c = 0; c < CT_MAX_CTAS; ++c) ctas += t[l * per + static_cast<size_t>(c) * CT_STAMPS] != 0;
    line += ", \"ctas\": " + std::to_string(ctas);
    {
      // SM clock of the launch: clock64 cycles over globaltimer ns, entry to exit
      std::vector<double> mhz;
      for (int c = 0; c < CT_MAX_CTAS; ++c) {
        const unsigned long long* r = t.data() + l * per + static_cast<size_t>(c) * CT_STAMPS;
        if (r[0] && r[3] > r[0] + 1000 && r[15] > r[14]) mhz.push_back(1e3 * (r[15] - r[14]) / double(r[3] - r[0]));
      }
      if (!mhz.empty()) {
        std::sort(mhz.begin(), mhz.end());
        char buf[64];
        std::snprintf(buf, sizeof(buf), ", \"sm_mhz\": %.0f", mhz[mhz.size() / 2]);
        line += buf;
      }
    }
    for (int k = 0; k < 14; ++k) {
      std::vector<double> v;
      for (int c = 0; c < CT_MAX_CTAS; ++c) {
        const unsigned long long x = t[l * per + static_cast<size_t>(c) * CT_STAMPS + k];
        if (x) v.push_back((static_cast<double>(x) - static_cast<double>(t0)) * 1e-3);
      }
      if (v.empty()) continue;
      std::sort(v.begin(), v.end());
      char buf[160];
      std::snprintf(buf, sizeof(buf), ", \"s%d\": [%.2f, %.2f, %.2f, %.2f]", k, v.front(), v[v.size() / 10],
                    v[v.size() / 2], v.back());
      line += buf;
    }
    line += ", \"cta0\": [";
    for (int k = 0; k < 14; ++k) {
      const unsigned long long x = t[l * per + k];
      char buf[32];
      std::snprintf(buf, sizeof(buf), "%s%.2f", k ? ", " : "",
                    x ? (static_cast<double>(x) - static_cast<double>(t0)) * 1e-3 : -1.0);
      line += buf;
    }
    std::fprintf(stderr, "%s]}\n", line.c_str());
  }
}

// The path a forward of T rows takes (never AUTO).
static int choose_path(const moe_layer* h, int T) {
  // the tensor-core path decodes 4-bit affine codes only
  if (h->bits != 4 || h->fmt != MOE_WFMT_AFFINE) return MOE_PATH_GEMV;
  if (h->path == MOE_PATH_GROUPED || (h->path == MOE_PATH_AUTO && T >= h->grouped_min_t))
    return MOE_PATH_GROUPED;
  return MOE_PATH_GEMV;
}

extern "C" {

static moe_status forward_impl(moe_layer* h, const void* x, int32_t T, void* out, void* stream,
                               int32_t* ext_ids, float* ext_w, float* delta) {
  if (!h) return MOE_ERR_INVALID_ARG;
  const moe_layer_config& c = h->cfg;
  if (!x || !out || T < 1 || T > c.max_tokens) {
    h->last_error = "x/out must be non-NULL and 1 <= T <= max_tokens";
    return MOE_ERR_INVALID_ARG;
  }
  const size_t adt = dt_size(c.act_dtype);
  const size_t nbytes = static_cast<size_t>(T) * c.hidden * adt;
  const char* xb = static_cast<const char*>(x);
  const char* ob = static_cast<const char*>(out);
  if (xb < ob + nbytes && ob < xb + nbytes) {
    h->last_error = "x and out overlap";
    return MOE_ERR_INVALID_ARG;
  }
  const int path = choose_path(h, T);
  const bool grouped = path == MOE_PATH_GROUPED;
  // With expert_split (MOE_EXPERT_SPLIT=1), AUTO's grouped path splits the
  // routed experts by load: an expert with at most `expert_pb` token pairs in
  // this batch goes to the int4 gemv kernel (one pass over its rows), a busier
  // one to the tcgen05 grouped GEMM; both launch and each skips the other's
  // experts.  Forced GROUPED runs every expert on the tensor cores.
  const bool split_experts = grouped && h->path != MOE_PATH_GROUPED && h->expert_split;
  const bool experts_gemv = !grouped || split_experts;
  const bool experts_tc = grouped;
  int nl = 0;   // kernel launches of this forward
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = c.hidden, E = c.n_experts, k = c.top_k, F = c.expert_ffn, Lt = c.latent;
  const int Fs = c.shared_ffn, kin = h->kin;
  const bool gated = c.act == MOE_ACT_SWIGLU;
  const int kout = Lt + Fs;
  const int mma_dt = c.act_dtype;
  cudaError_t e = cudaSuccess;
  // stage boundaries: profiling events and, with h->nvtx, one NVTX range per
  // stage inside the forward's range (popped on every exit)
  static const char* const kStageRange[MOE_NUM_STAGES] = {
      "moe dense_in (router, fc1_latent, shared gate/up)", "moe route", "moe expert up",
      "moe expert down + combine", "moe dense_out (fc2_latent, shared down, residual)"};
  int nvtx_open = 0;
  auto mark = [&](int i) {
    if (h->profiling) cudaEventRecord(h->ev[i], s);
    if (h->nvtx) {
      if (i > 0 && nvtx_open > 1) { nvtxRangePop(); --nvtx_open; }
      if (i < MOE_NUM_STAGES) { nvtxRangePushA(kStageRange[i]); ++nvtx_open; }
    }
  };
  if (h->nvtx) {
    nvtxRangePushA(grouped ? "moe_layer_forward grouped" : "moe_layer_forward gemv");
    ++nvtx_open;
  }
  // diagnostics: the stamp buffer of the next launch (null unless MOE_CTA_TRACE)
  auto tslot = [&](const char* name) -> unsigned long long* {
    if (!h->ct_trace || h->ct_n >= CT_SLOTS) return nullptr;
    h->ct_names[h->ct_n] = name;
    return h->ct_trace + static_cast<size_t>(h->ct_n++) * CT_MAX_CTAS * CT_STAMPS;
  };
  auto seg1 = [&](DenseSeg* segs, int& ns, const void* w, int dt, int rows, int row0) {
    DenseSeg& S = segs[ns++];
    S.part[0] = DensePart{w, dt, 0, H};
    S.nparts = 1;
    S.row0 = row0;
    S.rows = rows;
  };

  RouteArgs ra{};
  ra.logits = h->dense_in;
  ra.r_in = h->r_in;
  ra.bias = h->router_bias;
  ra.E = E;
  ra.k = k;
  ra.T = T;
  ra.router = c.router;
  ra.renorm = c.renormalize;
  ra.scale = c.routed_scale;
  ra.ids = h->ids;
  ra.w = h->wts;
  ra.meta = h->meta;
  ra.umax = h->umax;
  ra.ext_ids = ext_ids;
  ra.ext_w = ext_w;
  ra.status = h->status;
  ra.debug_times = h->debug_route;
#if MOE_CHECKS
  // planted out-of-range metadata index for the checks' own test (read per call)
  if (const char* env = std::getenv("MOE_DEBUG_BAD_INDEX")) ra.debug_bad = std::atoi(env);
#endif
  ra.max_w = h->route_max_w;
  {
    const int P = T * k;
    const int W = (T + 31) / 32;
    ra.mask_words = (P > 256 && static_cast<int64_t>(E) * W * 4 <= 160 * 1024) ? W : 0;
  }
  const bool big_route = T > h->route_small_t;
  const bool fuse_route = !grouped && h->fuse_route && !big_route;
  const bool pdl = h->use_pdl && (!grouped || h->pdl_grouped) && !h->profiling;
  // The shared expert does not depend on the routing.  On the gemv path its
  // gate/up rows (sa) and down rows (so, fp32 output added by the output
  // kernel) leave the routed chain (router and fc1 rows, top-k, expert up,
  // expert down with the combine): either as CTAs of their own inside the
  // expert launches (fill: sa beside the up projection, so beside the down
  // projection), or on a stream of their own (side).  Not while profiling: the
  // per-stage events time the kernels one after the other.
  DenseInArgs sa{};
  DenseOutArgs so{};
  if (Fs) {
    int ns = 0;
    if (gated) seg1(sa.seg, ns, h->sh_gate, c.act_dtype, Fs, 0);
    seg1(sa.seg, ns, h->sh_up, c.act_dtype, Fs, gated ? Fs : 0);
    sa.nseg = ns;
    sa.total_rows = ns * Fs;
    sa.out_ld = h->r_in;
    sa.K = H;
    sa.x = x;
    sa.x_dt = c.act_dtype;
    sa.out = h->dense_in + h->off_shg;
    sa.T = T;
    so.seg[0].part[0] = DensePart{h->sh_down, c.act_dtype, 0, Fs};
    so.seg[0].nparts = 1;
    so.seg[0].row0 = 0;
    so.seg[0].rows = H;
    so.nseg = 1;
    so.total_rows = H;
    so.K = Fs;
    so.shared = Fs;
    so.dense_in = h->dense_in;
    so.r_in = h->r_in;
    so.sh_g_off = h->off_shg;
    so.sh_u_off = h->off_shu;
    so.act = c.act;
    so.out_f32 = h->sdbuf;
    so.x = x;
    so.x_dt = c.act_dtype;
    so.T = T;
    so.prefetch = (h->prefetch >> 2) & 1;
  }
  // expert kernels of the gemv path: bulk-copied weight groups for up to
  // expert_bulk_max_t rows (latency-bound: every CTA's bytes requested at once),
  // register-streamed k_expert above (both give the same bits for a row)
  const int slots_e = std::min(E, T * k);   // distinct-expert slots of the expert launches
  // the warp-MMA expert kernel (4-bit codes in its tiled layout)
  EmLaunch em_up, em_dn;
  // (NVFP4 layers have no other expert kernel: their scale words cover 64
  // columns, sums of x 16)
  const bool fp4 = h->fmt != MOE_WFMT_AFFINE;
  const int Gm = fp4 ? 64 : c.group_size;
  const int gx = h->fmt == MOE_WFMT_NVFP4 ? 16 : (h->fmt == MOE_WFMT_MXFP4 ? 32 : 0);   // columns of a sum of x
  const bool use_mma = h->expert_mma && h->up_qt && (fp4 || T <= h->expert_mma_max_t);
  // (a gated up projection with 32-column groups folds twice per 64 columns and
  // two matrices: there the CUDA-core kernels measured faster, 59 vs 73 us at
  // T = 1 on the non-latent layer; the choice depends on the shape alone)
  const bool mma_up = use_mma && (fp4 || !(gated && c.group_size == 32)) &&
                      em_choose(kin, Gm, gated, T, h->expert_mma_pp, F, slots_e, h->num_sms, &em_up, gx);
  const bool mma_dn = use_mma && em_choose(F, Gm, false, T, h->expert_mma_pp, kin, slots_e,
                                           h->num_sms, &em_dn, gx);
  if (fp4 && !grouped && (!mma_up || !mma_dn)) {
    // (create refused layers without a plan at four pairs a pass, which every
    // batch size can fall back to)
    for (; nvtx_open > 0; --nvtx_open) nvtxRangePop();
    h->last_error = "no shared-memory plan of the NVFP4 expert kernel fits this shape";
    return MOE_ERR_UNSUPPORTED;
  }
  const bool use_bulk = h->expert_bulk && !grouped && T <= h->expert_bulk_max_t && h->bits == 4 && !fp4;
  EbLaunch eb_up, eb_dn;
  int cps_up = 1, cps_dn = 1;
  // pairs per pass: a distinct expert of a small batch holds one or two of its
  // rows, and its weights stay resident in the ring across passes
  const int eb_pb = std::min(pow2_at_least(T, 8), h->expert_bulk_pb);
  const bool bulk_up = use_bulk && eb_choose(kin, c.group_size, gated, eb_pb, F, slots_e,
                                             h->num_sms, &eb_up, &cps_up);
  const bool bulk_dn = use_bulk && eb_choose(F, c.group_size, false, eb_pb, kin, slots_e,
                                             h->num_sms, &eb_dn, &cps_dn);
  // the filler CTAs stage PB token rows of the dense rows' input: their shared
  // memory must fit beside the plan's CTAs per SM
  // fill: the shared expert's gate/up rows as a launch right after the first
  // kernel and its down rows right after the down projection, each starting
  // without a wait (its inputs are complete when it launches) beside the routed
  // chain's latency-bound kernels, and waiting for its predecessor only at its
  // end so that the stream's dependencies still run through it
  const bool fill = !grouped && Fs > 0 && h->fill && !h->profiling && h->use_pdl;
  const bool side = !grouped && !fill && Fs > 0 && h->side_stream && h->hi_s && !h->profiling;
  const bool shared_apart = side || fill;   // the shared expert is not in the first and last kernels
  const int fill_ctas = h->fill_ctas > 0 ? h->fill_ctas : h->num_sms;
  cudaStream_t cs = s;   // the routed chain's stream
  if (side) {
    if ((e = cudaEventRecord(h->ev_fork, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(h->hi_s, h->ev_fork, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(h->lo_s, h->ev_fork, 0)) != cudaSuccess)
      goto cuda_fail;
    cs = h->hi_s;
    const int sgrid = h->side_grid > 0 ? h->side_grid : h->num_sms;
    sa.trace = tslot("k_dense_in_shared");
    if ((e = launch_dense_in(sa, std::min(pow2_at_least(T, 8), dense_tb_cap(H)),
                             std::max(1, std::min(sgrid, (sa.total_rows + 3) / 4)), h->lo_s)) != cudaSuccess)
      goto cuda_fail;
    ++nl;
    so.trace = tslot("k_dense_out_shared");
    if ((e = launch_dense_out(so, std::min(pow2_at_least(T, 8), dense_tb_cap(Fs)),
                              std::max(1, std::min(sgrid, (H + 3) / 4)), h->lo_s, false)) != cudaSuccess)
      goto cuda_fail;
    ++nl;
    if ((e = cudaEventRecord(h->ev_side, h->lo_s)) != cudaSuccess) goto cuda_fail;
  }

  // 1. dense matrices that read x: router, fc1_latent_proj, shared gate/up
  mark(0);
  {
    const bool router_on_tc = grouped && c.router_dtype == c.act_dtype;
    DenseInArgs di{};
    int ns = 0;
    // the warp-MMA dense pass (bf16 layers on the gemv path)
    DmArgs dm{};
    DmLaunch dl_in;
    size_t rsm = 0;
    bool dm_in = false;
    if (!grouped && h->router_t && !shared_apart) {
      int n = 0;
      auto dseg = [&](const void* w, int rows, int col0) {
        dm.seg[n].w[0] = static_cast<const uint4*>(w);
        dm.seg[n].w[1] = nullptr;
        dm.seg[n].rows = rows;
        dm.seg[n].col0 = col0;
        ++n;
      };
      dseg(h->router_t, E, 0);
      if (Lt) dseg(h->fc1_t, Lt, h->off_fc1);
      if (Fs && gated) dseg(h->shg_t, Fs, h->off_shg);
      if (Fs) dseg(h->shu_t, Fs, h->off_shu);
      dm.nseg = n;
      dm.seg_t0[0] = 0;
      for (int i = 0; i < n; ++i) dm.seg_t0[i + 1] = dm.seg_t0[i] + (dm.seg[i].rows + 15) / 16;
      dm.in[0] = DmIn{x, c.act_dtype, H, 0, 0, 0, 0, H};
      dm.nparts = 1;
      dm.T = T;
      dm.out_mode = 0;
      dm.outf = h->dense_in;
      dm.out_ld = h->r_in;
      dm.status = h->status;
      dm.prefetch = 1;
      rsm = fuse_route ? ROUTE_SMEM_BYTES + static_cast<size_t>(E) * ra.mask_words * 4 : 0;
      dm_in = dm_choose(H, T, false, dm.seg_t0[n], dm.seg_t0[1], h->num_sms, fuse_route, rsm, &dl_in);
    }
    if (dm_in) {
      if (fuse_route) {
        dm.fuse_route = 1;
        dm.route = ra;
        dm.route_counter = h->route_counter;
        // MOE_DEBUG_STALL (tests of failure detection, read at every launch):
        // the routing CTA's bounded wait runs out
        const char* stall = std::getenv("MOE_DEBUG_STALL");
        dm.debug_stall = stall && std::atoi(stall) ? 1 : 0;
      }
      dm.trace = tslot("k_dense_mma_in");
      if ((e = launch_dense_mma(dm, dl_in, std::max(static_cast<size_t>(dl_in.plan.smem), rsm), cs, pdl)) != cudaSuccess)
        goto cuda_fail;
      ++nl;
    } else if (!grouped || !router_on_tc) {
      // CUDA-core pass: everything (gemv path) or only the router (grouped path
      // with a router dtype the tensor-core operands do not share)
      seg1(di.seg, ns, h->router_w, c.router_dtype, E, 0);
      if (!grouped) {
        if (Lt) seg1(di.seg, ns, h->fc1, c.act_dtype, Lt, h->off_fc1);
        if (Fs && gated && !shared_apart) seg1(di.seg, ns, h->sh_gate, c.act_dtype, Fs, h->off_shg);
        if (Fs && !shared_apart) seg1(di.seg, ns, h->sh_up, c.act_dtype, Fs, h->off_shu);
      }
      di.nseg = ns;
      di.total_rows = grouped ? E : (shared_apart ? E + Lt : h->r_in);
      di.out_ld = h->r_in;
      di.K = H;
      di.x = x;
      di.x_dt = c.act_dtype;
      di.out = h->dense_in;
      di.T = T;
      const int tb_in = std::min(pow2_at_least(T, 8), dense_tb_cap(H));
      int grid_in = std::max(1, std::min(h->num_sms * 2, (di.total_rows + 3) / 4));
      if (fuse_route) {
        di.fuse_route = 1;
        di.route = ra;
        di.route_counter = h->route_counter;
        // router rows get half the average rows per CTA
        const double share = static_cast<double>(E) / di.total_rows;
        int rc = static_cast<int>(grid_in * share * 2.0 + 0.5);
        if (h->route_warm) {
          // CTA 0 routes; CTAs 1..rc take the router rows, the rest the others
          const int rest = di.total_rows - E;
          grid_in = std::max(grid_in, rest ? 3 : 2);
          rc = rest ? std::max(1, std::min(rc, grid_in - 2)) : grid_in - 1;
          di.route_warm = 1;
          // MOE_DEBUG_STALL (tests of failure detection, read at every launch):
          // the routing CTA's bounded wait runs out
          const char* stall = std::getenv("MOE_DEBUG_STALL");
          di.debug_stall = stall && std::atoi(stall) ? 1 : 0;
        } else {
          rc = std::max(1, std::min(rc, std::min(E, grid_in - 1)));
          if (grid_in < 2) rc = 1;
        }
        di.route_ctas = rc;
        if (h->prefetch & 1) {
          di.prefetch_up = 1;
          di.pf_budget = 48ll << 20;
          di.pf_q = h->up_q;
          di.pf_sb = h->up_sb;
          di.pf_q2 = gated ? h->gate_q : nullptr;
          di.pf_sb2 = gated ? h->gate_sb : nullptr;
          di.pf_q_bytes = static_cast<int64_t>(F) * kin / 2;
          di.pf_sb_bytes = static_cast<int64_t>(F) * (kin / c.group_size) * 4;
        }
      }
      di.trace = tslot("k_dense_in");
      if ((e = launch_dense_in(di, tb_in, grid_in, cs)) != cudaSuccess) goto cuda_fail;
      ++nl;
      if (fill) {
        sa.dep_tail = 1;
        DbLaunch dl;
        if (h->dense_bulk && db_choose(sa.seg, sa.nseg, sa.total_rows, T, h->num_sms, &dl)) {
          DbArgs d = db_from_in(sa, h->dense_in, h->r_in, h->off_shg, h->status);
          d.trace = tslot("k_dense_bulk_shared_in");
          if ((e = launch_dense_bulk(d, dl, cs, true)) != cudaSuccess) goto cuda_fail;
        } else {
          sa.trace = tslot("k_dense_in_shared");
          if ((e = launch_dense_in_pdl(sa, std::min(pow2_at_least(T, 8), dense_tb_cap(H)),
                                       std::max(1, std::min(fill_ctas, (sa.total_rows + 3) / 4)), cs)) != cudaSuccess)
            goto cuda_fail;
        }
        ++nl;
      }
    }
    if (grouped) {
      UmmaArgs ua{};
      int n = 0;
      const int col0 = router_on_tc ? 0 : E;
      if (router_on_tc) seg1(ua.seg, n, h->router_w, c.router_dtype, E, 0);
      if (Lt) seg1(ua.seg, n, h->fc1, c.act_dtype, Lt, h->off_fc1 - col0);
      if (Fs && gated) seg1(ua.seg, n, h->sh_gate, c.act_dtype, Fs, h->off_shg - col0);
      if (Fs) seg1(ua.seg, n, h->sh_up, c.act_dtype, Fs, h->off_shu - col0);
      ua.nseg = n;
      ua.n_rows = h->r_in - col0;
      if (ua.n_rows > 0) {
        ua.experts = 0;
        ua.n_tokens = T;
        ua.K = H;
        ua.a_mode = UA_DENSE;
        ua.mma_dt = mma_dt;
        ua.b0 = x; ua.b0_stride = H; ua.b0_off = 0;
        if (Lt) {   // 16-bit copy of the latent columns: the experts' B operand
          ua.out16 = static_cast<unsigned short*>(h->xl16);
          ua.out16_ld = Lt;
          ua.c16_0 = h->off_fc1;
          ua.c16_1 = h->off_fc1 + Lt;
        }
        ua.epi = UE_DENSE_IN;
        ua.act = -1;
        ua.out_f32 = h->dense_in;
        ua.out_ld = h->r_in;
        ua.out_col0 = col0;
        ua.k = k;
        ua.status = h->status;
        if ((e = launch_umma(h, ua, T, s, &nl, pdl)) != cudaSuccess) goto cuda_fail;
      }
    }
  }

  // 2. routing (fused into the dense pass on the gemv path)
  mark(1);
  if (big_route) {
    // many rows: top-k over row blocks in parallel, then the lists in one CTA
    RouteArgs rr = ra;
    rr.mask_words = 0;
    // few rows per CTA while the grid stays small: four warps share a row's keys
    rr.rows_per_cta = T <= h->route_rpc_max_t ? h->route_rpc : ROUTE_ROWS_PER_CTA;
    if ((e = launch_ex<RouteArgs>(k_route_rows, (T + rr.rows_per_cta - 1) / rr.rows_per_cta,
                                  ROUTE_THREADS, ROUTE_SMEM_BYTES, cs, pdl, rr)) != cudaSuccess)
      goto cuda_fail;
    ++nl;
    ListArgs la{};
    la.ids = h->ids;
    la.T = T;
    la.k = k;
    la.E = E;
    la.umax = h->umax;
    la.meta = h->meta;
    la.mask = h->rmask;
    la.pref = h->rpref;
    la.W = (T + 31) / 32;
    if ((e = launch_ex<ListArgs>(k_route_lists, 1, LIST_THREADS, 0, cs, pdl, la)) != cudaSuccess)
      goto cuda_fail;
    ++nl;
  } else if (!fuse_route) {
    if ((e = launch_ex<RouteArgs>(k_route, 1, ROUTE_THREADS,
                                  ROUTE_SMEM_BYTES + static_cast<size_t>(E) * ra.mask_words * 4, cs,
                                  pdl, ra)) != cudaSuccess)
      goto cuda_fail;
    ++nl;
  }

  // 3. expert up (+gate) with the activation, 4. expert down
  {
    // token slots per pass of the gemv kernel; with the split, an expert with
    // at most pb_split pairs is the gemv kernel's, a busier one the GEMM's
    const int pb_split = std::min(std::min(pow2_at_least(T, h->expert_pb), expert_pb_cap(kin)),
                                  expert_pb_cap(F));
    // token slots per pass: most distinct experts hold one or two of the
    // batch's rows; experts with more loop over slot groups (L2 re-reads)
    const int pb_up = std::min(pow2_at_least(T, h->expert_pb), expert_pb_cap(kin));
    const int pb_dn = std::min(pow2_at_least(T, h->expert_pb), expert_pb_cap(F));
    // CTAs per distinct-expert slot: about expert_target resident CTAs per SM
    // over all slots (at most min(E, T*k) distinct experts), at least 8 rows each
    const int slots = std::min(E, T * k);
    const int target = h->num_sms * h->expert_target;
    ExpertArgs up{};
    UmmaArgs uup{};
    mark(2);
    if (experts_gemv) {
      up.n_rows = F;
      up.K = kin;
      up.G = Gm;
      up.wfmt = h->fmt;
      up.gsc = h->up_gs;          // (NVFP4 only; null otherwise)
      up.gsc_gate = gated ? h->gate_gs : nullptr;
      up.q = h->up_q;
      up.sb = h->up_sb;
      up.q_gate = gated ? h->gate_q : nullptr;
      up.sb_gate = gated ? h->gate_sb : nullptr;
      up.s_dt = c.scale_dtype;
      up.act = c.act;
      up.meta = h->meta;
      up.umax = h->umax;
      up.k = k;
      if (Lt) {
        up.xin = h->dense_in; up.xin_dt = DT_FP32; up.xin_stride = h->r_in; up.xin_off = h->off_fc1;
      } else {
        up.xin = x; up.xin_dt = c.act_dtype; up.xin_stride = H; up.xin_off = 0;
      }
      up.xin_by_pair = 0;
      up.out = h->hbuf;
      up.pre_wait_phase = 0;
      up.prefetch = 0;
      up.max_pairs = split_experts ? pb_split : 0;
      up.status = h->status;
      up.T = T;
      up.n_experts = E;
      up.gsh = c.group_size == 32 ? 0 : (c.group_size == 64 ? 1 : 2);
      if (mma_up) {
        up.qt = h->up_qt;
        up.sbt = h->up_sbt;
        up.qt_gate = gated ? h->gate_qt : nullptr;
        up.sbt_gate = gated ? h->gate_sbt : nullptr;
        up.trace = tslot("k_expert_mma_up");
        if ((e = launch_expert_mma(up, em_up, T, h->num_sms * em_up.per_sm, cs, pdl)) != cudaSuccess) goto cuda_fail;
        up.cps = em_up.cps;
      } else if (bulk_up) {
        // one wave: at most per_sm CTAs on every SM (one when the filler CTAs
        // take the other slot)
        up.cps = cps_up;
        up.nst = eb_up.nst;
        up.trace = tslot("k_expert_bulk_up");
        if ((e = launch_expert_bulk(up, eb_up, slots * up.cps, cs, pdl)) != cudaSuccess) goto cuda_fail;
      } else {
        up.cps = std::max(1, std::min(std::max(1, F / 8), (target + slots - 1) / slots));
        const int grid_up = slots * up.cps;
        up.trace = tslot("k_expert_up");
        if ((e = launch_expert(up, pb_up, grid_up, cs, pdl, h->bits)) != cudaSuccess) goto cuda_fail;
      }
      ++nl;

    }
    if (experts_tc) {
      uup.experts = 1;
      uup.min_pairs = split_experts ? pb_split + 1 : 0;
      uup.meta = h->meta;
      uup.umax = h->umax;
      uup.n_rows = F;
      uup.K = kin;
      uup.a_mode = UA_INT4;
      uup.q = h->up_q;
      uup.sb = h->up_sb;
      uup.q2 = gated ? h->gate_q : nullptr;
      uup.sb2 = gated ? h->gate_sb : nullptr;
      uup.G = c.group_size;
      uup.s_dt = c.scale_dtype;
      uup.mma_dt = mma_dt;
      if (Lt) {
        uup.b0 = h->xl16; uup.b0_stride = Lt; uup.b0_off = 0;
      } else {
        uup.b0 = x; uup.b0_stride = H; uup.b0_off = 0;
      }
      uup.out16 = static_cast<unsigned short*>(h->h16);   // the down GEMM's B operand
      uup.by_pair = 0;
      // hidden rows in the lists' sorted order (the down GEMM reads an expert's
      // rows as one block) unless the gemv kernel shares the buffer
      uup.out_sorted = (umma_is_v2(h, false, T) && !split_experts) ? 1 : 0;
      uup.sbT = h->up_sbT;
      uup.sbT2 = gated ? h->gate_sbT : nullptr;
      if (uup.out_sorted && h->xs && T >= h->gather_min_t && kin % 8 == 0 && uup.b0_stride % 8 == 0) {
        // the B rows in sorted pair order: an expert's rows are one block
        GatherArgs ga{};
        ga.meta = h->meta; ga.umax = h->umax; ga.k = k; ga.P = T * k; ga.K = kin;
        ga.status = h->status;
        ga.in = static_cast<const unsigned short*>(uup.b0); ga.in_stride = uup.b0_stride;
        ga.out = static_cast<unsigned short*>(h->xs);
        const int64_t n = static_cast<int64_t>(T) * k * (kin / 8);
        const int gg = static_cast<int>(std::min<int64_t>((n + 255) / 256, h->num_sms * 8));
        if ((e = launch_ex<GatherArgs>(k_gather_pairs, gg, 256, 0, s, pdl, ga)) != cudaSuccess) goto cuda_fail;
        ++nl;
        uup.b0 = h->xs; uup.b0_stride = kin; uup.b0_off = 0;
        uup.b_sorted = 1;
        uup.b_rows = T * k;
      }
      uup.k = k;
      uup.epi = UE_ROWS;
      uup.act = c.act;
      uup.out_f32 = h->hbuf;
      uup.status = h->status;
      uup.n_experts = E;
      uup.n_pairs = T * k;
      if ((e = launch_umma(h, uup, T, s, &nl, pdl)) != cudaSuccess) goto cuda_fail;

    }
    mark(3);
    if (experts_gemv) {
      ExpertArgs dn = up;
      dn.n_rows = kin;
      dn.K = F;
      dn.q = h->down_q;
      dn.sb = h->down_sb;
      dn.q_gate = nullptr;
      dn.sb_gate = nullptr;
      dn.act = -1;
      dn.xin = h->hbuf; dn.xin_dt = DT_FP32; dn.xin_stride = F; dn.xin_off = 0;
      dn.xin_by_pair = 1;
      dn.out = h->pexp;
      dn.pre_wait_phase = 1;
      dn.prefetch = (h->prefetch >> 1) & 1;
      if (!grouped) {
        // the weighted combine in the last CTA of each column range
        dn.comb = h->comb;
        dn.cwts = h->wts;
        dn.ccnt = h->ccnt;
        dn.T = T;
      }
      if (mma_dn) {
        dn.qt = h->down_qt;
        dn.sbt = h->down_sbt;
        dn.qt_gate = nullptr;
        dn.gsc = h->down_gs;
        dn.gsc_gate = nullptr;
        dn.sbt_gate = nullptr;
        dn.trace = tslot("k_expert_mma_down");
        if ((e = launch_expert_mma(dn, em_dn, T, h->num_sms * em_dn.per_sm, cs, pdl)) != cudaSuccess) goto cuda_fail;
      } else if (bulk_dn) {
        dn.cps = std::min(cps_dn, kCombineCounters);
        dn.nst = eb_dn.nst;
        dn.trace = tslot("k_expert_bulk_down");
        if ((e = launch_expert_bulk(dn, eb_dn, slots * dn.cps, cs, pdl)) != cudaSuccess) goto cuda_fail;
      } else {
        dn.cps = std::max(1, std::min(std::min(std::max(1, kin / 8), kCombineCounters),
                                      (target + slots - 1) / slots));
        dn.trace = tslot("k_expert_down");
        if ((e = launch_expert(dn, pb_dn, slots * dn.cps, cs, pdl, h->bits)) != cudaSuccess) goto cuda_fail;
      }
      if (fill) {
        so.dep_tail = 1;
        DbLaunch dl;
        if (h->dense_bulk && db_choose(so.seg, so.nseg, so.total_rows, T, h->num_sms, &dl)) {
          DbArgs d = db_from_out(so, h->status);
          d.trace = tslot("k_dense_bulk_shared_down");
          if ((e = launch_dense_bulk(d, dl, cs, true)) != cudaSuccess) goto cuda_fail;
        } else {
          so.trace = tslot("k_dense_out_shared");
          if ((e = launch_dense_out(so, std::min(pow2_at_least(T, 8), dense_tb_cap(Fs)),
                                    std::max(1, std::min(fill_ctas, (H + 3) / 4)), cs, true)) != cudaSuccess)
            goto cuda_fail;
        }
        ++nl;
      }
      ++nl;
    }
    if (experts_tc) {
      UmmaArgs udn = uup;
      udn.n_rows = kin;
      udn.K = F;
      udn.q = h->down_q;
      udn.sb = h->down_sb;
      udn.q2 = nullptr;
      udn.sb2 = nullptr;
      udn.b0 = h->h16; udn.b0_stride = F; udn.b0_off = 0;
      udn.out16 = nullptr;
      udn.by_pair = 1;
      udn.b_sorted = uup.out_sorted;
      udn.out_sorted = 0;
      udn.b_rows = T * k;
      udn.sbT = h->down_sbT;
      udn.sbT2 = nullptr;
      udn.act = -1;
      udn.out_f32 = h->pexp;
      if ((e = launch_umma(h, udn, T, s, &nl, pdl)) != cudaSuccess) goto cuda_fail;
    }
  }

  // 5. combine + fc2 + shared down + residual
  mark(4);
  if (grouped && kout) {
    PrepOutArgs pa{};
    pa.T = T; pa.L = Lt; pa.Fs = Fs; pa.k = k; pa.act = c.act; pa.mma_dt = mma_dt;
    pa.pexp = h->pexp; pa.wts = h->wts; pa.dense_in = h->dense_in; pa.r_in = h->r_in;
    pa.sh_g_off = h->off_shg; pa.sh_u_off = h->off_shu;
    pa.bout = static_cast<unsigned short*>(h->bout);
    const int64_t n = static_cast<int64_t>(T) * kout;
    if ((e = launch_ex<PrepOutArgs>(k_prep_out, static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096)), 256, 0,
                                    s, pdl, pa)) != cudaSuccess)
      goto cuda_fail;
    ++nl;
    UmmaArgs ua{};
    DenseSeg& S = ua.seg[0];
    S.nparts = 0;
    if (Lt) S.part[S.nparts++] = DensePart{h->fc2, c.act_dtype, 0, Lt};
    if (Fs) S.part[S.nparts++] = DensePart{h->sh_down, c.act_dtype, Lt, Fs};
    S.row0 = 0;
    S.rows = H;
    ua.nseg = 1;
    ua.experts = 0;
    ua.n_tokens = T;
    ua.n_rows = H;
    ua.K = kout;
    ua.a_mode = UA_DENSE;
    ua.mma_dt = mma_dt;
    ua.b0 = h->bout; ua.b0_stride = kout; ua.b0_off = 0;
    ua.k = k;
    ua.epi = UE_OUT;
    ua.x = x; ua.x_dt = c.act_dtype; ua.out = out; ua.delta = delta;
    ua.pexp = h->pexp; ua.wts = h->wts; ua.add_combine = Lt ? 0 : 1;
    ua.status = h->status;
    if ((e = launch_umma(h, ua, T, s, &nl, pdl)) != cudaSuccess) goto cuda_fail;
  } else {
    // the shared expert's output (side stream) is ready before the output kernel
    if (side && (e = cudaStreamWaitEvent(cs, h->ev_side, 0)) != cudaSuccess) goto cuda_fail;
    DenseOutArgs dout{};
    const int ks = Lt + (shared_apart ? 0 : Fs);   // staged width: [y (latent) | shared activation]
    dout.nseg = 0;
    if (ks) {
      DenseSeg& S = dout.seg[0];
      S.nparts = 0;
      if (Lt) S.part[S.nparts++] = DensePart{h->fc2, c.act_dtype, 0, Lt};
      if (Fs && !shared_apart) S.part[S.nparts++] = DensePart{h->sh_down, c.act_dtype, Lt, Fs};
      S.row0 = 0;
      S.rows = H;
      dout.nseg = 1;
    }
    dout.total_rows = H;
    dout.K = ks;
    dout.latent = Lt;
    dout.shared = shared_apart ? 0 : Fs;
    dout.staged = h->comb;          // y [T, kin] from the down projection's combine
    dout.staged_ld = kin;
    dout.dense_in = h->dense_in;
    dout.r_in = h->r_in;
    dout.sh_g_off = h->off_shg;
    dout.sh_u_off = h->off_shu;
    dout.act = c.act;
    if (grouped) {
      // grouped path without output projection: the experts wrote per-pick rows
      dout.pexp = h->pexp;
      dout.wts = h->wts;
      dout.k = k;
    } else {
      dout.y_add = Lt ? nullptr : h->comb;
    }
    dout.add_f32 = shared_apart ? h->sdbuf : nullptr;
    dout.x = x;
    dout.x_dt = c.act_dtype;
    dout.out = out;
    dout.delta = delta;
    dout.T = T;
    dout.prefetch = (h->prefetch >> 2) & 1;
    const int tb_out = ks ? std::min(pow2_at_least(T, 8), dense_tb_cap(ks)) : pow2_at_least(T, 8);
    const int grid_out = std::max(1, std::min(h->num_sms * 2, (H + 3) / 4));
    // the warp-MMA output pass (bf16 layers on the gemv path)
    DmArgs dmo{};
    DmLaunch dl_out;
    bool dm_out = false;
    if (!grouped && h->shd_t != nullptr && !shared_apart) {
      dmo.nseg = 1;
      dmo.seg[0].rows = H;
      dmo.seg[0].col0 = 0;
      dmo.seg_t0[0] = 0;
      dmo.seg_t0[1] = (H + 15) / 16;
      int np = 0;
      if (Lt) {
        dmo.seg[0].w[np] = static_cast<const uint4*>(h->fc2_t);
        dmo.in[np++] = DmIn{h->comb, DT_FP32, kin, 0, 0, 0, 0, Lt};
      }
      dmo.seg[0].w[np] = static_cast<const uint4*>(h->shd_t);
      dmo.in[np++] = DmIn{h->dense_in, DT_FP32, h->r_in, h->off_shu, h->off_shg, 1, c.act, Fs};
      dmo.nparts = np;
      dmo.T = T;
      dmo.out_mode = 1;
      dmo.x = x;
      dmo.x_dt = c.act_dtype;
      dmo.out = out;
      dmo.delta = delta;
      dmo.y_add = Lt ? nullptr : h->comb;
      dmo.H = H;
      dmo.status = h->status;
      dmo.prefetch = 1;
      dm_out = dm_choose(Lt + Fs, T, true, dmo.seg_t0[1], 0, h->num_sms, false, 0, &dl_out);
    }
    DbLaunch dl;
    if (dm_out) {
      dmo.trace = tslot("k_dense_mma_out");
      if ((e = launch_dense_mma(dmo, dl_out, static_cast<size_t>(dl_out.plan.smem), cs, pdl && !side)) != cudaSuccess)
        goto cuda_fail;
    } else if (h->dense_bulk && !grouped && ks && db_choose(dout.seg, dout.nseg, H, T, h->num_sms, &dl)) {
      DbArgs d = db_from_out(dout, h->status);
      d.trace = tslot("k_dense_bulk_out");
      if ((e = launch_dense_bulk(d, dl, cs, pdl && !side)) != cudaSuccess) goto cuda_fail;
    } else {
      dout.trace = tslot("k_dense_out");
      if ((e = launch_dense_out(dout, tb_out, grid_out, cs, pdl && !side)) != cudaSuccess) goto cuda_fail;
    }
    ++nl;
    if (side && ((e = cudaEventRecord(h->ev_chain, cs)) != cudaSuccess ||
                 (e = cudaStreamWaitEvent(s, h->ev_chain, 0)) != cudaSuccess))
      goto cuda_fail;
  }
  mark(5);
  for (; nvtx_open > 0; --nvtx_open) nvtxRangePop();
  if (h->profiling) h->profiled = true;
  h->last_launches = nl;
  if (h->um_trace) print_umma_trace(h, s);
  if (h->ct_trace && h->ct_n) print_cta_trace(h, s);
  return MOE_OK;
cuda_fail:
  for (; nvtx_open > 0; --nvtx_open) nvtxRangePop();
  h->last_error = std::string("launch failed: ") + cudaGetErrorString(e);
  return MOE_ERR_CUDA;
}

moe_status moe_layer_forward(moe_layer* h, const void* x, int32_t T, void* out, void* stream) {
  return forward_impl(h, x, T, out, stream, nullptr, nullptr, nullptr);
}

moe_status moe_layer_forward_ex(moe_layer* h, const void* x, int32_t T, void* out, void* stream,
                                int32_t* topk_ids, float* topk_w, float* delta_f32) {
  return forward_impl(h, x, T, out, stream, topk_ids, topk_w, delta_f32);
}

moe_status moe_layer_forward_host(moe_layer* h, const void* x_host, int32_t T, void* out_host,
                                  void* stream) {
  if (!h || !x_host || !out_host || T < 1 || T > h->cfg.max_tokens) {
    if (h) h->last_error = "host buffers must be non-NULL and 1 <= T <= max_tokens";
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = static_cast<size_t>(T) * h->cfg.hidden * dt_size(h->cfg.act_dtype);
  cudaError_t e = cudaMemcpyAsync(h->x_stage, x_host, n, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    h->last_error = std::string("input copy: ") + cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  moe_status st = forward_impl(h, h->x_stage, T, h->out_stage, stream, nullptr, nullptr, nullptr);
  if (st != MOE_OK) return st;
  e = cudaMemcpyAsync(out_host, h->out_stage, n, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    h->last_error = std::string("output copy: ") + cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_layer_set_path(moe_layer* h, int32_t path) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (path != MOE_PATH_AUTO && path != MOE_PATH_GEMV && path != MOE_PATH_GROUPED)
    return MOE_ERR_INVALID_ARG;
  if (path == MOE_PATH_GROUPED && h->cfg.act_dtype == MOE_DTYPE_FP32) {
    h->last_error = "the grouped path needs 16-bit activations";
    return MOE_ERR_UNSUPPORTED;
  }
  if (path == MOE_PATH_GROUPED && (h->bits != 4 || h->fmt != MOE_WFMT_AFFINE)) {
    h->last_error = "the grouped path decodes 4-bit affine codes only";
    return MOE_ERR_UNSUPPORTED;
  }
  h->path = path;
  return MOE_OK;
}

moe_status moe_layer_device_status(moe_layer* h, void* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v[4] = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(v, h->status, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->status, 0, sizeof(v), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    h->last_error = std::string("status read: ") + cudaGetErrorString(e);
    return MOE_ERR_CUDA;
  }
  if (v[0] & STATUS_INDEX) {
    static const char* const kSites[] = {"?", "k_expert expert id", "k_expert pair id",
                                         "k_expert_bulk expert id", "k_expert_bulk pair id",
                                         "k_gather_pairs pair id", "grouped GEMM expert id",
                                         "grouped GEMM pair id", "routing prefetch expert id",
                                         "distinct-expert pair range"};
    const int site = (v[1] >= 1 && v[1] <= 9) ? v[1] : 0;
    h->last_error = std::string("index check failed: ") + kSites[site] + " " + std::to_string(v[2]) +
                    " outside [0, " + std::to_string(v[3]) + ")";
    return MOE_ERR_INDEX;
  }
  if (v[0] & STATUS_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (v[0] & STATUS_NONFINITE) return MOE_ERR_NONFINITE;
  return MOE_OK;
}

moe_status moe_layer_profile(moe_layer* h, int32_t enable) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (enable && !h->profiling) {
    for (auto& e : h->ev) {
      if (cudaEventCreate(&e) != cudaSuccess) {
        h->free_events();
        h->last_error = "event creation failed";
        return MOE_ERR_CUDA;
      }
    }
  } else if (!enable && h->profiling) {
    cudaDeviceSynchronize();
    h->free_events();
  }
  h->profiling = enable != 0;
  h->profiled = false;
  return MOE_OK;
}

moe_status moe_layer_stage_times(moe_layer* h, float* ms, int32_t n) {
  if (!h || !ms || n < 0) return MOE_ERR_INVALID_ARG;
  if (!h->profiling || !h->profiled) {
    h->last_error = "no profiled forward";
    return MOE_ERR_INVALID_ARG;
  }
  if (cudaEventSynchronize(h->ev[MOE_NUM_STAGES]) != cudaSuccess) return MOE_ERR_CUDA;
  for (int i = 0; i < n && i < MOE_NUM_STAGES; ++i) {
    if (cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int64_t moe_layer_device_bytes(const moe_layer* h) { return h ? h->bytes : 0; }

int32_t moe_layer_path_for(const moe_layer* h, int32_t T) {
  if (!h || T < 1 || T > h->cfg.max_tokens) return -1;
  return choose_path(h, T);
}

int32_t moe_layer_last_launch_count(const moe_layer* h) { return h ? h->last_launches : 0; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_TOPK_GT_E: return "MOE_ERR_TOPK_GT_E";
    case MOE_ERR_LATENT_PROJ: return "MOE_ERR_LATENT_PROJ";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE";
    case MOE_ERR_INDEX: return "MOE_ERR_INDEX";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_layer_last_error(const moe_layer* h) {
  return h ? h->last_error.c_str() : g_create_error.c_str();
}

int64_t moe_debug_live_allocations(void) { return g_live_allocs.load(); }

void moe_debug_fail_allocation(int32_t n) { g_fail_countdown.store(n > 0 ? n : 0); }

}  // extern "C"
