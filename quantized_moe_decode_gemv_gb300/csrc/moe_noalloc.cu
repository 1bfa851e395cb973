// Router gemv + top-k for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc where they need the routing decision:
// a runtime whose device memory is all owned by its own caching allocator and
// which forbids side allocations, a serving engine that plans every byte of
// device memory up front, or code on a latency-critical path where a device
// allocation (which may synchronise the device) is not acceptable.  Creating a
// moe_layer handle allocates a workspace, so those callers use this entry
// point instead.  It runs a CUDA-core router gemv (k_dense_in) and the top-k
// selection rules of moe_layer_forward_ex (the same routing block, stopping
// after the ids and weights) and writes
// topk_ids / topk_w, but keeps its scratch -- the router logits, a completion
// counter and a status word -- in a fixed-size array declared in this file.
// The caller passes only inputs and outputs (and, optionally, a device word
// that receives the non-finite-key flag).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "moe_layer.h"
#include "moe_kernels.cuh"

using namespace moe;

namespace {

constexpr int NA_MAX_T = MOE_NOALLOC_MAX_TOKENS;
// word offsets inside the scratch array (the selection writes its ids and
// weights straight to the caller's outputs and builds no expert lists)
constexpr size_t NA_OFF_LOGITS = 0;                                          // fp32 [T, E]
constexpr size_t NA_OFF_COUNTER = NA_OFF_LOGITS + static_cast<size_t>(NA_MAX_T) * MAX_E;
constexpr size_t NA_OFF_STATUS = NA_OFF_COUNTER + 1;
constexpr size_t NA_WORDS = NA_OFF_STATUS + 63;

// The scratch.  Every GPU that loads the library holds it until the process
// exits (256 KB).  In host code this name is only a host-side stand-in, so
// its device address is looked up with cudaGetSymbolAddress (noalloc_setup).
static __device__ __align__(256) uint32_t g_noalloc_scratch[NA_WORDS];

constexpr int NA_MAX_DEVICES = 64;
constexpr int kSmemLimit = 227 * 1024;
std::mutex g_na_mutex;
uint32_t* g_na_ptr[NA_MAX_DEVICES] = {};
int g_na_sms[NA_MAX_DEVICES] = {};

template <int TB>
cudaError_t na_attr() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(k_dense_in<TB>));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(k_dense_in<TB>),
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemLimit - static_cast<int>(fa.sharedSizeBytes));
}

// Once per device, with that device current: the device address of the
// scratch array, the SM count and the kernels' shared-memory limit.  The first
// call of the entry point on a device runs this, so that first call should be
// made before any stream capture.
moe_status noalloc_setup(uint32_t** ptr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_ptr[dev]) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_DEVICE;
    if (!(major == 10 && minor == 3)) return MOE_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    if (na_attr<1>() != cudaSuccess || na_attr<2>() != cudaSuccess || na_attr<4>() != cudaSuccess ||
        na_attr<8>() != cudaSuccess)
      return MOE_ERR_CUDA;
    g_na_sms[dev] = n;
    g_na_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *ptr = g_na_ptr[dev];
  *sms = g_na_sms[dev];
  return MOE_OK;
}

size_t na_dense_smem(int tb, int K) { return static_cast<size_t>(tb) * (4ull * K + 4ull * RED_ROWS * NW); }

}  // namespace

extern "C" moe_status moe_router_topk_noalloc(const void* x, int32_t T, int32_t hidden,
                                              int32_t x_dtype, const void* router_w,
                                              int32_t router_dtype, const float* router_bias,
                                              int32_t n_experts, int32_t top_k, int32_t router,
                                              int32_t renormalize, float routed_scale,
                                              int32_t* topk_ids, float* topk_w,
                                              int32_t* key_status, void* stream) {
  if (!x || !router_w || !topk_ids || !topk_w || T < 1 || hidden < 64 || hidden % 64)
    return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_FP16) return MOE_ERR_INVALID_ARG;
  if (router_dtype < MOE_DTYPE_BF16 || router_dtype > MOE_DTYPE_FP32) return MOE_ERR_INVALID_ARG;
  if (router != MOE_ROUTER_SOFTMAX && router != MOE_ROUTER_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (router_bias && router != MOE_ROUTER_SIGMOID) return MOE_ERR_UNSUPPORTED;
  if (n_experts < 1 || top_k < 1 || top_k > n_experts) return MOE_ERR_TOPK_GT_E;
  // sizes beyond the scratch array or the shared-memory staging
  if (T > NA_MAX_T || n_experts > MAX_E || top_k > MAX_K) return MOE_ERR_UNSUPPORTED;
  int tb = 8;
  while (tb > 1 && (tb > T || na_dense_smem(tb, hidden) > kSmemLimit - 2048)) tb >>= 1;
  if (na_dense_smem(tb, hidden) > kSmemLimit - 2048) return MOE_ERR_UNSUPPORTED;

  uint32_t* scratch = nullptr;
  int sms = 0;
  moe_status st = noalloc_setup(&scratch, &sms);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* counter = reinterpret_cast<int*>(scratch + NA_OFF_COUNTER);
  // the status word: the caller's when given (an output, not scratch)
  int* status = key_status ? key_status : reinterpret_cast<int*>(scratch + NA_OFF_STATUS);
  // the scratch keeps the last call's contents: the completion counter and the
  // status word must start at zero
  if (cudaMemsetAsync(counter, 0, sizeof(int), s) != cudaSuccess ||
      cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess)
    return MOE_ERR_CUDA;

  DenseInArgs di{};
  DenseSeg& S = di.seg[0];
  S.part[0] = DensePart{router_w, router_dtype, 0, hidden};
  S.nparts = 1;
  S.row0 = 0;
  S.rows = n_experts;
  di.nseg = 1;
  di.total_rows = n_experts;
  di.out_ld = n_experts;
  di.K = hidden;
  di.x = x;
  di.x_dt = x_dtype;
  di.out = reinterpret_cast<float*>(scratch + NA_OFF_LOGITS);
  di.T = T;
  const int grid = std::max(1, std::min(sms * 2, (n_experts + 3) / 4));
  RouteArgs& ra = di.route;
  ra.logits = di.out;
  ra.r_in = n_experts;
  ra.bias = router_bias;
  ra.E = n_experts;
  ra.k = top_k;
  ra.T = T;
  ra.router = router;
  ra.renorm = renormalize;
  ra.scale = routed_scale;
  ra.ids = topk_ids;
  ra.w = topk_w;
  ra.meta = nullptr;
  ra.umax = 0;
  ra.ext_ids = nullptr;
  ra.ext_w = nullptr;
  ra.status = status;
  ra.mask_words = 0;
  ra.topk_only = 1;   // ids and weights only: no distinct-expert lists
  ra.max_w = 8;
  di.fuse_route = 1;
  di.route_counter = counter;
  di.route_ctas = grid;   // every CTA holds router rows
  const size_t smem = std::max<size_t>(na_dense_smem(tb, hidden), ROUTE_SMEM_BYTES);
  switch (tb) {
    case 1: k_dense_in<1><<<grid, NT, smem, s>>>(di); break;
    case 2: k_dense_in<2><<<grid, NT, smem, s>>>(di); break;
    case 4: k_dense_in<4><<<grid, NT, smem, s>>>(di); break;
    default: k_dense_in<8><<<grid, NT, smem, s>>>(di); break;
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
