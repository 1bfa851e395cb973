// Host launcher of the persistent layer kernel for one staging width TB
// (this file is compiled once per TB, with -DFZ_TB=<1|2|4|8>, so that the
// instantiations build in parallel).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>

#include "moe_fused.cuh"

#ifndef FZ_TB
#error "compile with -DFZ_TB=1, 2, 4 or 8"
#endif

namespace moe {

namespace {

constexpr int kSmemMax = 227 * 1024;

template <bool GATED>
cudaError_t launch(const FusedArgs& a, size_t smem, int num_sms, FusedLaunchCache* cache, cudaStream_t s) {
  void (*kern)(FusedArgs) = k_fused<FZ_TB, fused_pb(FZ_TB), GATED>;
  if (cache->grid == 0 || cache->smem != smem) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemMax - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess) return e;
    // resident CTAs per SM at this shared memory; the kernel is compiled for two
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NT, smem);
    if (e != cudaSuccess) return e;
    cache->smem = smem;
    cache->grid = num_sms * std::min(nb, 2);
  }
  if (cache->grid < 2) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cache->grid);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

#define FZ_CAT2(a, b) a##b
#define FZ_CAT(a, b) FZ_CAT2(a, b)
cudaError_t FZ_CAT(fused_launch_tb, FZ_TB)(const FusedArgs& a, bool gated, size_t smem, int num_sms,
                                           FusedLaunchCache* cache, cudaStream_t s) {
  // MOE_DEBUG_STALL (tests of failure detection): make CTA 0's first wait run out
  const char* stall = std::getenv("MOE_DEBUG_STALL");
  if (stall && std::atoi(stall)) {
    FusedArgs b = a;
    b.debug_stall = 1;
    return gated ? launch<true>(b, smem, num_sms, cache, s) : launch<false>(b, smem, num_sms, cache, s);
  }
  return gated ? launch<true>(a, smem, num_sms, cache, s) : launch<false>(a, smem, num_sms, cache, s);
}

}  // namespace moe
