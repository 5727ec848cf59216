// Launch of the SM-pair grouped expert GEMM (clusters of 2 CTAs).
#include <cstring>

#include "gemm_grouped2.cuh"
#include "kernels.h"

namespace lmoe {

template <int MODE, bool F8>
static cudaError_t launch_pair_impl(const CUtensorMap& tok, const CUtensorMap& w0,
                                    const CUtensorMap& w1, const GroupedArgs& a, int sms,
                                    cudaStream_t s) {
  static int max_clusters_of[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  int& max_clusters = max_clusters_of[dev];
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGThreads, 1, 1);
  cfg.dynamicSmemBytes = kPSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_grouped_pair_kernel<MODE, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPSmemBytes);
    if (e != cudaSuccess) return e;
    // as many pairs as can be resident at once (persistent tile loop)
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_grouped_pair_kernel<MODE, F8>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters = n < sms / 2 ? n : sms / 2;
  }
  return launch_kernel(gemm_grouped_pair_kernel<MODE, F8>, dim3(2 * max_clusters),
                       dim3(kGThreads), kPSmemBytes, s, 2, false, tok, w0, w1, a);
}

cudaError_t launch_gemm_grouped_pair(int mode, bool f8, const CUtensorMap& tok,
                                     const CUtensorMap& w0, const CUtensorMap& w1,
                                     const GroupedArgs& a, int sms, cudaStream_t s) {
  if (f8)
    return mode == kGrpSwiglu ? launch_pair_impl<kGrpSwiglu, true>(tok, w0, w1, a, sms, s)
                              : launch_pair_impl<kGrpPlain, true>(tok, w0, w1, a, sms, s);
  return mode == kGrpSwiglu ? launch_pair_impl<kGrpSwiglu, false>(tok, w0, w1, a, sms, s)
                            : launch_pair_impl<kGrpPlain, false>(tok, w0, w1, a, sms, s);
}


}  // namespace lmoe
