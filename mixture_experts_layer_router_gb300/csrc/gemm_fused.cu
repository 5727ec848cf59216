// Launch of the fused expert kernel (both expert GEMMs, clusters of 2 CTAs).
#include <cstring>

#include "gemm_fused.cuh"
#include "kernels.h"

namespace lmoe {

template <bool F8>
static cudaError_t launch_fused_impl(const CUtensorMap& z, const CUtensorMap& wg,
                                     const CUtensorMap& wu, const CUtensorMap& h,
                                     const CUtensorMap& wd, const FusedExpertArgs& a, int sms,
                                     cudaStream_t s) {
  static int max_clusters_of[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  int& max_clusters = max_clusters_of[dev];
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_expert_fused_kernel<F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kGThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_expert_fused_kernel<F8>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters = n < sms / 2 ? n : sms / 2;
  }
  // one pair per two SMs; the tile order needs no co-residency (gemm_fused.cuh)
  return launch_kernel(gemm_expert_fused_kernel<F8>, dim3(2 * max_clusters), dim3(kGThreads),
                       kPSmemBytes, s, 2, false, z, wg, wu, h, wd, a);
}

cudaError_t launch_expert_fused(bool f8, const CUtensorMap& z, const CUtensorMap& wg,
                                const CUtensorMap& wu, const CUtensorMap& h,
                                const CUtensorMap& wd, const FusedExpertArgs& a, int sms,
                                cudaStream_t s) {
  return f8 ? launch_fused_impl<true>(z, wg, wu, h, wd, a, sms, s)
            : launch_fused_impl<false>(z, wg, wu, h, wd, a, sms, s);
}

}  // namespace lmoe
