// Launch helper shared by the GEMM instantiation units: the one-SM kernel,
// or, for dense GEMMs given pair_sms > 0, the SM-pair kernel (clusters of 2).
#pragma once

#include <cstring>

#include "gemm2.cuh"
#include "kernels.h"

namespace lmoe {

template <int MODE, bool DUAL, bool F8>
static cudaError_t launch_gemm_pair_impl(const GemmMaps& m, const GemmArgs& a, int pair_sms,
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
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairGemmSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_pair_kernel<MODE, DUAL, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPairGemmSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (pair_sms / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel<MODE, DUAL, F8>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters = n;
  }
  // persistent pairs: no more than can be resident, than the SMs given, or
  // than there are pair tiles
  const long long tiles = static_cast<long long>((a.M + kPairBM - 1) / kPairBM) * a.n_tiles;
  long long pairs = pair_sms / 2;
  if (pairs > max_clusters) pairs = max_clusters;
  if (pairs > tiles) pairs = tiles;
  if (pairs < 1) pairs = 1;
  return launch_kernel(gemm_tc_pair_kernel<MODE, DUAL, F8>,
                       dim3(static_cast<unsigned>(2 * pairs)), dim3(kGemmThreads),
                       kPairGemmSmemBytes, s, 2, false, m.a, m.b, m.bu, m.a2, m.b2, a);
}

template <int MODE, bool DUAL, bool F8 = false>
static cudaError_t launch_gemm_impl(const GemmMaps& m, const GemmArgs& a, int grid,
                                    cudaStream_t s, int pair_sms = 0) {
  if (pair_sms >= 2 && !a.grouped) return launch_gemm_pair_impl<MODE, DUAL, F8>(m, a, pair_sms, s);
  static bool smem_set[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MODE, DUAL, F8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  return launch_kernel(gemm_tc_kernel<MODE, DUAL, F8>, dim3(grid), dim3(kGemmThreads),
                       kGemmSmemBytes, s, 1, false, m.a, m.b, m.bu, m.a2, m.b2, a);
}

}  // namespace lmoe
