// Launch helper shared by the GEMM instantiation units.
#pragma once

#include "gemm.cuh"
#include "kernels.h"

namespace lmoe {

template <int MODE, bool DUAL, bool F8 = false>
static cudaError_t launch_gemm_impl(const GemmMaps& m, const GemmArgs& a, int grid,
                                    cudaStream_t s) {
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
  gemm_tc_kernel<MODE, DUAL, F8><<<grid, kGemmThreads, kGemmSmemBytes, s>>>(m.a, m.b, m.bu, m.a2,
                                                                            m.b2, a);
  return cudaGetLastError();
}

}  // namespace lmoe
