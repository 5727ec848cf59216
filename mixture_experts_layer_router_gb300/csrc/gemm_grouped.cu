// Grouped expert GEMMs (weights on the M side): SwiGLU gate+up and plain
// down, with bf16 or E4M3 operands.
#include "gemm_grouped.cuh"
#include "kernels.h"

namespace lmoe {

template <int MODE, bool F8>
static cudaError_t launch_grouped_impl(const CUtensorMap& tok, const CUtensorMap& w0,
                                       const CUtensorMap& w1, const GroupedArgs& a, int grid,
                                       cudaStream_t s) {
  static bool smem_set[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_grouped_kernel<MODE, F8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kGSmemBytes);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  return launch_kernel(gemm_grouped_kernel<MODE, F8>, dim3(grid), dim3(kGThreads), kGSmemBytes,
                       s, 1, false, tok, w0, w1, a);
}

cudaError_t launch_gemm_grouped(int mode, bool f8, const CUtensorMap& tok, const CUtensorMap& w0,
                                const CUtensorMap& w1, const GroupedArgs& a, int grid,
                                cudaStream_t s) {
  if (f8)
    return mode == kGrpSwiglu ? launch_grouped_impl<kGrpSwiglu, true>(tok, w0, w1, a, grid, s)
                              : launch_grouped_impl<kGrpPlain, true>(tok, w0, w1, a, grid, s);
  return mode == kGrpSwiglu ? launch_grouped_impl<kGrpSwiglu, false>(tok, w0, w1, a, grid, s)
                            : launch_grouped_impl<kGrpPlain, false>(tok, w0, w1, a, grid, s);
}

}  // namespace lmoe
