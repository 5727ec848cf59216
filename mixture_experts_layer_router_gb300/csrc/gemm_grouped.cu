// Grouped expert GEMMs (weights on the M side): SwiGLU gate+up and plain down.
#include "gemm_grouped.cuh"
#include "kernels.h"

namespace lmoe {

template <int MODE>
static cudaError_t launch_grouped_impl(const CUtensorMap& tok, const CUtensorMap& w0,
                                       const CUtensorMap& w1, const GroupedArgs& a, int grid,
                                       cudaStream_t s) {
  static bool smem_set = false;
  if (!smem_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        gemm_grouped_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmemBytes);
    if (e != cudaSuccess) return e;
    smem_set = true;
  }
  gemm_grouped_kernel<MODE><<<grid, kGThreads, kGSmemBytes, s>>>(tok, w0, w1, a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_grouped(int mode, const CUtensorMap& tok, const CUtensorMap& w0,
                                const CUtensorMap& w1, const GroupedArgs& a, int grid,
                                cudaStream_t s) {
  return mode == kGrpSwiglu ? launch_grouped_impl<kGrpSwiglu>(tok, w0, w1, a, grid, s)
                            : launch_grouped_impl<kGrpPlain>(tok, w0, w1, a, grid, s);
}

}  // namespace lmoe
