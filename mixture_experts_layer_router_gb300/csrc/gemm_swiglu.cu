// Gate+up GEMM with the SwiGLU epilogue (expert and shared-expert FFN input).
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_swiglu(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_gemm_impl<kEpiSwiglu, false>(m, a, grid, s);
}
}  // namespace lmoe
