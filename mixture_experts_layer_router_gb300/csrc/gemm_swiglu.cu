// Gate+up GEMM with the SwiGLU epilogue (the shared expert's FFN input):
// bf16 output, or E4M3 operands and E4M3 output.
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_swiglu(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s,
                               bool f8, int pair_sms) {
  if (f8) return launch_gemm_impl<kEpiSwigluF8, false, true>(m, a, grid, s, pair_sms);
  return launch_gemm_impl<kEpiSwiglu, false>(m, a, grid, s, pair_sms);
}
}  // namespace lmoe
