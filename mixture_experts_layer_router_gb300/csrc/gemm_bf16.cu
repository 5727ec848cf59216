// bf16-output GEMM (expert down-projection, latent up-projection, with or
// without the shared expert's K-concatenated second operand pair).
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_bf16(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                             cudaStream_t s) {
  return dual ? launch_gemm_impl<kEpiBf16, true>(m, a, grid, s)
              : launch_gemm_impl<kEpiBf16, false>(m, a, grid, s);
}
}  // namespace lmoe
