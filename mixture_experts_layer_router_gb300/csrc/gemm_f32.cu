// fp32-output GEMM (router logits with optional bias; fp32 layer output).
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_f32(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                            cudaStream_t s) {
  return dual ? launch_gemm_impl<kEpiF32, true>(m, a, grid, s)
              : launch_gemm_impl<kEpiF32, false>(m, a, grid, s);
}
}  // namespace lmoe
