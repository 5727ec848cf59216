// Latent down-projection whose epilogue writes each token's row to its k
// expert-sorted slots (the dispatch, fused into the producing GEMM).
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_scatter(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s,
                                int pair_sms) {
  return launch_gemm_impl<kEpiScatter, false>(m, a, grid, s, pair_sms);
}
}  // namespace lmoe
