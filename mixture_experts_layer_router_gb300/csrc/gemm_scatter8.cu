// Latent down-projection with the scatter epilogue writing E4M3 codes of z
// (the token rows of the E4M3 expert GEMMs) and recording max |z|; bf16 or
// E4M3 operands.
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_scatter_f8(const GemmMaps& m, const GemmArgs& a, int grid,
                                   cudaStream_t s, bool f8, int pair_sms) {
  if (f8) return launch_gemm_impl<kEpiScatterF8, false, true>(m, a, grid, s, pair_sms);
  return launch_gemm_impl<kEpiScatterF8, false>(m, a, grid, s, pair_sms);
}
}  // namespace lmoe
