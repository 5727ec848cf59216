// bf16-output GEMM (latent up-projection, with or without the shared
// expert's K-concatenated second operand pair; E4M3 operands with an fp32
// addend for the E4M3 shared expert).
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_bf16(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                             cudaStream_t s, bool f8, int pair_sms) {
  if (f8) return launch_gemm_impl<kEpiBf16, false, true>(m, a, grid, s, pair_sms);
  return dual ? launch_gemm_impl<kEpiBf16, true>(m, a, grid, s, pair_sms)
              : launch_gemm_impl<kEpiBf16, false>(m, a, grid, s, pair_sms);
}
}  // namespace lmoe
