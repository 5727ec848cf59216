// fp32-output GEMM (fp32 layer output; the E4M3 up-projection's partial sum).
#include "gemm_launch.cuh"

namespace lmoe {
cudaError_t launch_gemm_f32(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                            cudaStream_t s, bool f8, int pair_sms) {
  if (f8) return launch_gemm_impl<kEpiF32, false, true>(m, a, grid, s, pair_sms);
  return dual ? launch_gemm_impl<kEpiF32, true>(m, a, grid, s, pair_sms)
              : launch_gemm_impl<kEpiF32, false>(m, a, grid, s, pair_sms);
}
}  // namespace lmoe
