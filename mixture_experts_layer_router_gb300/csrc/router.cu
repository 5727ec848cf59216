// Router GEMM + softmax + stable top-k (one fused kernel); see router.cuh.
#include "kernels.h"
#include "router.cuh"

namespace lmoe {

template <int KMAX, int BK>
static cudaError_t launch_router_impl(const CUtensorMap& x, const CUtensorMap& w, RouterArgs a,
                                      int sms, cudaStream_t s) {
  const int per_stage = router_stage_bytes(a.E);
  const int fixed = router_fixed_smem<KMAX>();
  a.stages = (kRMaxSmem - fixed) / per_stage;
  if (a.stages > kRMaxStages) a.stages = kRMaxStages;
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  const int smem = fixed + a.stages * per_stage;
  static bool smem_set[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!smem_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        router_topk_kernel<KMAX, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRMaxSmem);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  const int m_tiles = (a.T + 127) / 128;
  const int grid = m_tiles < sms ? m_tiles : sms;
  return launch_kernel(router_topk_kernel<KMAX, BK>, dim3(grid), dim3(kRThreads), smem, s, 1,
                       false, x, w, a);
}

cudaError_t launch_router_topk(const CUtensorMap& x, const CUtensorMap& w, RouterArgs a, int sms,
                               cudaStream_t s) {
  if (router_bk(a.E) == 128) {
    if (a.k <= 2) return launch_router_impl<2, 128>(x, w, a, sms, s);
    if (a.k <= 4) return launch_router_impl<4, 128>(x, w, a, sms, s);
    if (a.k <= 8) return launch_router_impl<8, 128>(x, w, a, sms, s);
    return launch_router_impl<16, 128>(x, w, a, sms, s);
  }
  if (router_bk(a.E) == 64) {
    if (a.k <= 2) return launch_router_impl<2, 64>(x, w, a, sms, s);
    if (a.k <= 4) return launch_router_impl<4, 64>(x, w, a, sms, s);
    if (a.k <= 8) return launch_router_impl<8, 64>(x, w, a, sms, s);
    return launch_router_impl<16, 64>(x, w, a, sms, s);
  }
  if (a.k <= 2) return launch_router_impl<2, 32>(x, w, a, sms, s);
  if (a.k <= 4) return launch_router_impl<4, 32>(x, w, a, sms, s);
  if (a.k <= 8) return launch_router_impl<8, 32>(x, w, a, sms, s);
  return launch_router_impl<16, 32>(x, w, a, sms, s);
}

}  // namespace lmoe
