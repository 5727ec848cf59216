// Delayed scaling of the E4M3 activations.
//
// "The Training and RL Infrastructure Behind MAI-Thinking-1", section
// "2. Numerics": the scales of FP8 tensors come from a 1,024-step history of
// absolute maxima. Forward n quantizes with scale[i]; its kernels record
// amax[i] as they go; this kernel, launched after them on the same stream,
// enters amax[i] into the ring at position n mod 1024 and sets
//   scale[i] = max(ring[i]) / 448   (fp32, correctly rounded),
// leaving the scale unchanged while every entry of the ring is zero.
#include "fp8.cuh"
#include "kernels.h"

namespace lmoe {

__global__ void __launch_bounds__(256) fp8_update_kernel(Fp8State* st, int n) {
  __shared__ float red[8];
  const int slot = static_cast<int>(st->steps % kFp8History);
  for (int i = 0; i < n; ++i) {
    const float cur = __uint_as_float(st->amax[i]);
    float m = 0.0f;
    for (int j = threadIdx.x; j < kFp8History; j += blockDim.x)
      m = fmaxf(m, j == slot ? cur : st->hist[i][j]);
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mm = red[0];
      for (int w = 1; w < 8; ++w) mm = fmaxf(mm, red[w]);
      st->hist[i][slot] = cur;
      st->last_amax[i] = cur;
      st->amax[i] = 0u;
      if (mm > 0.0f) st->scale[i] = __fdiv_rn(mm, kE4M3Max);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) st->steps += 1;
}

cudaError_t launch_fp8_update(Fp8State* st, int n, cudaStream_t s) {
  if (n < 1 || n > kFp8Tensors) return cudaErrorInvalidValue;
  fp8_update_kernel<<<1, 256, 0, s>>>(st, n);
  return cudaGetLastError();
}

}  // namespace lmoe
