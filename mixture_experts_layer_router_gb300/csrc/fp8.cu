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

// E4M3 codes of a bf16 activation tensor with its current scale, recording
// max |x| (one atomic per block). 16 values per thread and step.
__global__ void __launch_bounds__(256) quantize_act_kernel(const uint4* __restrict__ src,
                                                           uint4* __restrict__ dst,
                                                           long long pieces,
                                                           const float* __restrict__ scale,
                                                           unsigned* __restrict__ amax) {
  __shared__ float red[8];
  const float inv = inv_scale(*scale);
  float m = 0.0f;
  for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < pieces;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 a = src[2 * q], b = src[2 * q + 1];
    const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
    float f[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(ha[i]);
      const float2 y = __bfloat1622float2(hb[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
      f[8 + 2 * i] = y.x;
      f[8 + 2 * i + 1] = y.y;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[i]));
    uint4 o;
    o.x = quant4_e4m3(f[0], f[1], f[2], f[3], inv);
    o.y = quant4_e4m3(f[4], f[5], f[6], f[7], inv);
    o.z = quant4_e4m3(f[8], f[9], f[10], f[11], inv);
    o.w = quant4_e4m3(f[12], f[13], f[14], f[15], inv);
    dst[q] = o;
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = red[0];
    for (int w = 1; w < 8; ++w) mm = fmaxf(mm, red[w]);
    atomic_max_nonneg(amax, mm);
  }
}

cudaError_t launch_quantize_act(const __nv_bfloat16* src, uint8_t* dst, long long n,
                                const float* scale, unsigned* amax, int sms, cudaStream_t s) {
  if (n % 16) return cudaErrorInvalidValue;
  const long long pieces = n / 16;
  long long grid = (pieces + 255) / 256;
  if (grid > static_cast<long long>(sms) * 8) grid = static_cast<long long>(sms) * 8;
  if (grid < 1) grid = 1;
  quantize_act_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), pieces, scale, amax);
  return cudaGetLastError();
}

cudaError_t launch_fp8_update(Fp8State* st, int n, cudaStream_t s) {
  if (n < 1 || n > kFp8Tensors) return cudaErrorInvalidValue;
  fp8_update_kernel<<<1, 256, 0, s>>>(st, n);
  return cudaGetLastError();
}

}  // namespace lmoe
