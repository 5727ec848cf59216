// Gate-weighted combine: c[t] = sum_j g[t,j] * o[pos[t,j]], accumulated in
// fp32 in slot order j and rounded once to bf16.
//
// "The Training and RL Infrastructure Behind MAI-Thinking-1", section
// "2. Numerics": the MoE combine is one of the steps kept in FP32; section
// "Bitwise determinism": fixed-order accumulation instead of atomics. A
// gather (each token reads its k expert rows) needs no atomics at all.
//
// Bandwidth-bound: one block per token, each thread moves 16-byte vectors
// (8 bf16) of the k rows and of the output row.
//
// E4M3 variant: the expert outputs are read in fp32 (the E4M3 path keeps them
// unrounded) and the fp32 sum is quantized straight to E4M3 codes for the
// E4M3 up-projection.
#include "fp8.cuh"
#include "kernels.h"

namespace lmoe {

// F8: c is written as E4M3 codes of c * (1 / scale) (the latent input of the
// E4M3 up-projection) and max |c| is recorded in amax (one atomic per block).
// OF32: o is fp32 (kept unrounded for the E4M3 path) instead of bf16.
template <bool F8, bool OF32>
__global__ void __launch_bounds__(128) combine_kernel(const void* __restrict__ o_raw,
                                                      const float* __restrict__ gates,
                                                      const int* __restrict__ pos, int k, int l,
                                                      void* __restrict__ c,
                                                      const float* __restrict__ scale,
                                                      unsigned* __restrict__ amax,
                                                      long long o_rows, unsigned* status) {
  __shared__ float red[4];
  pdl_wait();
  pdl_launch_dependents();
  const float inv = F8 ? inv_scale(*scale) : 1.0f;
  float m = 0.0f;
  __shared__ int sp[16];
  __shared__ float sg[16];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    sp[threadIdx.x] = pos[static_cast<long long>(t) * k + threadIdx.x];
    sg[threadIdx.x] = gates[static_cast<long long>(t) * k + threadIdx.x];
  }
  __syncthreads();
  for (int col = threadIdx.x * 8; col < l; col += blockDim.x * 8) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int p = sp[j];
      if (p < 0 || !in_bounds(p, o_rows, status)) continue;
      const float g = sg[j];
      if constexpr (OF32) {
        const float4* src = reinterpret_cast<const float4*>(
            static_cast<const float*>(o_raw) + static_cast<long long>(p) * l + col);
        const float4 f0 = src[0], f1 = src[1];
        const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, f[i], acc[i]);
      } else {
        const uint4 raw = *reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(o_raw) + static_cast<long long>(p) * l + col);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h2[i]);
          acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
        }
      }
    }
    if constexpr (F8) {
      uint2 out;
      out.x = quant4_e4m3(acc[0], acc[1], acc[2], acc[3], inv);
      out.y = quant4_e4m3(acc[4], acc[5], acc[6], acc[7], inv);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(acc[i]));
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(c) + static_cast<long long>(t) * l + col) =
          out;
    } else {
      uint4 out;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
      for (int i = 0; i < 4; ++i) ow[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(c) + static_cast<long long>(t) * l +
                                col) = out;
    }
  }
  if constexpr (F8) {
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0)
      atomic_max_nonneg(amax, fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])));
  }
}

cudaError_t launch_combine(const __nv_bfloat16* o, const float* gates, const int* pos, int T,
                           int k, int l, __nv_bfloat16* c, long long o_rows, unsigned* status,
                           cudaStream_t s) {
  const cudaError_t e = launch_kernel(combine_kernel<false, false>, dim3(T), dim3(128), 0, s, 1,
                                      false, static_cast<const void*>(o), gates, pos, k, l,
                                      static_cast<void*>(c), static_cast<const float*>(nullptr),
                                      static_cast<unsigned*>(nullptr), o_rows, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_combine_f8(const float* o, const float* gates, const int* pos, int T, int k,
                              int l, uint8_t* c, const float* scale, unsigned* amax,
                              long long o_rows, unsigned* status, cudaStream_t s) {
  const cudaError_t e = launch_kernel(combine_kernel<true, true>, dim3(T), dim3(128), 0, s, 1,
                                      false, static_cast<const void*>(o), gates, pos, k, l,
                                      static_cast<void*>(c), scale, amax, o_rows, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace lmoe
