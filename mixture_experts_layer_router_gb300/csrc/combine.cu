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
#include "kernels.h"

namespace lmoe {

__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const float* __restrict__ gates,
                                                      const int* __restrict__ pos, int k, int l,
                                                      __nv_bfloat16* __restrict__ c) {
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
      if (p < 0) continue;
      const uint4 raw = *reinterpret_cast<const uint4*>(o + static_cast<long long>(p) * l + col);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
      const float g = sg[j];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h2[i]);
        acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
      }
    }
    uint4 out;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) ow[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4*>(c + static_cast<long long>(t) * l + col) = out;
  }
}

cudaError_t launch_combine(const __nv_bfloat16* o, const float* gates, const int* pos, int T,
                           int k, int l, __nv_bfloat16* c, cudaStream_t s) {
  combine_kernel<<<T, 128, 0, s>>>(o, gates, pos, k, l, c);
  return cudaGetLastError();
}

}  // namespace lmoe
