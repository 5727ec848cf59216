// FP8 E4M3 helpers: quantization with a per-tensor scale, and the running
// absolute maximum that delayed scaling records.
//
// "The Training and RL Infrastructure Behind MAI-Thinking-1", section
// "2. Numerics": forward GEMMs in FP8 E4M3 with delayed per-tensor scaling.
// A tensor t with scale s is stored as the codes E4M3(t * (1/s)), rounded to
// nearest even and saturated at +-448, and stands for code * s.
#pragma once

#include <cuda_fp8.h>

#include "ptx.cuh"

namespace lmoe {

constexpr float kE4M3Max = 448.0f;

// Two codes, `lo` in the low byte. The product with the reciprocal scale is
// rounded to fp32 first, then converted (round to nearest even, saturating).
__device__ __forceinline__ uint32_t quant2_e4m3(float lo, float hi, float inv) {
  const float2 v = make_float2(__fmul_rn(lo, inv), __fmul_rn(hi, inv));
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Four codes, `a` in the low byte.
__device__ __forceinline__ uint32_t quant4_e4m3(float a, float b, float c, float d, float inv) {
  return quant2_e4m3(a, b, inv) | (quant2_e4m3(c, d, inv) << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Running maximum of non-negative floats kept as their bit patterns (which
// order like the values), so atomicMax on unsigned is a float max.
__device__ __forceinline__ void atomic_max_nonneg(unsigned* slot, float v) {
  if (v > 0.0f) atomicMax(slot, __float_as_uint(v));
}

// 1 / s, correctly rounded, for the quantizing side.
__device__ __forceinline__ float inv_scale(float s) { return __frcp_rn(s); }

}  // namespace lmoe
