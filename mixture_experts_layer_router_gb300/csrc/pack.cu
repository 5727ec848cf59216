// Weight preparation for the grouped expert GEMMs: tile packing, and E4M3
// quantization with one scale per expert matrix.
//
// A row-major matrix of rows x row_bytes is rewritten as tiles of 128 rows x
// 128 bytes, each tile one contiguous 16 KB block:
//   P[rt][kb][r][c] = W[rt*128 + r][kb*128 + c] (bytes), tile index rt * (row_bytes/128) + kb.
// The grouped GEMM then reads every weight tile with one sequential TMA load
// instead of 128 short pieces of rows that lie row_bytes apart. 128 bytes
// are kGBK bf16 or kGBK8 E4M3 columns.
//
// E4M3 weights ("The Training and RL Infrastructure Behind MAI-Thinking-1",
// section "2. Numerics": FP8 E4M3 forward GEMMs with per-tensor scales):
// for each expert matrix W_g, s = max |W| / 448 in fp32 and the codes are
// E4M3(W * (1/s)), so the largest weight maps to 448.
#include "fp8.cuh"
#include "kernels.h"

namespace lmoe {

namespace {

constexpr int kTileRowPieces = 8;                      // 16-byte pieces per 128-byte tile row
constexpr int kTilePieces = 128 * kTileRowPieces;      // pieces per tile

// Position (in 16-byte pieces) of piece (row, c16) of a row-major matrix with
// `row_pieces` pieces per row, in the packed tile layout.
__device__ __forceinline__ long long packed_piece(long long row, long long c16,
                                                  long long row_pieces) {
  const long long kb_count = row_pieces / kTileRowPieces;
  const long long rt = row >> 7;
  const int r = static_cast<int>(row & 127);
  const long long kb = c16 / kTileRowPieces;
  const int c = static_cast<int>(c16 - kb * kTileRowPieces);
  return (rt * kb_count + kb) * kTilePieces + r * kTileRowPieces + c;
}

}  // namespace

__global__ void __launch_bounds__(256) pack_tiles_kernel(const uint4* __restrict__ src,
                                                         uint4* __restrict__ dst, long long rows,
                                                         long long row_pieces) {
  const long long pieces = rows * row_pieces;
  for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < pieces;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = q / row_pieces;
    const long long c16 = q - row * row_pieces;
    dst[packed_piece(row, c16, row_pieces)] = src[q];
  }
}

cudaError_t launch_pack_tiles(const void* src, void* dst, long long rows, long long row_bytes,
                              int sms, cudaStream_t s) {
  pack_tiles_kernel<<<sms * 8, 256, 0, s>>>(static_cast<const uint4*>(src),
                                            static_cast<uint4*>(dst), rows, row_bytes / 16);
  return cudaGetLastError();
}

// grid.y = group; every block strides over its group's 8-element vectors.
__global__ void __launch_bounds__(256) absmax_groups_kernel(const uint4* __restrict__ src,
                                                            long long group_vecs,
                                                            unsigned* __restrict__ amax_bits) {
  const uint4* g = src + blockIdx.y * group_vecs;
  float m = 0.0f;
  for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < group_vecs;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 raw = g[q];
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h2[i]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomic_max_nonneg(&amax_bits[blockIdx.y], m);
}

cudaError_t launch_absmax_groups(const __nv_bfloat16* src, long long groups, long long group_elems,
                                 unsigned* amax_bits, int sms, cudaStream_t s) {
  if (groups < 1 || groups > 65535 || group_elems % 8) return cudaErrorInvalidValue;
  const long long vecs = group_elems / 8;
  long long bx = (static_cast<long long>(sms) * 8 + groups - 1) / groups;
  const long long need = (vecs + 255) / 256;
  if (bx > need) bx = need;
  if (bx < 1) bx = 1;
  absmax_groups_kernel<<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(groups)), 256, 0,
                         s>>>(reinterpret_cast<const uint4*>(src), vecs, amax_bits);
  return cudaGetLastError();
}

__global__ void scales_from_amax_kernel(const unsigned* __restrict__ amax_bits, int n,
                                        float* __restrict__ scale) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float m = __uint_as_float(amax_bits[i]);
    scale[i] = m > 0.0f ? __fdiv_rn(m, kE4M3Max) : 1.0f;
  }
}

cudaError_t launch_scales_from_amax(const unsigned* amax_bits, int n, float* scale,
                                    cudaStream_t s) {
  scales_from_amax_kernel<<<(n + 255) / 256, 256, 0, s>>>(amax_bits, n, scale);
  return cudaGetLastError();
}

// One thread per 16 output codes (two 16-byte source vectors).
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const uint4* __restrict__ src,
                                                            uint4* __restrict__ dst,
                                                            long long rows, long long row_pieces,
                                                            long long rows_per_group,
                                                            const float* __restrict__ scale,
                                                            int packed) {
  const long long pieces = rows * row_pieces;
  for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < pieces;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = q / row_pieces;
    const long long c16 = q - row * row_pieces;
    const float inv = inv_scale(scale[row / rows_per_group]);
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
    uint4 o;
    o.x = quant4_e4m3(f[0], f[1], f[2], f[3], inv);
    o.y = quant4_e4m3(f[4], f[5], f[6], f[7], inv);
    o.z = quant4_e4m3(f[8], f[9], f[10], f[11], inv);
    o.w = quant4_e4m3(f[12], f[13], f[14], f[15], inv);
    dst[packed ? packed_piece(row, c16, row_pieces) : q] = o;
  }
}

cudaError_t launch_quantize_e4m3(const __nv_bfloat16* src, uint8_t* dst, long long rows,
                                 long long K, long long rows_per_group, const float* scale,
                                 bool packed, int sms, cudaStream_t s) {
  if (K % 16 || rows_per_group < 1 || (packed && (K % 128 || rows_per_group % 128)))
    return cudaErrorInvalidValue;
  quantize_e4m3_kernel<<<sms * 8, 256, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                               reinterpret_cast<uint4*>(dst), rows, K / 16,
                                               rows_per_group, scale, packed ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace lmoe
