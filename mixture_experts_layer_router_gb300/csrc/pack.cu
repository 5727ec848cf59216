// Weight repacking for the grouped expert GEMMs.
//
// A stack of weight rows W [rows, K] (bf16, K contiguous) is rewritten as
// tiles of 128 rows x kGBK columns, each tile one contiguous block:
//   P[rt][kb][r][c] = W[rt*128 + r][kb*kGBK + c],  tile index rt * (K/kGBK) + kb.
// The grouped GEMM then reads every weight tile with one sequential TMA load
// instead of 128 short pieces of rows that lie K*2 bytes apart.
#include "kernels.h"

namespace lmoe {

__global__ void __launch_bounds__(256) pack_weight_tiles_kernel(const uint4* __restrict__ src,
                                                                uint4* __restrict__ dst,
                                                                long long rows, int K) {
  constexpr int kRowPieces = kGBK / 8;            // 16-byte pieces per tile row
  constexpr int kTilePieces = 128 * kRowPieces;   // pieces per tile
  const int kb_count = K / kGBK;
  const long long pieces = rows * (K / 8);
  for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < pieces;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long tile = q / kTilePieces;
    const int within = static_cast<int>(q - tile * kTilePieces);
    const int r = within / kRowPieces;
    const int c = within - r * kRowPieces;
    const long long rt = tile / kb_count;
    const int kb = static_cast<int>(tile - rt * kb_count);
    const long long src_row = rt * 128 + r;
    dst[q] = src[(src_row * K + static_cast<long long>(kb) * kGBK) / 8 + c];
  }
}

cudaError_t launch_pack_tiles(const __nv_bfloat16* src, __nv_bfloat16* dst, long long rows, int K,
                              int sms, cudaStream_t s) {
  pack_weight_tiles_kernel<<<sms * 8, 256, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                                   reinterpret_cast<uint4*>(dst), rows, K);
  return cudaGetLastError();
}

}  // namespace lmoe
