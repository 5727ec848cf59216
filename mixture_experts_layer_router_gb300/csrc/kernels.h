// Host-side launchers of the library's kernels (internal interface).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gemm.cuh"
#include "gemm_grouped.cuh"
#include "router.cuh"

namespace lmoe {

struct GemmMaps {
  CUtensorMap a, b, bu, a2, b2;
};

// One launch of gemm_tc_kernel<MODE, DUAL>; `grid` persistent CTAs.
cudaError_t launch_gemm_bf16(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                             cudaStream_t s);
cudaError_t launch_gemm_f32(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                            cudaStream_t s);
cudaError_t launch_gemm_swiglu(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gemm_scatter(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s);

// One launch of gemm_grouped_kernel<mode> (kGrpSwiglu or kGrpPlain):
// tok = token rows (64-row boxes), w0/w1 = weight rows (128-row boxes).
cudaError_t launch_gemm_grouped(int mode, const CUtensorMap& tok, const CUtensorMap& w0,
                                const CUtensorMap& w1, const GroupedArgs& a, int grid,
                                cudaStream_t s);

// Rewrite W [rows, K] (rows % 128 == 0, K % kGBK == 0) as contiguous
// 128 x kGBK tiles, tile index (row / 128) * (K / kGBK) + k / kGBK.
cudaError_t launch_pack_tiles(const __nv_bfloat16* src, __nv_bfloat16* dst, long long rows, int K,
                              int sms, cudaStream_t s);

// Router GEMM fused with softmax and stable top-k: logits [T,E] fp32 (+bias),
// idx [T,k], gates [T,k]; x map in 128-row boxes, W_r map in 256-row boxes.
cudaError_t launch_router_topk(const CUtensorMap& x, const CUtensorMap& w, RouterArgs a, int sms,
                               cudaStream_t s);

// Softmax over E and stable top-k per token: idx [T,k] int32, gates [T,k].
// With sel_bias, the choice ranks logits + bias; gates stay unbiased.
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renorm,
                              const float* sel_bias, int* idx, float* gates, cudaStream_t s);

// prob_sum[e] = sum_t softmax(logits_t)_e, deterministic. Scratch: partial
// [ceil(T / kLblTokens), E] floats. Two launches.
constexpr int kLblTokens = 256;
cudaError_t launch_lbl_prob_sum(const float* logits, int T, int E, float* partial, float* out,
                                cudaStream_t s);

// Router replay: gates[t,j] = softmax(logits[t])[idx[t,j]] (0 for ids outside
// [0, E)), divided by their sum with renorm.
cudaError_t launch_replay_gates(const float* logits, int T, int E, const int* idx, int k,
                                int renorm, float* gates, cudaStream_t s);

// Counting sort of the T*k slots by expert. Scratch: cnt and cbase, each
// sort_scratch_ints(S, E) ints. Three launches.
constexpr int kSortChunk = 1024;
inline long long sort_scratch_ints(long long S, long long E) {
  return ((S + kSortChunk - 1) / kSortChunk) * E;
}
cudaError_t launch_sort(const int* idx, int S, int k, int E, int* cnt, int* cbase, int* counts,
                        int* offsets, int* perm, int* pos, unsigned* status, cudaStream_t s);
constexpr int kSortLaunches = 3;

// c[t] = sum_j gates[t,j] * o[pos[t,j]] in fp32, j order; bf16 out.
cudaError_t launch_combine(const __nv_bfloat16* o, const float* gates, const int* pos, int T,
                           int k, int l, __nv_bfloat16* c, cudaStream_t s);

}  // namespace lmoe
