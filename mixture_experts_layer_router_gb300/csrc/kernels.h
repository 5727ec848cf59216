// Host-side launchers of the library's kernels (internal interface).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <string.h>

#include "gemm.cuh"
#include "gemm_grouped.cuh"
#include "router.cuh"

namespace lmoe {

// Kernel attributes (the dynamic shared-memory limit) and occupancy answers
// belong to a device: launchers keep one "done" flag per device ordinal.
// Setting an attribute twice from racing threads is harmless.
constexpr int kMaxDevices = 64;
inline int current_device_index() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

// Programmatic dependent launch for the kernels this host thread enqueues
// while a PdlScope with `on` is alive (the forward's launch sequence); every
// kernel calls pdl_wait() before reading what earlier kernels wrote.
inline bool& pdl_flag() {
  thread_local bool on = false;
  return on;
}
struct PdlScope {
  bool prev;
  explicit PdlScope(bool on) : prev(pdl_flag()) { pdl_flag() = on; }
  ~PdlScope() { pdl_flag() = prev; }
};

// One launch through cudaLaunchKernelEx: `cluster` CTAs per cluster (1: no
// cluster), with the programmatic-serialization attribute when pdl_flag() is
// set, and cooperative (every CTA resident at once) when `cooperative`.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, int cluster, bool cooperative, Args... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute at[3];
  unsigned n = 0;
  if (cluster > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl_flag()) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cooperative) {
    at[n].id = cudaLaunchAttributeCooperative;
    at[n].val.cooperative = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct GemmMaps {
  CUtensorMap a, b, bu, a2, b2;
};

// One launch of gemm_tc_kernel<MODE, DUAL, F8>; `grid` persistent CTAs.
// f8: E4M3 operands (a_scale, b_scale set; not with dual). pair_sms > 0 (dense
// GEMMs only): the SM-pair kernel instead, on up to pair_sms / 2 clusters of
// two CTAs (fewer if fewer are resident at once or there are fewer tiles).
cudaError_t launch_gemm_bf16(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                             cudaStream_t s, bool f8 = false, int pair_sms = 0);
cudaError_t launch_gemm_f32(const GemmMaps& m, const GemmArgs& a, int grid, bool dual,
                            cudaStream_t s, bool f8 = false, int pair_sms = 0);
// SwiGLU epilogue; with f8 the output is E4M3 codes (out_scale, out_amax,
// b_scale2 set).
cudaError_t launch_gemm_swiglu(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s,
                               bool f8 = false, int pair_sms = 0);
cudaError_t launch_gemm_scatter(const GemmMaps& m, const GemmArgs& a, int grid, cudaStream_t s,
                                int pair_sms = 0);
// kEpiScatterF8: the scatter with E4M3 output (out_scale, out_amax set).
cudaError_t launch_gemm_scatter_f8(const GemmMaps& m, const GemmArgs& a, int grid,
                                   cudaStream_t s, bool f8 = false, int pair_sms = 0);

// One launch of gemm_grouped_kernel<mode, f8> (kGrpSwiglu or kGrpPlain;
// bf16 or E4M3 operands): tok = token rows (64-row boxes), w0/w1 = packed
// weight tiles.
cudaError_t launch_gemm_grouped(int mode, bool f8, const CUtensorMap& tok, const CUtensorMap& w0,
                                const CUtensorMap& w1, const GroupedArgs& a, int grid,
                                cudaStream_t s);

// The same GEMMs on SM pairs (clusters of 2, tcgen05 cta_group::2):
// a.fblocks counts pair feature blocks (SwiGLU: F / 256; plain: l / 512).
// Needs F % 256 == 0 (SwiGLU) or l % 512 == 0 (plain). Grid: as many pairs
// as can be resident at once, at most sms / 2.
cudaError_t launch_gemm_grouped_pair(int mode, bool f8, const CUtensorMap& tok,
                                     const CUtensorMap& w0, const CUtensorMap& w1,
                                     const GroupedArgs& a, int sms, cudaStream_t s);

// Both expert GEMMs in one launch (gemm_fused.cuh): z, W_g, W_u (packed) ->
// h -> W_d (packed) -> o, with a.gu and a.dn set as for the two pair launches
// above (seg_offsets form only). Needs F % 256 == 0 and l % 512 == 0.
// a.dep ([E * F / 256]) and a.tile_counter ([2]) are zero at launch and are
// left zero. As many pairs as can be resident at once.
struct FusedExpertArgs;
cudaError_t launch_expert_fused(bool f8, const CUtensorMap& z, const CUtensorMap& wg,
                                const CUtensorMap& wu, const CUtensorMap& h,
                                const CUtensorMap& wd, const FusedExpertArgs& a, int sms,
                                cudaStream_t s);

// Rewrite a row-major matrix of `rows` rows of `row_bytes` bytes (rows % 128
// == 0, row_bytes % 128 == 0) as contiguous tiles of 128 rows x 128 bytes,
// tile index (row / 128) * (row_bytes / 128) + byte / 128: kGBK bf16 or
// kGBK8 E4M3 columns per tile.
cudaError_t launch_pack_tiles(const void* src, void* dst, long long rows, long long row_bytes,
                              int sms, cudaStream_t s);

// Per-group absolute maximum of bf16 W [groups, rows, cols] (float bits,
// accumulated with atomicMax into amax_bits[groups], which the caller
// zeroes), then scale[g] = amax / 448 (1 for an all-zero group).
cudaError_t launch_absmax_groups(const __nv_bfloat16* src, long long groups, long long group_elems,
                                 unsigned* amax_bits, int sms, cudaStream_t s);
cudaError_t launch_scales_from_amax(const unsigned* amax_bits, int n, float* scale,
                                    cudaStream_t s);

// E4M3 codes of bf16 W [groups * rows_per_group, K] with the group's scale,
// written either row-major (packed = false) or as the 128 x 128-byte tiles
// of launch_pack_tiles (packed = true; rows_per_group % 128 == 0, K % 128 == 0).
cudaError_t launch_quantize_e4m3(const __nv_bfloat16* src, uint8_t* dst, long long rows,
                                 long long K, long long rows_per_group, const float* scale,
                                 bool packed, int sms, cudaStream_t s);

// Delayed scaling of n activation tensors (n <= kFp8Tensors): enter this
// forward's maxima into the 1024-step history, form the next scales, clear
// the maxima. One launch of one block.
constexpr int kFp8Tensors = 8;
constexpr int kFp8History = 1024;
struct Fp8State {
  float scale[kFp8Tensors];      // scales the next forward quantizes with
  unsigned amax[kFp8Tensors];    // maxima being recorded by this forward (float bits)
  float last_amax[kFp8Tensors];  // maxima of the last finished forward
  long long steps;               // forwards entered so far
  float hist[kFp8Tensors][kFp8History];
};
cudaError_t launch_fp8_update(Fp8State* st, int n, cudaStream_t s);

// Router GEMM fused with softmax and stable top-k: logits [T,E] fp32 (+bias),
// idx [T,k], gates [T,k]; x map in 128-row boxes, W_r map in boxes of
// router_w_box_rows(E) rows.
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
// The same sort in one cooperative launch (kSortChunk slots per CTA, every
// CTA resident at once): sort_fused_fits says whether the device holds the
// ceil(S / kSortChunk) CTAs at once. sync: two counters, zero before the
// first launch; every launch leaves them at zero again.
bool sort_fused_fits(int S, int E);
// The same sort in one CTA of 1024 threads (no grid barrier), for at most
// kBlockSortMaxSlots slots and E <= kMaxGroups; counts, offsets, perm, pos as
// above (cnt and cbase are not used).
constexpr int kBlockSortMaxSlots = 4096;
cudaError_t launch_sort_block(const int* idx, int S, int k, int E, int* counts, int* offsets,
                              int* perm, int* pos, unsigned* status, cudaStream_t s);
cudaError_t launch_sort_fused(const int* idx, int S, int k, int E, int* cnt, int* cbase,
                              int* counts, int* offsets, int* perm, int* pos, unsigned* status,
                              unsigned* sync, cudaStream_t s);

// Multi-round fixed-capacity schedule (capacity C per expert per round,
// groups of G consecutive experts, at most max_rounds rounds): per round r,
// rlen[r*E+e] slots of expert e starting at row rin[r*E+e] of the
// expert-sorted slots, placed at row rout[r*(E+1)+e] of the round buffer
// (rout[r*(E+1)+E] = the round's total); info = {rounds used, slots left
// over}. Slots left over set kStatusRounds. One launch of one block.
cudaError_t launch_round_schedule(const int* counts, const int* offsets, int E, int C, int G,
                                  int max_rounds, int* rin, int* rout, int* rlen, int* info,
                                  unsigned* status, cudaStream_t s);

// c[t] = sum_j gates[t,j] * o[pos[t,j]] in fp32, j order; bf16 out. o has
// o_rows rows (checked in the bounds-checked build, which reports to status).
cudaError_t launch_combine(const __nv_bfloat16* o, const float* gates, const int* pos, int T,
                           int k, int l, __nv_bfloat16* c, long long o_rows, unsigned* status,
                           cudaStream_t s);
// The same from fp32 o, with c written as E4M3 codes with *scale and max |c|
// into *amax.
cudaError_t launch_combine_f8(const float* o, const float* gates, const int* pos, int T, int k,
                              int l, uint8_t* c, const float* scale, unsigned* amax,
                              long long o_rows, unsigned* status, cudaStream_t s);
// E4M3 codes of bf16 src [n] (n % 16 == 0) with *scale; max |src| into *amax.
cudaError_t launch_quantize_act(const __nv_bfloat16* src, uint8_t* dst, long long n,
                                const float* scale, unsigned* amax, int sms, cudaStream_t s);

}  // namespace lmoe
