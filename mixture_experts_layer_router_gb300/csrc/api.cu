// C ABI of the LatentMoE layer forward (declared in include/latentmoe.h).
//
// Host code only: validation, workspace, TMA descriptors and the launch
// sequence. All arithmetic of the layer runs in the kernels of this library.
//
// Launch sequence of latentmoe_forward, all on the caller's stream with no
// host synchronisation (token counts per expert stay on the device, as in
// "Frontier Pre-training at Microsoft AI", section "Reducing per-expert
// overhead"):
//   0 router          logits = x W_r^T (+ b), softmax, stable tcgen05, fused
//                     top-k, gates                           epilogue
//   1 replay_gates    (router replay without gates only)
//   2 sort            counts, offsets, perm, pos             3 small kernels
//   3 down_proj       z = x W_dn^T, written to the k slots   tcgen05, scatter
//   4 expert_gate_up  h = SiLU(z W_g^T) * (z W_u^T)          tcgen05, grouped
//   5 expert_down     o = h W_d^T                            tcgen05, grouped
//   6 combine         c[t] = sum_j g[t,j] o[pos[t,j]]        gather, fp32
//   7 shared_gate_up  s = SiLU(x W_gs^T) * (x W_us^T)        tcgen05 (F_s > 0)
//   8 up_proj         y = c W_up^T (+ s W_ds^T)              tcgen05, dual-K
//   9 fp8_scales      (E4M3 experts only) delayed-scaling update of the
//                     scales of z and h                      1 small kernel
//
// With LATENTMOE_FP8_EXPERTS the expert GEMMs (4, 5) take E4M3 operands:
// down_proj writes z as E4M3 codes, expert_gate_up writes h as E4M3 codes,
// and both record their maxima for the scale update.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gemm_fused.cuh"
#include "kernels.h"
#include "latentmoe.h"

using lmoe::GemmArgs;
using lmoe::GemmMaps;

namespace {

constexpr int kNumStages = 10;
const char* const kStageNames[kNumStages] = {
    "router",      "replay_gates", "sort",           "down_proj", "expert_gate_up",
    "expert_down", "combine",      "shared_gate_up", "up_proj",   "fp8_scales"};
// scaled activations: 0 = z, 1 = h (expert GEMMs), 2 = x, 3 = c, 4 = the
// shared expert's hidden (dense GEMMs)
constexpr int kFp8Acts = LATENTMOE_FP8_TENSORS;
constexpr int kDenseW = 5;  // E4M3 dense weights: W_dn, W_up, W_gs, W_us, W_ds

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (row stride `ld` elements) read in boxes of
// 64 columns x box_rows rows with 128-byte swizzle; out-of-range reads are 0.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
              uint32_t box_rows, uint32_t box_cols = 64) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || ptr == nullptr || rows == 0 || cols == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor (E4M3 codes) [rows, cols] read in boxes of 128 columns x
// box_rows rows with 128-byte swizzle.
bool make_map_u8(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                 uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || ptr == nullptr || rows == 0 || cols == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token rows for the grouped kernel: boxes of kGTokBox rows x 128 bytes
// (kGBK bf16 or kGBK8 E4M3 columns).
bool make_token_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                    bool f8 = false) {
  if (f8) return make_map_u8(map, ptr, rows, cols, cols, lmoe::kGTokBox);
  return make_map(map, ptr, rows, cols, cols, lmoe::kGTokBox, lmoe::kGBK);
}

// Packed weight tiles (see pack.cu): `tiles` contiguous blocks of 128 rows x
// 128 bytes, read one whole tile per box with the grouped kernel's swizzle.
bool make_tile_map(CUtensorMap* map, const void* ptr, uint64_t tiles, bool f8 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || ptr == nullptr || tiles == 0) return false;
  const cuuint64_t cols = f8 ? lmoe::kGBK8 : lmoe::kGBK;
  const cuuint64_t dims[3] = {cols, 128, tiles};
  const cuuint64_t strides[2] = {128, 128 * 128};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(cols), 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// SM count of the current device (looked up once per device).
int num_sms() {
  static int n_of[lmoe::kMaxDevices] = {};
  const int dev = lmoe::current_device_index();
  if (dev < 0) return 1;
  if (n_of[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    n_of[dev] = n > 0 ? n : 1;
  }
  return n_of[dev];
}

}  // namespace

struct latentmoe {
  latentmoe_dims dims;
  int k = 0;
  uint32_t flags = 0;
  int device = 0;
  int sms = 1;
  bool loaded = false;
  bool fp8 = false;             // E4M3 expert GEMMs
  bool fp8_dense = false;       // E4M3 latent projections and shared expert
  float* dw_scale = nullptr;    // [kDenseW] scales of the E4M3 dense weights (in wmem)
  uint8_t* x8 = nullptr;        // [T, d] E4M3 codes of x
  float* y32 = nullptr;         // [T, d] fp32 partial of the E4M3 up-projection (shared expert)
  bool sm_pairs = true;         // SM-pair grouped kernels where the shapes allow
  // multi-round fixed-capacity expert schedule (capacity 0: one dropless pass)
  int64_t cap = 0;
  int cap_group = 0;
  int cap_rounds = 0;
  void* cap_mem = nullptr;      // round buffer of h, then the schedule arrays
  void* hround = nullptr;       // [E * cap, F] bf16 or E4M3 codes
  int* rin = nullptr;           // [cap_rounds, E]
  int* rout = nullptr;          // [cap_rounds, E + 1]
  int* rlen = nullptr;          // [cap_rounds, E]
  int* rinfo = nullptr;         // {rounds used, slots left over}
  latentmoe_weights w;          // the library-owned copies below
  float* w_scale = nullptr;     // E4M3: [3E] scales of W_g, W_u, W_d per expert (in wmem)
  lmoe::Fp8State* f8 = nullptr; // E4M3: delayed-scaling state (in ws)
  void* wmem = nullptr;          // one allocation holding every weight copy
  GemmMaps m_down, m_shared, m_up;  // dense GEMM maps (every box 128 rows)
  CUtensorMap m_wg, m_wu, m_wd;  // packed expert weights (grouped kernel)
  CUtensorMap m_wr;              // router weights in router_box_cols(E)-column boxes (router kernel)
  // workspace
  void* ws = nullptr;
  float* logits = nullptr;
  int* idx = nullptr;
  float* gates = nullptr;
  int* cnt = nullptr;
  int* cbase = nullptr;
  int* counts = nullptr;
  float* lbl_partial = nullptr;
  int* offsets = nullptr;
  int* perm = nullptr;
  int* pos = nullptr;
  __nv_bfloat16* zp = nullptr;
  __nv_bfloat16* hb = nullptr;
  __nv_bfloat16* ob = nullptr;
  __nv_bfloat16* cb = nullptr;
  __nv_bfloat16* sh = nullptr;
  unsigned* status = nullptr;
  // {tile counter, exit count} of the SM-pair down GEMM, then the fused
  // sort's {barrier arrivals, exits}: zero at create, and every launch leaves
  // them zero (a wait that gave up may not: latentmoe_get_status clears them)
  int* tile_counter = nullptr;
  unsigned* sort_sync = nullptr;
  // both expert GEMMs in one launch (SM pairs, one pass): 0 never, 1 where the
  // shapes allow, 2 (default) where they allow and the layer is small (see
  // experts_fused); dep: the gate+up tiles done per (expert, feature block
  // of 256), zero between launches
  int fuse_experts = 2;
  int* dep = nullptr;  // [E * F / 256], null where the shapes do not allow the fused kernel
  bool pdl = true;              // programmatic dependent launch between the forward's kernels
  int64_t last_T = 0;
  // host-buffer forward staging
  void* x_stage = nullptr;
  void* y_stage = nullptr;
  // pipelined host-buffer forward: two staging slots, a stream for the
  // copies in and one for the copies out, and per slot the events that order
  // them with the forwards (created on the first call)
  void* xs[2] = {nullptr, nullptr};
  void* ys[2] = {nullptr, nullptr};
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t ev_in[2] = {nullptr, nullptr};   // slot's x copied in
  cudaEvent_t ev_fwd[2] = {nullptr, nullptr};  // slot's forward done (x read, y written)
  cudaEvent_t ev_out[2] = {nullptr, nullptr};  // slot's y copied out
  int64_t host_steps = 0;
  // profiling
  std::vector<cudaEvent_t> events;
  int prof_slots = 0;
  int64_t forwards = 0;
  int64_t launches = 0;
  int last_cuda = 0;
};

namespace {

int fail_cuda(latentmoe* h, cudaError_t e) {
  if (h != nullptr) h->last_cuda = static_cast<int>(e);
  return e == cudaErrorMemoryAllocation ? LATENTMOE_ERR_OUT_OF_MEMORY : LATENTMOE_ERR_CUDA;
}

#define LMOE_CK(h, call)                          \
  do {                                            \
    const cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return fail_cuda(h, e_); \
  } while (0)

GemmArgs base_args(const latentmoe* h) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.group_m = 16;
  a.status = h->status;
  return a;
}

int dense_grid(const latentmoe* h, int M, int n_tiles) {
  const long long tiles = static_cast<long long>((M + lmoe::kBM - 1) / lmoe::kBM) * n_tiles;
  return static_cast<int>(tiles < h->sms ? tiles : h->sms);
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// SMs offered to the SM-pair dense GEMM kernel (0: the one-SM kernel).
int dense_pair_sms(const latentmoe* h) { return h->sm_pairs ? h->sms : 0; }

void record(latentmoe* h, int slot_base, int i, cudaStream_t s) {
  if (h->prof_slots > 0) cudaEventRecord(h->events[slot_base + i], s);
}

// NVTX ranges named after the forward's stages ("latentmoe:router", ...), so
// that a profiler's timeline shows which stage enqueued which kernels. next(i)
// closes the open range and opens stage i's (i = kNumStages opens none); the
// destructor closes a range left open by an early error return. Without a
// profiler attached the NVTX calls do nothing.
class NvtxStages {
 public:
  void next(int i) {
    if (open_) nvtxRangePop();
    open_ = false;
    if (i < kNumStages) {
      char name[48];
      snprintf(name, sizeof(name), "latentmoe:%s", kStageNames[i]);
      nvtxRangePushA(name);
      open_ = true;
    }
  }
  ~NvtxStages() {
    if (open_) nvtxRangePop();
  }

 private:
  bool open_ = false;
};

// Counting sort of the workspace idx into counts, offsets, perm, pos.
int run_sort(latentmoe* h, int T, cudaStream_t s) {
  const int E = static_cast<int>(h->dims.num_experts);
  const int S = T * h->k;
  if (S <= lmoe::kBlockSortMaxSlots) {
    // one CTA
    LMOE_CK(h, lmoe::launch_sort_block(h->idx, S, h->k, E, h->counts, h->offsets, h->perm,
                                       h->pos, h->status, s));
    h->launches += 1;
    return LATENTMOE_OK;
  }
  if (lmoe::sort_fused_fits(S, E)) {
    // one cooperative launch
    LMOE_CK(h, lmoe::launch_sort_fused(h->idx, S, h->k, E, h->cnt, h->cbase, h->counts,
                                       h->offsets, h->perm, h->pos, h->status, h->sort_sync, s));
    h->launches += 1;
    return LATENTMOE_OK;
  }
  LMOE_CK(h, lmoe::launch_sort(h->idx, T * h->k, h->k, E, h->cnt, h->cbase, h->counts,
                               h->offsets, h->perm, h->pos, h->status, s));
  h->launches += lmoe::kSortLaunches;
  return LATENTMOE_OK;
}

// Routing half shared by forward and route_from_logits: logits -> idx,
// gates -> counts, offsets, perm, pos (workspace buffers).
int run_routing(latentmoe* h, const float* logits, int T, cudaStream_t s, int slot_base) {
  const int E = static_cast<int>(h->dims.num_experts);
  const float* sel_bias = (h->flags & LATENTMOE_SELECT_BIAS) ? h->w.b_r : nullptr;
  LMOE_CK(h, lmoe::launch_route_topk(logits, T, E, h->k, (h->flags & LATENTMOE_RENORM) ? 1 : 0,
                                     sel_bias, h->idx, h->gates, s));
  h->launches += 1;
  record(h, slot_base, 2, s);
  const int r = run_sort(h, T, s);
  if (r != LATENTMOE_OK) return r;
  record(h, slot_base, 3, s);
  return LATENTMOE_OK;
}

// The arguments of the gate+up GEMM (one-SM form: fblocks = F / 128).
void gate_up_args(latentmoe* h, lmoe::GroupedArgs& a) {
  const int E = static_cast<int>(h->dims.num_experts);
  const int l = static_cast<int>(h->dims.latent), F = static_cast<int>(h->dims.ffn);
  a.num_groups = E;
  a.fblocks = F / 128;
  a.kb = l / (h->fp8 ? lmoe::kGBK8 : lmoe::kGBK);
  a.w_group_rows = F;
  a.n_out = F;
  a.ldo = F;
  a.status = h->status;
  if (a.out_rows == 0) a.out_rows = h->dims.max_tokens * h->k;
  if (h->fp8) {
    a.w_scale0 = h->w_scale;
    a.w_scale1 = h->w_scale + E;
    a.in_scale = &h->f8->scale[0];
    a.out_scale = &h->f8->scale[1];
    a.out_amax = &h->f8->amax[1];
  }
}

// One launch of the grouped gate+up GEMM over the groups described in `a`
// (segments and output set by the caller): weights, scales and the kernel
// (SM pairs where F % 256 == 0) from the handle.
int launch_expert_gate_up(latentmoe* h, lmoe::GroupedArgs a, const CUtensorMap& tok,
                          cudaStream_t s) {
  const int F = static_cast<int>(h->dims.ffn);
  gate_up_args(h, a);
  if (h->sm_pairs && F % 256 == 0) {
    a.fblocks = F / 256;
    LMOE_CK(h, lmoe::launch_gemm_grouped_pair(lmoe::kGrpSwiglu, h->fp8, tok, h->m_wg, h->m_wu, a,
                                              h->sms, s));
  } else {
    LMOE_CK(h, lmoe::launch_gemm_grouped(lmoe::kGrpSwiglu, h->fp8, tok, h->m_wg, h->m_wu, a,
                                         h->sms, s));
  }
  h->launches += 1;
  return LATENTMOE_OK;
}

// The arguments of the down GEMM (one-SM form: fblocks = ceil(l / 256)).
void down_args(latentmoe* h, lmoe::GroupedArgs& a) {
  const int E = static_cast<int>(h->dims.num_experts);
  const int l = static_cast<int>(h->dims.latent), F = static_cast<int>(h->dims.ffn);
  a.num_groups = E;
  a.fblocks = ceil_div(l, 256);
  a.kb = F / (h->fp8 ? lmoe::kGBK8 : lmoe::kGBK);
  a.w_group_rows = l;
  a.n_out = l;
  a.ldo = l;
  a.status = h->status;
  if (a.out_rows == 0) a.out_rows = h->dims.max_tokens * h->k;
  a.w_scale0 = a.w_scale1 = a.in_scale = a.out_scale = nullptr;
  a.out_amax = nullptr;
  a.out_f32 = h->fp8_dense ? 1 : 0;
  if (h->fp8) {
    a.w_scale0 = a.w_scale1 = h->w_scale + 2 * E;
    a.in_scale = &h->f8->scale[1];
  }
}

// The same for the grouped down GEMM (SM pairs where l % 512 == 0).
int launch_expert_down(latentmoe* h, lmoe::GroupedArgs a, const CUtensorMap& tok, cudaStream_t s) {
  const int l = static_cast<int>(h->dims.latent);
  down_args(h, a);
  if (h->sm_pairs && l % 512 == 0) {
    a.fblocks = l / 512;
    // few long tiles per pair: dynamic tile order balances the last wave
    a.tile_counter = h->tile_counter;
    LMOE_CK(h, lmoe::launch_gemm_grouped_pair(lmoe::kGrpPlain, h->fp8, tok, h->m_wd, h->m_wd, a,
                                              h->sms, s));
  } else {
    LMOE_CK(h, lmoe::launch_gemm_grouped(lmoe::kGrpPlain, h->fp8, tok, h->m_wd, h->m_wd, a,
                                         h->sms, s));
  }
  h->launches += 1;
  return LATENTMOE_OK;
}

// Whether the one-pass forward of T tokens runs both expert GEMMs as one
// launch. Automatic mode: when each SM pair has at most 400 k-blocks of work
// in the two GEMMs (expected from E, l, F and T k: E * F/256 * c gate+up
// tiles of l/BK k-blocks and E * l/512 * c down tiles of F/BK, c = the token
// chunks of an expert of T k / E slots), the second launch's tail is a large
// part of the layer and the fused launch takes it in (measured 1-5% faster
// on the expert GEMMs of T = 4096, E = 64, l = 1024, F = 2048: about 160
// k-blocks per pair). With more work per pair (the MAI-Base shapes, and 1/16
// of MAI-Base-1 at about 1200) the interleaved order read 3% more from DRAM
// and measured 1.5-4.5% slower, so the two launches run.
bool experts_fused(const latentmoe* h, int64_t T) {
  if (h->fuse_experts == 0 || !h->sm_pairs || h->dep == nullptr || h->cap > 0) return false;
  if (h->fuse_experts == 1) return true;
  const int64_t E = h->dims.num_experts, S = T * h->k;
  const int64_t l = h->dims.latent, F = h->dims.ffn;
  const int64_t bk = h->fp8 ? lmoe::kGBK8 : lmoe::kGBK;
  const int64_t chunks = S > 256 * E ? (S + 256 * E - 1) / (256 * E) : 1;
  const int64_t kblocks = E * chunks * ((F / 256) * (l / bk) + (l / 512) * (F / bk));
  return kblocks <= 400 * static_cast<int64_t>(h->sms / 2);
}

// Both expert GEMMs in one launch over the expert segments (h->offsets):
// z (map mzp) -> h (hb, map mh) -> o (ob).
int launch_experts_fused(latentmoe* h, const CUtensorMap& mzp, const CUtensorMap& mh,
                         cudaStream_t s) {
  const int E = static_cast<int>(h->dims.num_experts);
  const int l = static_cast<int>(h->dims.latent), F = static_cast<int>(h->dims.ffn);
  lmoe::FusedExpertArgs f;
  memset(&f, 0, sizeof(f));
  f.gu.seg_offsets = h->offsets;
  f.gu.out = h->hb;
  gate_up_args(h, f.gu);
  f.gu.fblocks = F / 256;
  f.dn.seg_offsets = h->offsets;
  f.dn.out = h->ob;
  down_args(h, f.dn);
  f.dn.fblocks = l / 512;
  f.dep = h->dep;
  f.tile_counter = h->tile_counter;
  // the down tiles of an expert come about 1.5 waves of pair tiles (F / 256
  // gate+up tiles per expert of up to 256 slots) after its gate+up tiles
  const int npairs = h->sms / 2;
  const int per = F / 256;
  const int lag = (3 * npairs + 2 * per - 1) / (2 * per);
  f.lag = lag < 1 ? 1 : (lag > E ? E : lag);
  LMOE_CK(h, lmoe::launch_expert_fused(h->fp8, mzp, h->m_wg, h->m_wu, mh, h->m_wd, f, h->sms,
                                       s));
  h->launches += 1;
  return LATENTMOE_OK;
}

// Both expert GEMMs under the multi-round fixed-capacity schedule: the
// schedule kernel, then per round r the gate+up of the round's slots (rows
// rin of the expert-sorted z) into the round buffer (rows rout) and the down
// GEMM from the round buffer back to the slots' rows of o. Rounds past the
// ones the routing needs have no slots and end at once.
int run_expert_rounds(latentmoe* h, const CUtensorMap& mzp, cudaStream_t s) {
  const int E = static_cast<int>(h->dims.num_experts);
  const int F = static_cast<int>(h->dims.ffn);
  LMOE_CK(h, lmoe::launch_round_schedule(h->counts, h->offsets, E, static_cast<int>(h->cap),
                                         h->cap_group, h->cap_rounds, h->rin, h->rout, h->rlen,
                                         h->rinfo, h->status, s));
  h->launches += 1;
  CUtensorMap mhr;
  if (!make_token_map(&mhr, h->hround, static_cast<uint64_t>(E) * h->cap, F, h->fp8))
    return LATENTMOE_ERR_CUDA;
  for (int r = 0; r < h->cap_rounds; ++r) {
    lmoe::GroupedArgs a;
    memset(&a, 0, sizeof(a));
    a.seg_len = h->rlen + r * E;
    a.in_start = h->rin + r * E;
    a.out_start = h->rout + r * (E + 1);
    a.out = h->hround;
    a.out_rows = h->dims.num_experts * h->cap;
    int rc = launch_expert_gate_up(h, a, mzp, s);
    if (rc != LATENTMOE_OK) return rc;
    lmoe::GroupedArgs b;
    memset(&b, 0, sizeof(b));
    b.seg_len = h->rlen + r * E;
    b.in_start = h->rout + r * (E + 1);
    b.out_start = h->rin + r * E;
    b.out = h->ob;
    rc = launch_expert_down(h, b, mhr, s);
    if (rc != LATENTMOE_OK) return rc;
  }
  return LATENTMOE_OK;
}

}  // namespace

extern "C" {

int latentmoe_num_stages(void) { return kNumStages; }

const char* latentmoe_stage_name(int stage) {
  return (stage >= 0 && stage < kNumStages) ? kStageNames[stage] : nullptr;
}

const char* latentmoe_strerror(int code) {
  switch (code) {
    case LATENTMOE_OK: return "ok";
    case LATENTMOE_ERR_INVALID_ARG: return "invalid argument";
    case LATENTMOE_ERR_UNSUPPORTED: return "unsupported dimensions, flags or alignment";
    case LATENTMOE_ERR_NOT_LOADED: return "weights not loaded";
    case LATENTMOE_ERR_CUDA: return "CUDA error";
    case LATENTMOE_ERR_TIMEOUT: return "a bounded device wait timed out";
    case LATENTMOE_ERR_DEVICE_STATUS: return "a kernel flagged invalid data";
    case LATENTMOE_ERR_OUT_OF_MEMORY: return "out of device memory";
    default: return "unknown error";
  }
}

int latentmoe_create(const latentmoe_dims* dims, int top_k, uint32_t flags, latentmoe_t* out) {
  if (out == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (dims == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  const latentmoe_dims d = *dims;
  if (flags & ~static_cast<uint32_t>(LATENTMOE_RENORM | LATENTMOE_ROUTER_BIAS |
                                     LATENTMOE_OUT_FP32 | LATENTMOE_SELECT_BIAS |
                                     LATENTMOE_FP8_EXPERTS | LATENTMOE_FP8_DENSE))
    return LATENTMOE_ERR_INVALID_ARG;
  if ((flags & LATENTMOE_FP8_DENSE) && !(flags & LATENTMOE_FP8_EXPERTS))
    return LATENTMOE_ERR_INVALID_ARG;
  if ((flags & LATENTMOE_ROUTER_BIAS) && (flags & LATENTMOE_SELECT_BIAS))
    return LATENTMOE_ERR_INVALID_ARG;
  if (d.num_experts < 1 || d.max_tokens < 1 || d.hidden < 1 || d.latent < 1 || d.ffn < 1 ||
      d.shared_ffn < 0)
    return LATENTMOE_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > 16 || top_k > d.num_experts) return LATENTMOE_ERR_INVALID_ARG;
  if (d.num_experts > lmoe::kMaxGroups) return LATENTMOE_ERR_UNSUPPORTED;
  if (d.hidden % 128 || d.latent % 128 || d.ffn % 128 || d.shared_ffn % 128)
    return LATENTMOE_ERR_UNSUPPORTED;
  const long long S = d.max_tokens * top_k;
  if (S > (1ll << 30) || d.hidden > (1 << 20) || d.latent > (1 << 20) || d.ffn > (1 << 20) ||
      d.shared_ffn > (1 << 20))
    return LATENTMOE_ERR_UNSUPPORTED;
  // rows of the stacked expert weights are addressed with int32 TMA coordinates
  if (d.num_experts * d.ffn >= (1ll << 31) || d.num_experts * d.latent >= (1ll << 31))
    return LATENTMOE_ERR_UNSUPPORTED;

  latentmoe* h = new (std::nothrow) latentmoe();
  if (h == nullptr) return LATENTMOE_ERR_OUT_OF_MEMORY;
  h->dims = d;
  h->k = top_k;
  h->flags = flags;
  h->fp8 = (flags & LATENTMOE_FP8_EXPERTS) != 0;
  h->fp8_dense = (flags & LATENTMOE_FP8_DENSE) != 0;
  memset(&h->w, 0, sizeof(h->w));
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) {
    delete h;
    return LATENTMOE_ERR_CUDA;
  }
  h->sms = num_sms();

  const long long T = d.max_tokens, E = d.num_experts, l = d.latent, F = d.ffn;
  const long long Fs = d.shared_ffn;
  const long long nb_ints = lmoe::sort_scratch_ints(S, E);
  const size_t al = 1024;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, al);
    return o;
  };
  const size_t o_logits = take(T * E * 4);
  const size_t o_idx = take(S * 4), o_gates = take(S * 4), o_perm = take(S * 4),
               o_pos = take(S * 4);
  const size_t o_cnt = take(nb_ints * 4), o_cbase = take(nb_ints * 4);
  const size_t o_counts = take(E * 4), o_offsets = take((E + 1) * 4);
  const size_t o_lbl = take(((T + lmoe::kLblTokens - 1) / lmoe::kLblTokens) * E * 4);
  // o is kept in fp32 when it feeds the E4M3 up-projection
  const size_t o_zp = take(S * l * 2), o_h = take(S * F * 2);
  const size_t o_o = take(S * l * ((flags & LATENTMOE_FP8_DENSE) ? 4 : 2));
  const size_t o_c = take(T * l * 2), o_sh = take(Fs > 0 ? T * Fs * 2 : 16);
  const size_t o_status = take(16);
  const size_t o_tcount = take(16);
  const bool fusable = F % 256 == 0 && l % 512 == 0;
  const size_t o_dep = take(fusable ? E * (F / 256) * 4 : 16);
  const size_t o_f8 = take(sizeof(lmoe::Fp8State));
  const size_t o_x8 = take(h->fp8_dense ? T * d.hidden : 16);
  const size_t o_y32 = take(h->fp8_dense && Fs > 0 ? T * d.hidden * 4 : 16);
  e = cudaMalloc(&h->ws, off);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return e == cudaErrorMemoryAllocation ? LATENTMOE_ERR_OUT_OF_MEMORY : LATENTMOE_ERR_CUDA;
  }
  char* base = static_cast<char*>(h->ws);
  h->logits = reinterpret_cast<float*>(base + o_logits);
  h->idx = reinterpret_cast<int*>(base + o_idx);
  h->gates = reinterpret_cast<float*>(base + o_gates);
  h->perm = reinterpret_cast<int*>(base + o_perm);
  h->pos = reinterpret_cast<int*>(base + o_pos);
  h->cnt = reinterpret_cast<int*>(base + o_cnt);
  h->cbase = reinterpret_cast<int*>(base + o_cbase);
  h->counts = reinterpret_cast<int*>(base + o_counts);
  h->lbl_partial = reinterpret_cast<float*>(base + o_lbl);
  h->offsets = reinterpret_cast<int*>(base + o_offsets);
  h->zp = reinterpret_cast<__nv_bfloat16*>(base + o_zp);
  h->hb = reinterpret_cast<__nv_bfloat16*>(base + o_h);
  h->ob = reinterpret_cast<__nv_bfloat16*>(base + o_o);
  h->cb = reinterpret_cast<__nv_bfloat16*>(base + o_c);
  h->sh = reinterpret_cast<__nv_bfloat16*>(base + o_sh);
  h->status = reinterpret_cast<unsigned*>(base + o_status);
  h->tile_counter = reinterpret_cast<int*>(base + o_tcount);
  h->sort_sync = reinterpret_cast<unsigned*>(h->tile_counter + 2);
  h->dep = fusable ? reinterpret_cast<int*>(base + o_dep) : nullptr;
  h->f8 = reinterpret_cast<lmoe::Fp8State*>(base + o_f8);
  h->x8 = reinterpret_cast<uint8_t*>(base + o_x8);
  h->y32 = reinterpret_cast<float*>(base + o_y32);
  e = cudaMemset(h->status, 0, 16);
  if (e == cudaSuccess) e = cudaMemset(h->tile_counter, 0, 16);
  if (e == cudaSuccess && h->dep) e = cudaMemset(h->dep, 0, E * (F / 256) * 4);
  if (e == cudaSuccess) {
    // delayed scaling starts with an empty history and unit scales
    lmoe::Fp8State init;
    memset(&init, 0, sizeof(init));
    for (int i = 0; i < lmoe::kFp8Tensors; ++i) init.scale[i] = 1.0f;
    e = cudaMemcpy(h->f8, &init, sizeof(init), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return LATENTMOE_ERR_CUDA;
  }
  *out = h;
  return LATENTMOE_OK;
}

int latentmoe_destroy(latentmoe_t h) {
  if (h == nullptr) return LATENTMOE_OK;
  for (cudaEvent_t ev : h->events) cudaEventDestroy(ev);
  if (h->x_stage) cudaFree(h->x_stage);
  if (h->y_stage) cudaFree(h->y_stage);
  if (h->copy_in) cudaStreamSynchronize(h->copy_in);
  if (h->copy_out) cudaStreamSynchronize(h->copy_out);
  for (int i = 0; i < 2; ++i) {
    if (h->xs[i]) cudaFree(h->xs[i]);
    if (h->ys[i]) cudaFree(h->ys[i]);
    if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
    if (h->ev_fwd[i]) cudaEventDestroy(h->ev_fwd[i]);
    if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
  }
  if (h->copy_in) cudaStreamDestroy(h->copy_in);
  if (h->copy_out) cudaStreamDestroy(h->copy_out);
  if (h->ws) cudaFree(h->ws);
  if (h->wmem) cudaFree(h->wmem);
  if (h->cap_mem) cudaFree(h->cap_mem);
  delete h;
  return LATENTMOE_OK;
}

int latentmoe_load_weights(latentmoe_t h, const latentmoe_weights* w,
                           latentmoe_stream_t stream) {
  if (h == nullptr || w == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  const latentmoe_dims& d = h->dims;
  const bool shared = d.shared_ffn > 0;
  const bool bias = (h->flags & (LATENTMOE_ROUTER_BIAS | LATENTMOE_SELECT_BIAS)) != 0;
  if (!w->w_r || !w->w_dn || !w->w_g || !w->w_u || !w->w_d || !w->w_up)
    return LATENTMOE_ERR_INVALID_ARG;
  if (bias && !w->b_r) return LATENTMOE_ERR_INVALID_ARG;
  if (shared && (!w->w_gs || !w->w_us || !w->w_ds)) return LATENTMOE_ERR_INVALID_ARG;
  const void* ptrs[] = {w->w_r, w->w_dn, w->w_g, w->w_u, w->w_d, w->w_up};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LATENTMOE_ERR_UNSUPPORTED;
  if (shared && (!aligned16(w->w_gs) || !aligned16(w->w_us) || !aligned16(w->w_ds)))
    return LATENTMOE_ERR_UNSUPPORTED;
  if (bias && (reinterpret_cast<uintptr_t>(w->b_r) & 3u)) return LATENTMOE_ERR_UNSUPPORTED;
  LMOE_CK(h, cudaSetDevice(h->device));

  const uint64_t E = d.num_experts, dd = d.hidden, l = d.latent, F = d.ffn, Fs = d.shared_ffn;
  // layout of the owned copy: dense weights as given, expert weights packed
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 1024);
    return o;
  };
  // dense weights: bf16 as given, or E4M3 codes (one scale per matrix)
  const uint64_t db = h->fp8_dense ? 1 : 2;
  const size_t o_r = take(E * dd * 2), o_b = take(bias ? E * 4 : 16), o_dn = take(l * dd * db);
  const size_t o_up = take(dd * l * db);
  // expert weights: packed bf16 tiles, or packed E4M3 codes plus their scales
  const uint64_t eb = h->fp8 ? 1 : 2;
  const size_t o_g = take(E * F * l * eb), o_u = take(E * F * l * eb), o_d = take(E * l * F * eb);
  const size_t o_ws = take(h->fp8 ? 3 * E * 4 : 16), o_wa = take(h->fp8 ? 3 * E * 4 : 16);
  const size_t o_gs = take(shared ? Fs * dd * db : 16), o_us = take(shared ? Fs * dd * db : 16);
  const size_t o_ds = take(shared ? dd * Fs * db : 16);
  const size_t o_dws = take(kDenseW * 4), o_dwa = take(kDenseW * 4);
  // the caller's writes to its weights are complete or ordered before `s`;
  // replacing earlier weights frees them (cudaFree waits for the device)
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  h->loaded = false;
  if (h->wmem) {
    cudaFree(h->wmem);
    h->wmem = nullptr;
  }
  {
    const cudaError_t e = cudaMalloc(&h->wmem, off);
    if (e != cudaSuccess) {
      cudaGetLastError();
      h->wmem = nullptr;
      return fail_cuda(h, e);
    }
  }
  char* base = static_cast<char*>(h->wmem);
  latentmoe_weights o;
  memset(&o, 0, sizeof(o));
  o.w_r = base + o_r;
  o.b_r = bias ? reinterpret_cast<const float*>(base + o_b) : nullptr;
  o.w_dn = base + o_dn;
  o.w_up = base + o_up;
  o.w_g = base + o_g;
  o.w_u = base + o_u;
  o.w_d = base + o_d;
  if (shared) {
    o.w_gs = base + o_gs;
    o.w_us = base + o_us;
    o.w_ds = base + o_ds;
  }
  h->w_scale = h->fp8 ? reinterpret_cast<float*>(base + o_ws) : nullptr;
  h->dw_scale = reinterpret_cast<float*>(base + o_dws);
  const auto dd2d = cudaMemcpyDeviceToDevice;
  LMOE_CK(h, cudaMemcpyAsync(const_cast<void*>(o.w_r), w->w_r, E * dd * 2, dd2d, s));
  if (bias) LMOE_CK(h, cudaMemcpyAsync(const_cast<float*>(o.b_r), w->b_r, E * 4, dd2d, s));
  {
    // dense weights: W_dn, W_up, W_gs, W_us, W_ds (the shared three only with F_s > 0)
    const void* dsrc[kDenseW] = {w->w_dn, w->w_up, w->w_gs, w->w_us, w->w_ds};
    void* ddst[kDenseW] = {const_cast<void*>(o.w_dn), const_cast<void*>(o.w_up),
                           const_cast<void*>(o.w_gs), const_cast<void*>(o.w_us),
                           const_cast<void*>(o.w_ds)};
    const uint64_t drows[kDenseW] = {l, dd, Fs, Fs, dd};
    const uint64_t dcols[kDenseW] = {dd, l, dd, dd, Fs};
    const int nd = shared ? kDenseW : 2;
    if (h->fp8_dense) {
      // s = max |W| / 448 per matrix, codes row-major (the dense GEMM's layout)
      unsigned* damax = reinterpret_cast<unsigned*>(base + o_dwa);
      LMOE_CK(h, cudaMemsetAsync(damax, 0, kDenseW * 4, s));
      for (int m = 0; m < nd; ++m)
        LMOE_CK(h, lmoe::launch_absmax_groups(static_cast<const __nv_bfloat16*>(dsrc[m]), 1,
                                              static_cast<long long>(drows[m] * dcols[m]),
                                              damax + m, h->sms, s));
      LMOE_CK(h, lmoe::launch_scales_from_amax(damax, kDenseW, h->dw_scale, s));
      for (int m = 0; m < nd; ++m)
        LMOE_CK(h, lmoe::launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(dsrc[m]),
                                              static_cast<uint8_t*>(ddst[m]),
                                              static_cast<long long>(drows[m]),
                                              static_cast<long long>(dcols[m]),
                                              static_cast<long long>(drows[m]), h->dw_scale + m,
                                              false, h->sms, s));
    } else {
      for (int m = 0; m < nd; ++m)
        LMOE_CK(h, cudaMemcpyAsync(ddst[m], dsrc[m], drows[m] * dcols[m] * 2, dd2d, s));
    }
  }
  typedef const __nv_bfloat16* cbf;
  const void* srcs[3] = {w->w_g, w->w_u, w->w_d};
  void* dsts[3] = {const_cast<void*>(o.w_g), const_cast<void*>(o.w_u), const_cast<void*>(o.w_d)};
  const long long mrows[3] = {static_cast<long long>(F), static_cast<long long>(F),
                              static_cast<long long>(l)};
  const long long mcols[3] = {static_cast<long long>(l), static_cast<long long>(l),
                              static_cast<long long>(F)};
  if (h->fp8) {
    // s = max |W_e| / 448 per expert matrix, then codes in the packed layout
    unsigned* amax = reinterpret_cast<unsigned*>(base + o_wa);
    LMOE_CK(h, cudaMemsetAsync(amax, 0, 3 * E * 4, s));
    for (int m = 0; m < 3; ++m)
      LMOE_CK(h, lmoe::launch_absmax_groups(static_cast<cbf>(srcs[m]), static_cast<long long>(E),
                                            mrows[m] * mcols[m], amax + m * E, h->sms, s));
    LMOE_CK(h, lmoe::launch_scales_from_amax(amax, static_cast<int>(3 * E), h->w_scale, s));
    for (int m = 0; m < 3; ++m)
      LMOE_CK(h, lmoe::launch_quantize_e4m3(static_cast<cbf>(srcs[m]),
                                            static_cast<uint8_t*>(dsts[m]),
                                            static_cast<long long>(E) * mrows[m], mcols[m],
                                            mrows[m], h->w_scale + m * E, true, h->sms, s));
  } else {
    for (int m = 0; m < 3; ++m)
      LMOE_CK(h, lmoe::launch_pack_tiles(srcs[m], dsts[m], static_cast<long long>(E) * mrows[m],
                                         mcols[m] * 2, h->sms, s));
  }
  // the caller may free or reuse its buffers once this returns
  LMOE_CK(h, cudaStreamSynchronize(s));

  bool ok = true;
  ok &= make_map(&h->m_wr, o.w_r, E, dd, dd,
                 static_cast<uint32_t>(lmoe::router_w_box_rows(static_cast<int>(E))),
                 static_cast<uint32_t>(lmoe::router_box_cols(static_cast<int>(E))));
  if (h->fp8_dense)
    ok &= make_map_u8(&h->m_down.b, o.w_dn, l, dd, dd, 128);
  else
    ok &= make_map(&h->m_down.b, o.w_dn, l, dd, dd, 128);
  // tiles of 128 rows x 128 bytes
  ok &= make_tile_map(&h->m_wg, o.w_g, E * F / 128 * (l * eb / 128), h->fp8);
  ok &= make_tile_map(&h->m_wu, o.w_u, E * F / 128 * (l * eb / 128), h->fp8);
  ok &= make_tile_map(&h->m_wd, o.w_d, E * l / 128 * (F * eb / 128), h->fp8);
  if (h->fp8_dense) {
    ok &= make_map_u8(&h->m_up.b, o.w_up, dd, l, l, 128);
    if (shared) {
      ok &= make_map_u8(&h->m_shared.b, o.w_gs, Fs, dd, dd, 128);
      ok &= make_map_u8(&h->m_shared.bu, o.w_us, Fs, dd, dd, 128);
      ok &= make_map_u8(&h->m_up.b2, o.w_ds, dd, Fs, Fs, 128);
    }
  } else {
    ok &= make_map(&h->m_up.b, o.w_up, dd, l, l, 128);
    if (shared) {
      ok &= make_map(&h->m_shared.b, o.w_gs, Fs, dd, dd, 128);
      ok &= make_map(&h->m_shared.bu, o.w_us, Fs, dd, dd, 128);
      ok &= make_map(&h->m_up.b2, o.w_ds, dd, Fs, Fs, 128);
    }
  }
  if (!ok) return LATENTMOE_ERR_CUDA;
  // unused map slots still travel as kernel parameters: give them a valid copy
  h->m_down.bu = h->m_down.a2 = h->m_down.b2 = h->m_down.b;
  if (shared) {
    h->m_shared.a2 = h->m_shared.b2 = h->m_shared.b;
  } else {
    h->m_up.b2 = h->m_up.b;
  }
  h->m_up.bu = h->m_up.b;
  h->w = o;
  h->loaded = true;
  return LATENTMOE_OK;
}

namespace {

// The forward. With replay_idx the expert choices are the caller's (router
// replay); with replay_gates as well the router is not run at all.
int forward_impl(latentmoe_t h, const void* x, void* out, int64_t T, cudaStream_t s,
                 const int32_t* replay_idx, const float* replay_gates) {
  LMOE_CK(h, cudaSetDevice(h->device));
  const lmoe::PdlScope pdl_scope(h->pdl);
  NvtxStages nv;
  const latentmoe_dims& d = h->dims;
  const int E = static_cast<int>(d.num_experts), k = h->k;
  const int dd = static_cast<int>(d.hidden), l = static_cast<int>(d.latent);
  const int F = static_cast<int>(d.ffn), Fs = static_cast<int>(d.shared_ffn);
  const int Ti = static_cast<int>(T), S = Ti * k;
  const bool out32 = (h->flags & LATENTMOE_OUT_FP32) != 0;

  // activation maps for this call
  CUtensorMap mx, mxr, mzp, mh, mc, msh;
  bool ok = make_map(&mx, x, T, dd, dd, 128);
  ok &= make_map(&mxr, x, T, dd, dd, 128,
                 static_cast<uint32_t>(lmoe::router_box_cols(static_cast<int>(E))));
  ok &= make_token_map(&mzp, h->zp, S, l, h->fp8);
  ok &= make_token_map(&mh, h->hb, S, F, h->fp8);
  CUtensorMap mx8;
  if (h->fp8_dense) {
    // E4M3 codes of x, c and the shared hidden, 128-row boxes
    ok &= make_map_u8(&mx8, h->x8, T, dd, dd, 128);
    ok &= make_map_u8(&mc, h->cb, T, l, l, 128);
    if (Fs > 0) ok &= make_map_u8(&msh, h->sh, T, Fs, Fs, 128);
  } else {
    ok &= make_map(&mc, h->cb, T, l, l, 128);
    if (Fs > 0) ok &= make_map(&msh, h->sh, T, Fs, Fs, 128);
  }
  if (!ok) return LATENTMOE_ERR_CUDA;

  const int slot_base = h->prof_slots > 0
                            ? static_cast<int>(h->forwards % h->prof_slots) * (kNumStages + 1)
                            : 0;
  h->forwards += 1;
  record(h, slot_base, 0, s);
  nv.next(0);

  // 0: router GEMM + softmax + stable top-k (fused); skipped when the caller
  // replays both choices and gates
  if (replay_gates == nullptr) {
    lmoe::RouterArgs ra;
    memset(&ra, 0, sizeof(ra));
    ra.T = Ti;
    ra.E = E;
    ra.k = k;
    ra.renorm = (h->flags & LATENTMOE_RENORM) ? 1 : 0;
    ra.kb = dd / lmoe::router_bk(static_cast<int>(E));
    ra.bias = (h->flags & (LATENTMOE_ROUTER_BIAS | LATENTMOE_SELECT_BIAS)) ? h->w.b_r : nullptr;
    ra.bias_select = (h->flags & LATENTMOE_SELECT_BIAS) ? 1 : 0;
    ra.logits = h->logits;
    ra.idx = h->idx;
    ra.gates = h->gates;
    ra.status = h->status;
    LMOE_CK(h, lmoe::launch_router_topk(mxr, h->m_wr, ra, h->sms, s));
    h->launches += 1;
  }
  record(h, slot_base, 1, s);
  nv.next(1);
  // 1: replayed choices (and gates from the router's softmax if not given)
  if (replay_idx != nullptr) {
    LMOE_CK(h, cudaMemcpyAsync(h->idx, replay_idx, static_cast<size_t>(S) * 4,
                               cudaMemcpyDeviceToDevice, s));
    if (replay_gates != nullptr) {
      LMOE_CK(h, cudaMemcpyAsync(h->gates, replay_gates, static_cast<size_t>(S) * 4,
                                 cudaMemcpyDeviceToDevice, s));
    } else {
      LMOE_CK(h, lmoe::launch_replay_gates(h->logits, Ti, E, h->idx, k,
                                           (h->flags & LATENTMOE_RENORM) ? 1 : 0, h->gates, s));
      h->launches += 1;
    }
  }
  record(h, slot_base, 2, s);
  nv.next(2);
  // 2: counting sort
  {
    const int r = run_sort(h, Ti, s);
    if (r != LATENTMOE_OK) return r;
  }
  record(h, slot_base, 3, s);
  nv.next(3);
  // 3: latent down-projection scattered to the expert-sorted slots (with
  // E4M3 dense GEMMs, x is quantized first)
  if (h->fp8_dense) {
    LMOE_CK(h, lmoe::launch_quantize_act(static_cast<const __nv_bfloat16*>(x), h->x8,
                                         static_cast<long long>(T) * dd, &h->f8->scale[2],
                                         &h->f8->amax[2], h->sms, s));
    h->launches += 1;
  }
  {
    GemmMaps m = h->m_down;
    m.a = h->fp8_dense ? mx8 : mx;
    GemmArgs a = base_args(h);
    a.M = Ti;
    a.N = l;
    a.n_tiles = ceil_div(l, lmoe::kBN);
    a.kb1 = dd / (h->fp8_dense ? lmoe::kBK8 : lmoe::kBK);
    a.out = h->zp;
    a.ldo = l;
    a.out_rows = h->dims.max_tokens * h->k;
    a.pos = h->pos;
    a.topk = k;
    if (h->fp8) {
      a.out_scale = &h->f8->scale[0];
      a.out_amax = &h->f8->amax[0];
      a.a_scale = &h->f8->scale[2];
      a.b_scale = &h->dw_scale[0];
      LMOE_CK(h, lmoe::launch_gemm_scatter_f8(m, a, dense_grid(h, Ti, a.n_tiles), s,
                                              h->fp8_dense, dense_pair_sms(h)));
    } else {
      LMOE_CK(h, lmoe::launch_gemm_scatter(m, a, dense_grid(h, Ti, a.n_tiles), s,
                                           dense_pair_sms(h)));
    }
    h->launches += 1;
  }
  record(h, slot_base, 4, s);
  nv.next(4);
  if (h->cap > 0) {
    // 4+5: multi-round fixed-capacity schedule: per round, gate+up of the
    // round's slots into the fixed round buffer, then down back to the slots
    const int r = run_expert_rounds(h, mzp, s);
    if (r != LATENTMOE_OK) return r;
    record(h, slot_base, 5, s);
    nv.next(5);
  } else if (experts_fused(h, Ti)) {
    // 4+5: both expert GEMMs in one launch (timed as stage 4; stage 5 is empty)
    const int r = launch_experts_fused(h, mzp, mh, s);
    if (r != LATENTMOE_OK) return r;
    record(h, slot_base, 5, s);
    nv.next(5);
  } else {
    // 4: grouped gate+up with SwiGLU (weights on the M side, tokens on N)
    lmoe::GroupedArgs a;
    memset(&a, 0, sizeof(a));
    a.seg_offsets = h->offsets;
    a.out = h->hb;
    int r = launch_expert_gate_up(h, a, mzp, s);
    if (r != LATENTMOE_OK) return r;
    record(h, slot_base, 5, s);
    nv.next(5);
    // 5: grouped expert down-projection
    a.out = h->ob;
    r = launch_expert_down(h, a, mh, s);
    if (r != LATENTMOE_OK) return r;
  }
  record(h, slot_base, 6, s);
  nv.next(6);
  // 6: combine (E4M3 dense GEMMs: c written as codes)
  if (h->fp8_dense)
    LMOE_CK(h, lmoe::launch_combine_f8(reinterpret_cast<const float*>(h->ob), h->gates, h->pos,
                                       Ti, k, l,
                                       reinterpret_cast<uint8_t*>(h->cb), &h->f8->scale[3],
                                       &h->f8->amax[3], h->dims.max_tokens * h->k, h->status,
                                       s));
  else
    LMOE_CK(h, lmoe::launch_combine(h->ob, h->gates, h->pos, Ti, k, l, h->cb,
                                    h->dims.max_tokens * h->k, h->status, s));
  h->launches += 1;
  record(h, slot_base, 7, s);
  nv.next(7);
  // 7: shared expert gate+up on the full width
  if (Fs > 0) {
    GemmMaps m = h->m_shared;
    m.a = h->fp8_dense ? mx8 : mx;
    GemmArgs a = base_args(h);
    a.M = Ti;
    a.N = Fs;
    a.n_tiles = Fs / (lmoe::kBN / 2);
    a.kb1 = dd / (h->fp8_dense ? lmoe::kBK8 : lmoe::kBK);
    a.out = h->sh;
    a.ldo = Fs;
    a.out_rows = h->dims.max_tokens;
    if (h->fp8_dense) {
      a.a_scale = &h->f8->scale[2];
      a.b_scale = &h->dw_scale[2];
      a.b_scale2 = &h->dw_scale[3];
      a.out_scale = &h->f8->scale[4];
      a.out_amax = &h->f8->amax[4];
    }
    LMOE_CK(h, lmoe::launch_gemm_swiglu(m, a, dense_grid(h, Ti, a.n_tiles), s, h->fp8_dense,
                                        dense_pair_sms(h)));
    h->launches += 1;
  }
  record(h, slot_base, 8, s);
  nv.next(8);
  // 8: up-projection (+ shared expert's down-projection, K-concatenated; with
  // E4M3 dense GEMMs the two products have their own scales: the
  // up-projection leaves an fp32 partial that the shared down GEMM adds)
  if (h->fp8_dense) {
    GemmArgs a = base_args(h);
    a.M = Ti;
    a.N = dd;
    a.n_tiles = ceil_div(dd, lmoe::kBN);
    a.a_scale = &h->f8->scale[3];
    a.b_scale = &h->dw_scale[1];
    a.kb1 = l / lmoe::kBK8;
    const int grid = dense_grid(h, Ti, a.n_tiles);
    GemmMaps m = h->m_up;
    m.a = mc;
    m.a2 = mc;
    m.b2 = h->m_up.b;
    if (Fs > 0) {
      a.out = h->y32;
      a.ldo = dd;
      a.out_rows = h->dims.max_tokens;
      LMOE_CK(h, lmoe::launch_gemm_f32(m, a, grid, false, s, true, dense_pair_sms(h)));
      h->launches += 1;
      GemmMaps m2 = h->m_up;
      m2.a = msh;
      m2.b = h->m_up.b2;
      m2.a2 = msh;
      GemmArgs b = a;
      b.a_scale = &h->f8->scale[4];
      b.b_scale = &h->dw_scale[4];
      b.kb1 = Fs / lmoe::kBK8;
      b.addend = h->y32;
      b.ld_add = dd;
      b.out = out;
      b.ldo = dd;
      b.out_rows = T;
      if (out32)
        LMOE_CK(h, lmoe::launch_gemm_f32(m2, b, grid, false, s, true, dense_pair_sms(h)));
      else
        LMOE_CK(h, lmoe::launch_gemm_bf16(m2, b, grid, false, s, true, dense_pair_sms(h)));
    } else {
      a.out = out;
      a.ldo = dd;
      a.out_rows = T;
      if (out32)
        LMOE_CK(h, lmoe::launch_gemm_f32(m, a, grid, false, s, true, dense_pair_sms(h)));
      else
        LMOE_CK(h, lmoe::launch_gemm_bf16(m, a, grid, false, s, true, dense_pair_sms(h)));
    }
    h->launches += 1;
  } else {
    GemmMaps m = h->m_up;
    m.a = mc;
    if (Fs > 0) m.a2 = msh; else m.a2 = mc;
    GemmArgs a = base_args(h);
    a.M = Ti;
    a.N = dd;
    a.n_tiles = ceil_div(dd, lmoe::kBN);
    a.kb1 = l / lmoe::kBK;
    a.kb2 = Fs / lmoe::kBK;
    a.out = out;
    a.ldo = dd;
    a.out_rows = T;
    const int grid = dense_grid(h, Ti, a.n_tiles);
    if (out32)
      LMOE_CK(h, lmoe::launch_gemm_f32(m, a, grid, Fs > 0, s, false, dense_pair_sms(h)));
    else
      LMOE_CK(h, lmoe::launch_gemm_bf16(m, a, grid, Fs > 0, s, false, dense_pair_sms(h)));
    h->launches += 1;
  }
  record(h, slot_base, 9, s);
  nv.next(9);
  // 9: delayed scaling: this forward's maxima enter the history, next scales
  if (h->fp8) {
    LMOE_CK(h, lmoe::launch_fp8_update(h->f8, kFp8Acts, s));
    h->launches += 1;
  }
  record(h, slot_base, 10, s);
  nv.next(10);
  h->last_T = T;
  return LATENTMOE_OK;
}

int check_forward_args(latentmoe_t h, const void* x, void* out, int64_t T) {
  if (h == nullptr || x == nullptr || out == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->dims.max_tokens) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->loaded) return LATENTMOE_ERR_NOT_LOADED;
  if (!aligned16(x) || !aligned16(out)) return LATENTMOE_ERR_UNSUPPORTED;
  return LATENTMOE_OK;
}

}  // namespace

int latentmoe_forward(latentmoe_t h, const void* x, void* out, int64_t T, latentmoe_stream_t st) {
  const int r = check_forward_args(h, x, out, T);
  if (r != LATENTMOE_OK) return r;
  return forward_impl(h, x, out, T, reinterpret_cast<cudaStream_t>(st), nullptr, nullptr);
}

int latentmoe_forward_routed(latentmoe_t h, const void* x, const int32_t* idx,
                             const float* gates, void* out, int64_t T, latentmoe_stream_t st) {
  const int r = check_forward_args(h, x, out, T);
  if (r != LATENTMOE_OK) return r;
  if (idx == nullptr || (reinterpret_cast<uintptr_t>(idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(gates) & 3u))
    return LATENTMOE_ERR_INVALID_ARG;
  return forward_impl(h, x, out, T, reinterpret_cast<cudaStream_t>(st), idx, gates);
}

int latentmoe_forward_host(latentmoe_t h, const void* x_host, void* out_host, int64_t T,
                           latentmoe_stream_t st) {
  if (h == nullptr || x_host == nullptr || out_host == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->dims.max_tokens) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->loaded) return LATENTMOE_ERR_NOT_LOADED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const size_t x_bytes = static_cast<size_t>(T) * h->dims.hidden * 2;
  const size_t y_bytes =
      static_cast<size_t>(T) * h->dims.hidden * ((h->flags & LATENTMOE_OUT_FP32) ? 4 : 2);
  if (h->x_stage == nullptr) {
    LMOE_CK(h, cudaMalloc(&h->x_stage, static_cast<size_t>(h->dims.max_tokens) * h->dims.hidden * 2));
    LMOE_CK(h, cudaMalloc(&h->y_stage, static_cast<size_t>(h->dims.max_tokens) * h->dims.hidden * 4));
  }
  LMOE_CK(h, cudaMemcpyAsync(h->x_stage, x_host, x_bytes, cudaMemcpyHostToDevice, s));
  const int r = latentmoe_forward(h, h->x_stage, h->y_stage, T, st);
  if (r != LATENTMOE_OK) return r;
  LMOE_CK(h, cudaMemcpyAsync(out_host, h->y_stage, y_bytes, cudaMemcpyDeviceToHost, s));
  LMOE_CK(h, cudaStreamSynchronize(s));
  return LATENTMOE_OK;
}

int latentmoe_forward_host_async(latentmoe_t h, const void* x_host, void* out_host, int64_t T,
                                 latentmoe_stream_t st) {
  if (h == nullptr || x_host == nullptr || out_host == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->dims.max_tokens) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->loaded) return LATENTMOE_ERR_NOT_LOADED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const size_t x_bytes = static_cast<size_t>(T) * h->dims.hidden * 2;
  const size_t y_bytes =
      static_cast<size_t>(T) * h->dims.hidden * ((h->flags & LATENTMOE_OUT_FP32) ? 4 : 2);
  if (h->copy_in == nullptr) {
    // first call: staging slots, copy streams and events
    const size_t xcap = static_cast<size_t>(h->dims.max_tokens) * h->dims.hidden * 2;
    const size_t ycap = static_cast<size_t>(h->dims.max_tokens) * h->dims.hidden * 4;
    for (int i = 0; i < 2; ++i) {
      LMOE_CK(h, cudaMalloc(&h->xs[i], xcap));
      LMOE_CK(h, cudaMalloc(&h->ys[i], ycap));
      LMOE_CK(h, cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming));
      LMOE_CK(h, cudaEventCreateWithFlags(&h->ev_fwd[i], cudaEventDisableTiming));
      LMOE_CK(h, cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming));
    }
    LMOE_CK(h, cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking));
    LMOE_CK(h, cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking));
  }
  const int slot = static_cast<int>(h->host_steps & 1);
  // x in: once the forward two steps back has read this slot
  if (h->host_steps >= 2) LMOE_CK(h, cudaStreamWaitEvent(h->copy_in, h->ev_fwd[slot], 0));
  LMOE_CK(h, cudaMemcpyAsync(h->xs[slot], x_host, x_bytes, cudaMemcpyHostToDevice, h->copy_in));
  LMOE_CK(h, cudaEventRecord(h->ev_in[slot], h->copy_in));
  // the forward on the caller's stream: after its x is in and after the
  // output copy of two steps back has read this slot's y
  LMOE_CK(h, cudaStreamWaitEvent(s, h->ev_in[slot], 0));
  if (h->host_steps >= 2) LMOE_CK(h, cudaStreamWaitEvent(s, h->ev_out[slot], 0));
  const int r = latentmoe_forward(h, h->xs[slot], h->ys[slot], T, st);
  if (r != LATENTMOE_OK) return r;
  LMOE_CK(h, cudaEventRecord(h->ev_fwd[slot], s));
  // y out, behind the forward
  LMOE_CK(h, cudaStreamWaitEvent(h->copy_out, h->ev_fwd[slot], 0));
  LMOE_CK(h, cudaMemcpyAsync(out_host, h->ys[slot], y_bytes, cudaMemcpyDeviceToHost,
                             h->copy_out));
  LMOE_CK(h, cudaEventRecord(h->ev_out[slot], h->copy_out));
  h->host_steps += 1;
  return LATENTMOE_OK;
}

int latentmoe_host_wait(latentmoe_t h) {
  if (h == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  LMOE_CK(h, cudaSetDevice(h->device));
  if (h->copy_in) LMOE_CK(h, cudaStreamSynchronize(h->copy_in));
  if (h->copy_out) LMOE_CK(h, cudaStreamSynchronize(h->copy_out));
  return LATENTMOE_OK;
}

int latentmoe_route_from_logits(latentmoe_t h, const float* logits, int64_t T, int32_t* idx,
                                float* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
                                int32_t* pos, latentmoe_stream_t st) {
  if (h == nullptr || logits == nullptr || idx == nullptr || gates == nullptr)
    return LATENTMOE_ERR_INVALID_ARG;
  if (T < 1 || T > h->dims.max_tokens) return LATENTMOE_ERR_INVALID_ARG;
  // a selection-only bias comes with the weights
  if ((h->flags & LATENTMOE_SELECT_BIAS) && !h->loaded) return LATENTMOE_ERR_NOT_LOADED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const int r = run_routing(h, logits, static_cast<int>(T), s, 0);
  if (r != LATENTMOE_OK) return r;
  const size_t S = static_cast<size_t>(T) * h->k;
  const size_t E = static_cast<size_t>(h->dims.num_experts);
  LMOE_CK(h, cudaMemcpyAsync(idx, h->idx, S * 4, cudaMemcpyDeviceToDevice, s));
  LMOE_CK(h, cudaMemcpyAsync(gates, h->gates, S * 4, cudaMemcpyDeviceToDevice, s));
  if (counts) LMOE_CK(h, cudaMemcpyAsync(counts, h->counts, E * 4, cudaMemcpyDeviceToDevice, s));
  if (offsets)
    LMOE_CK(h, cudaMemcpyAsync(offsets, h->offsets, (E + 1) * 4, cudaMemcpyDeviceToDevice, s));
  if (perm) LMOE_CK(h, cudaMemcpyAsync(perm, h->perm, S * 4, cudaMemcpyDeviceToDevice, s));
  if (pos) LMOE_CK(h, cudaMemcpyAsync(pos, h->pos, S * 4, cudaMemcpyDeviceToDevice, s));
  return LATENTMOE_OK;
}

int latentmoe_get_routing(latentmoe_t h, float* logits, int32_t* idx, float* gates,
                          int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                          latentmoe_stream_t st) {
  if (h == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (h->last_T == 0) return LATENTMOE_ERR_NOT_LOADED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const size_t T = static_cast<size_t>(h->last_T);
  const size_t S = T * h->k;
  const size_t E = static_cast<size_t>(h->dims.num_experts);
  const auto dd = cudaMemcpyDeviceToDevice;
  if (logits) LMOE_CK(h, cudaMemcpyAsync(logits, h->logits, T * E * 4, dd, s));
  if (idx) LMOE_CK(h, cudaMemcpyAsync(idx, h->idx, S * 4, dd, s));
  if (gates) LMOE_CK(h, cudaMemcpyAsync(gates, h->gates, S * 4, dd, s));
  if (counts) LMOE_CK(h, cudaMemcpyAsync(counts, h->counts, E * 4, dd, s));
  if (offsets) LMOE_CK(h, cudaMemcpyAsync(offsets, h->offsets, (E + 1) * 4, dd, s));
  if (perm) LMOE_CK(h, cudaMemcpyAsync(perm, h->perm, S * 4, dd, s));
  if (pos) LMOE_CK(h, cudaMemcpyAsync(pos, h->pos, S * 4, dd, s));
  return LATENTMOE_OK;
}

int latentmoe_lbl_stats(latentmoe_t h, float* prob_sum, int32_t* counts,
                        latentmoe_stream_t st) {
  if (h == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (h->last_T == 0) return LATENTMOE_ERR_NOT_LOADED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const int E = static_cast<int>(h->dims.num_experts);
  if (prob_sum) {
    LMOE_CK(h, lmoe::launch_lbl_prob_sum(h->logits, static_cast<int>(h->last_T), E,
                                         h->lbl_partial, prob_sum, s));
    h->launches += 2;
  }
  if (counts)
    LMOE_CK(h, cudaMemcpyAsync(counts, h->counts, static_cast<size_t>(E) * 4,
                               cudaMemcpyDeviceToDevice, s));
  return LATENTMOE_OK;
}

int latentmoe_get_status(latentmoe_t h, uint32_t* device_status) {
  if (h == nullptr || device_status == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  LMOE_CK(h, cudaSetDevice(h->device));
  LMOE_CK(h, cudaDeviceSynchronize());
  unsigned v = 0;
  LMOE_CK(h, cudaMemcpy(&v, h->status, 4, cudaMemcpyDeviceToHost));
  LMOE_CK(h, cudaMemset(h->status, 0, 4));
  // a wait that gave up may have left the scheduling counters non-zero
  if (v & LATENTMOE_STATUS_TIMEOUT) {
    LMOE_CK(h, cudaMemset(h->tile_counter, 0, 16));
    if (h->dep)
      LMOE_CK(h, cudaMemset(h->dep, 0, h->dims.num_experts * (h->dims.ffn / 256) * 4));
  }
  *device_status = v;
  if (v & LATENTMOE_STATUS_TIMEOUT) return LATENTMOE_ERR_TIMEOUT;
  if (v != 0) return LATENTMOE_ERR_DEVICE_STATUS;
  return LATENTMOE_OK;
}

int latentmoe_set_profiling(latentmoe_t h, int slots) {
  if (h == nullptr || slots < 0 || slots > 4096) return LATENTMOE_ERR_INVALID_ARG;
  LMOE_CK(h, cudaSetDevice(h->device));
  for (cudaEvent_t ev : h->events) cudaEventDestroy(ev);
  h->events.clear();
  h->prof_slots = 0;
  h->forwards = 0;
  const size_t n = static_cast<size_t>(slots) * (kNumStages + 1);
  for (size_t i = 0; i < n; ++i) {
    cudaEvent_t ev;
    LMOE_CK(h, cudaEventCreate(&ev));
    h->events.push_back(ev);
  }
  h->prof_slots = slots;
  return LATENTMOE_OK;
}

int latentmoe_get_stage_times(latentmoe_t h, int slot, float* ms, int count) {
  if (h == nullptr || ms == nullptr || slot < 0 || slot >= h->prof_slots || count < 0)
    return LATENTMOE_ERR_INVALID_ARG;
  const int base = slot * (kNumStages + 1);
  LMOE_CK(h, cudaEventSynchronize(h->events[base + kNumStages]));
  for (int i = 0; i < count && i < kNumStages; ++i) {
    float t = 0.0f;
    LMOE_CK(h, cudaEventElapsedTime(&t, h->events[base + i], h->events[base + i + 1]));
    ms[i] = t;
  }
  return LATENTMOE_OK;
}

int latentmoe_set_capacity(latentmoe_t h, int64_t capacity, int64_t group_size,
                           int64_t max_rounds) {
  if (h == nullptr || capacity < 0 || max_rounds < 0) return LATENTMOE_ERR_INVALID_ARG;
  const int64_t E = h->dims.num_experts, F = h->dims.ffn;
  if (capacity > 0 && (group_size < 1 || group_size > E)) return LATENTMOE_ERR_INVALID_ARG;
  LMOE_CK(h, cudaSetDevice(h->device));
  LMOE_CK(h, cudaDeviceSynchronize());
  if (h->cap_mem) {
    cudaFree(h->cap_mem);
    h->cap_mem = nullptr;
  }
  h->cap = 0;
  h->cap_group = 0;
  h->cap_rounds = 0;
  h->hround = nullptr;
  h->rin = h->rout = h->rlen = h->rinfo = nullptr;
  if (capacity == 0) return LATENTMOE_OK;
  if (capacity * E > (1ll << 30)) return LATENTMOE_ERR_UNSUPPORTED;
  int64_t rounds = max_rounds;
  if (rounds == 0) {
    // worst case: every token puts min(k, g) of its slots into the smallest group
    const int64_t gmin = E % group_size ? E % group_size : group_size;
    const int64_t per = h->dims.max_tokens * (h->k < gmin ? h->k : gmin);
    rounds = (per + gmin * capacity - 1) / (gmin * capacity);
    if (rounds < 1) rounds = 1;
  }
  if (rounds > 4096) return LATENTMOE_ERR_UNSUPPORTED;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 1024);
    return o;
  };
  const size_t o_h = take(static_cast<size_t>(E * capacity) * F * (h->fp8 ? 1 : 2));
  const size_t o_in = take(static_cast<size_t>(rounds * E) * 4);
  const size_t o_out = take(static_cast<size_t>(rounds * (E + 1)) * 4);
  const size_t o_len = take(static_cast<size_t>(rounds * E) * 4);
  const size_t o_info = take(16);
  {
    const cudaError_t e = cudaMalloc(&h->cap_mem, off);
    if (e != cudaSuccess) {
      cudaGetLastError();
      h->cap_mem = nullptr;
      return fail_cuda(h, e);
    }
  }
  char* base = static_cast<char*>(h->cap_mem);
  h->hround = base + o_h;
  h->rin = reinterpret_cast<int*>(base + o_in);
  h->rout = reinterpret_cast<int*>(base + o_out);
  h->rlen = reinterpret_cast<int*>(base + o_len);
  h->rinfo = reinterpret_cast<int*>(base + o_info);
  LMOE_CK(h, cudaMemset(h->rinfo, 0, 16));
  h->cap = capacity;
  h->cap_group = static_cast<int>(group_size);
  h->cap_rounds = static_cast<int>(rounds);
  return LATENTMOE_OK;
}

int latentmoe_get_rounds(latentmoe_t h, int32_t* take, int32_t* info) {
  if (h == nullptr || info == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (h->cap == 0) return LATENTMOE_ERR_UNSUPPORTED;
  LMOE_CK(h, cudaSetDevice(h->device));
  LMOE_CK(h, cudaDeviceSynchronize());
  int32_t v[2];
  LMOE_CK(h, cudaMemcpy(v, h->rinfo, 8, cudaMemcpyDeviceToHost));
  info[0] = v[0];
  info[1] = v[1];
  info[2] = h->cap_rounds;
  if (take)
    LMOE_CK(h, cudaMemcpy(take, h->rlen,
                          static_cast<size_t>(h->cap_rounds) * h->dims.num_experts * 4,
                          cudaMemcpyDeviceToDevice));
  return LATENTMOE_OK;
}

int latentmoe_set_sm_pairs(latentmoe_t h, int enable) {
  if (h == nullptr || (enable != 0 && enable != 1)) return LATENTMOE_ERR_INVALID_ARG;
  h->sm_pairs = enable != 0;
  return LATENTMOE_OK;
}

int latentmoe_set_expert_fusion(latentmoe_t h, int mode) {
  if (h == nullptr || mode < 0 || mode > 2) return LATENTMOE_ERR_INVALID_ARG;
  h->fuse_experts = mode;
  return LATENTMOE_OK;
}

int latentmoe_set_pdl(latentmoe_t h, int enable) {
  if (h == nullptr || (enable != 0 && enable != 1)) return LATENTMOE_ERR_INVALID_ARG;
  h->pdl = enable != 0;
  return LATENTMOE_OK;
}

int latentmoe_get_launch_count(latentmoe_t h, int64_t* launches) {
  if (h == nullptr || launches == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  *launches = h->launches;
  return LATENTMOE_OK;
}

int latentmoe_last_cuda_error(latentmoe_t h) { return h ? h->last_cuda : 0; }

// ---------------------------------------------------------------- E4M3
int latentmoe_get_fp8_state(latentmoe_t h, float* scales, float* last_amax, int64_t* steps) {
  if (h == nullptr || scales == nullptr || last_amax == nullptr || steps == nullptr)
    return LATENTMOE_ERR_INVALID_ARG;
  if (!h->fp8) return LATENTMOE_ERR_UNSUPPORTED;
  LMOE_CK(h, cudaSetDevice(h->device));
  LMOE_CK(h, cudaDeviceSynchronize());
  lmoe::Fp8State st;
  LMOE_CK(h, cudaMemcpy(&st, h->f8, offsetof(lmoe::Fp8State, hist), cudaMemcpyDeviceToHost));
  for (int i = 0; i < kFp8Acts; ++i) {
    scales[i] = st.scale[i];
    last_amax[i] = st.last_amax[i];
  }
  *steps = st.steps;
  return LATENTMOE_OK;
}

int latentmoe_get_fp8_codes(latentmoe_t h, uint8_t* z_codes, uint8_t* h_codes,
                            latentmoe_stream_t st) {
  if (h == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->fp8) return LATENTMOE_ERR_UNSUPPORTED;
  if (h->last_T < 1) return LATENTMOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const size_t S = static_cast<size_t>(h->last_T) * h->k;
  if (z_codes)
    LMOE_CK(h, cudaMemcpyAsync(z_codes, h->zp, S * h->dims.latent, cudaMemcpyDeviceToDevice, s));
  if (h_codes)
    LMOE_CK(h, cudaMemcpyAsync(h_codes, h->hb, S * h->dims.ffn, cudaMemcpyDeviceToDevice, s));
  return LATENTMOE_OK;
}

int latentmoe_set_fp8_scales(latentmoe_t h, const float* scales) {
  if (h == nullptr || scales == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->fp8) return LATENTMOE_ERR_UNSUPPORTED;
  for (int i = 0; i < kFp8Acts; ++i)
    if (!(scales[i] > 0.0f) || !(scales[i] < 3.0e38f)) return LATENTMOE_ERR_INVALID_ARG;
  LMOE_CK(h, cudaSetDevice(h->device));
  LMOE_CK(h, cudaDeviceSynchronize());
  lmoe::Fp8State init;
  memset(&init, 0, sizeof(init));
  for (int i = 0; i < lmoe::kFp8Tensors; ++i) init.scale[i] = i < kFp8Acts ? scales[i] : 1.0f;
  LMOE_CK(h, cudaMemcpy(h->f8, &init, sizeof(init), cudaMemcpyHostToDevice));
  return LATENTMOE_OK;
}

int latentmoe_get_fp8_weight_scales(latentmoe_t h, float* scales) {
  if (h == nullptr || scales == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->fp8) return LATENTMOE_ERR_UNSUPPORTED;
  if (!h->loaded) return LATENTMOE_ERR_NOT_LOADED;
  LMOE_CK(h, cudaSetDevice(h->device));
  LMOE_CK(h, cudaDeviceSynchronize());
  LMOE_CK(h, cudaMemcpy(scales, h->w_scale, 3 * h->dims.num_experts * 4, cudaMemcpyDeviceToHost));
  float* dense = scales + 3 * h->dims.num_experts;
  if (h->fp8_dense) {
    LMOE_CK(h, cudaMemcpy(dense, h->dw_scale, kDenseW * 4, cudaMemcpyDeviceToHost));
  } else {
    for (int i = 0; i < kDenseW; ++i) dense[i] = 1.0f;
  }
  return LATENTMOE_OK;
}

int latentmoe_get_fp8_dense_codes(latentmoe_t h, uint8_t* x_codes, uint8_t* c_codes,
                                  uint8_t* sh_codes, latentmoe_stream_t st) {
  if (h == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  if (!h->fp8_dense) return LATENTMOE_ERR_UNSUPPORTED;
  if (h->last_T < 1 || (sh_codes != nullptr && h->dims.shared_ffn == 0))
    return LATENTMOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  LMOE_CK(h, cudaSetDevice(h->device));
  const size_t T = static_cast<size_t>(h->last_T);
  if (x_codes)
    LMOE_CK(h, cudaMemcpyAsync(x_codes, h->x8, T * h->dims.hidden, cudaMemcpyDeviceToDevice, s));
  if (c_codes)
    LMOE_CK(h, cudaMemcpyAsync(c_codes, h->cb, T * h->dims.latent, cudaMemcpyDeviceToDevice, s));
  if (sh_codes)
    LMOE_CK(h, cudaMemcpyAsync(sh_codes, h->sh, T * h->dims.shared_ffn, cudaMemcpyDeviceToDevice,
                               s));
  return LATENTMOE_OK;
}

int latentmoe_quantize_e4m3(const void* src, int64_t groups, int64_t rows, int64_t cols,
                            uint8_t* codes, float* scales, latentmoe_stream_t st) {
  if (src == nullptr || codes == nullptr || scales == nullptr || groups < 1 || rows < 1 ||
      cols < 1)
    return LATENTMOE_ERR_INVALID_ARG;
  if (cols % 16 || groups > 65535 || !aligned16(src) || !aligned16(codes) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u))
    return LATENTMOE_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  const int sms = num_sms();
  // the scale buffer first holds the maxima (float bits), then the scales
  unsigned* amax = reinterpret_cast<unsigned*>(scales);
  if (cudaMemsetAsync(amax, 0, groups * 4, s) != cudaSuccess) return LATENTMOE_ERR_CUDA;
  typedef const __nv_bfloat16* cbf;
  if (lmoe::launch_absmax_groups(static_cast<cbf>(src), groups, rows * cols, amax, sms, s) !=
          cudaSuccess ||
      lmoe::launch_scales_from_amax(amax, static_cast<int>(groups), scales, s) != cudaSuccess ||
      lmoe::launch_quantize_e4m3(static_cast<cbf>(src), codes, groups * rows, cols, rows, scales,
                                 false, sms, s) != cudaSuccess)
    return LATENTMOE_ERR_CUDA;
  return LATENTMOE_OK;
}

// ---------------------------------------------------------------- debug GEMM
int latentmoe_debug_status(uint32_t* device_status);

namespace {
unsigned* debug_status_word() {
  static unsigned* p = nullptr;
  if (p == nullptr) {
    if (cudaMalloc(&p, 16) != cudaSuccess) return nullptr;
    cudaMemset(p, 0, 16);
  }
  return p;
}

int debug_gemm_impl(const void* A, const void* B, void* C, const int32_t* offsets, int64_t G,
                    int64_t M, int64_t N, int64_t K, int mode_bits, cudaStream_t s) {
  const bool pair = (mode_bits & 4) != 0;
  const int mode = mode_bits & ~4;
  if (!A || !B || !C || M < 1 || N < 1 || K < 1 || mode < 0 || mode > 2 ||
      (pair && offsets != nullptr && mode == 1))
    return LATENTMOE_ERR_INVALID_ARG;
  if (pair && offsets && ((mode == 2 && N % 256) || (mode == 0 && N % 512)))
    return LATENTMOE_ERR_UNSUPPORTED;
  if (K % 128 || (mode != 1 && N % 128) || M > (1 << 30) || N > (1 << 20))
    return LATENTMOE_ERR_UNSUPPORTED;
  if (offsets && (G < 1 || G > lmoe::kMaxGroups)) return LATENTMOE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return LATENTMOE_ERR_UNSUPPORTED;
  unsigned* status = debug_status_word();
  if (status == nullptr) return LATENTMOE_ERR_CUDA;
  const int64_t groups = offsets ? G : 1;
  if (offsets && mode != 1) {
    // the grouped kernel reads packed weight tiles: pack B into a temporary
    const long long brows = groups * N * (mode == 2 ? 2 : 1);
    __nv_bfloat16* bp = nullptr;
    if (cudaMalloc(&bp, brows * K * 2) != cudaSuccess) {
      cudaGetLastError();
      return LATENTMOE_ERR_OUT_OF_MEMORY;
    }
    if (lmoe::launch_pack_tiles(B, bp, brows, K * 2, num_sms(), s) != cudaSuccess) {
      cudaFree(bp);
      return LATENTMOE_ERR_CUDA;
    }
    const uint64_t tiles_half = static_cast<uint64_t>(groups * N / 128 * (K / lmoe::kGBK));
    CUtensorMap tok, w0, w1;
    bool ok = make_token_map(&tok, A, M, K);
    ok &= make_tile_map(&w0, bp, tiles_half);
    if (mode == 2)
      ok &= make_tile_map(&w1, bp + groups * N * K, tiles_half);
    else
      w1 = w0;
    if (!ok) {
      cudaFree(bp);
      return LATENTMOE_ERR_CUDA;
    }
    lmoe::GroupedArgs ga;
    memset(&ga, 0, sizeof(ga));
    ga.num_groups = static_cast<int>(groups);
    ga.seg_offsets = offsets;
    ga.fblocks = mode == 2 ? static_cast<int>(N / 128) : ceil_div(N, 256);
    ga.kb = static_cast<int>(K / lmoe::kGBK);
    ga.w_group_rows = static_cast<int>(N);
    ga.n_out = static_cast<int>(N);
    ga.out = C;
    ga.ldo = N;
    ga.out_rows = M;
    ga.status = status;
    cudaError_t e;
    if (pair) {
      ga.fblocks = static_cast<int>(mode == 2 ? N / 256 : N / 512);
      ga.tile_counter = reinterpret_cast<int*>(status) + 2;
      e = cudaMemsetAsync(ga.tile_counter, 0, 2 * sizeof(int), s);
      if (e == cudaSuccess)
        e = lmoe::launch_gemm_grouped_pair(mode == 2 ? lmoe::kGrpSwiglu : lmoe::kGrpPlain, false,
                                         tok, w0, w1, ga, num_sms(), s);
    } else {
      e = lmoe::launch_gemm_grouped(mode == 2 ? lmoe::kGrpSwiglu : lmoe::kGrpPlain, false, tok,
                                    w0, w1, ga, num_sms(), s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(bp);
    return e == cudaSuccess ? LATENTMOE_OK : LATENTMOE_ERR_CUDA;
  }
  GemmMaps m;
  bool ok = make_map(&m.a, A, M, K, K, 128);
  if (mode == 2) {
    ok &= make_map(&m.b, B, groups * N, K, K, 128);
    ok &= make_map(&m.bu, static_cast<const __nv_bfloat16*>(B) + groups * N * K, groups * N, K,
                   K, 128);
  } else {
    ok &= make_map(&m.b, B, groups * N, K, K, 128);
    m.bu = m.b;
  }
  if (!ok) return LATENTMOE_ERR_CUDA;
  m.a2 = m.a;
  m.b2 = m.b;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.grouped = offsets ? 1 : 0;
  a.num_groups = static_cast<int>(groups);
  a.seg_offsets = offsets;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.n_tiles = mode == 2 ? static_cast<int>(N / 128) : ceil_div(N, lmoe::kBN);
  a.kb1 = static_cast<int>(K / lmoe::kBK);
  a.b_group_rows = static_cast<int>(N);
  a.group_m = 16;
  a.out = C;
  a.ldo = N;
  a.out_rows = M;
  a.status = status;
  const long long tiles = static_cast<long long>(ceil_div(M, lmoe::kBM)) * a.n_tiles;
  const int grid = offsets ? num_sms() : static_cast<int>(tiles < num_sms() ? tiles : num_sms());
  const int pair_sms = pair ? num_sms() : 0;
  cudaError_t e;
  if (mode == 0) e = lmoe::launch_gemm_bf16(m, a, grid, false, s, false, pair_sms);
  else if (mode == 1) e = lmoe::launch_gemm_f32(m, a, grid, false, s, false, pair_sms);
  else e = lmoe::launch_gemm_swiglu(m, a, grid, s, false, pair_sms);
  return e == cudaSuccess ? LATENTMOE_OK : LATENTMOE_ERR_CUDA;
}
}  // namespace

int latentmoe_debug_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         int mode, latentmoe_stream_t st) {
  return debug_gemm_impl(A, B, C, nullptr, 1, M, N, K, mode, reinterpret_cast<cudaStream_t>(st));
}

int latentmoe_debug_grouped_gemm(const void* A, const void* B, void* C, const int32_t* offsets,
                                 int64_t groups, int64_t M, int64_t N, int64_t K, int mode,
                                 latentmoe_stream_t st) {
  if (offsets == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  return debug_gemm_impl(A, B, C, offsets, groups, M, N, K, mode,
                         reinterpret_cast<cudaStream_t>(st));
}

int latentmoe_debug_grouped_gemm_e4m3(const uint8_t* A, const uint8_t* B, const float* scales,
                                      void* C, uint32_t* amax, const int32_t* offsets,
                                      int64_t G, int64_t M, int64_t N, int64_t K, int mode_bits,
                                      latentmoe_stream_t st) {
  const bool pair = (mode_bits & 4) != 0;
  const int mode = mode_bits & ~4;
  if (!A || !B || !scales || !C || !offsets || M < 1 || N < 1 || K < 1 || G < 1 ||
      (mode != 1 && mode != 2) || (mode == 2 && amax == nullptr))
    return LATENTMOE_ERR_INVALID_ARG;
  if (pair && ((mode == 2 && N % 256) || (mode == 1 && N % 512))) return LATENTMOE_ERR_UNSUPPORTED;
  if (K % 128 || N % 128 || M > (1 << 30) || N > (1 << 20) || G > lmoe::kMaxGroups)
    return LATENTMOE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u) || (reinterpret_cast<uintptr_t>(amax) & 3u))
    return LATENTMOE_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(st);
  unsigned* status = debug_status_word();
  if (status == nullptr) return LATENTMOE_ERR_CUDA;
  const long long brows = G * N * (mode == 2 ? 2 : 1);
  uint8_t* bp = nullptr;
  if (cudaMalloc(&bp, brows * K) != cudaSuccess) {
    cudaGetLastError();
    return LATENTMOE_ERR_OUT_OF_MEMORY;
  }
  if (lmoe::launch_pack_tiles(B, bp, brows, K, num_sms(), s) != cudaSuccess) {
    cudaFree(bp);
    return LATENTMOE_ERR_CUDA;
  }
  const uint64_t tiles_half = static_cast<uint64_t>(G * N / 128 * (K / 128));
  CUtensorMap tok, w0, w1;
  bool ok = make_token_map(&tok, A, M, K, true);
  ok &= make_tile_map(&w0, bp, tiles_half, true);
  if (mode == 2)
    ok &= make_tile_map(&w1, bp + G * N * K, tiles_half, true);
  else
    w1 = w0;
  if (!ok) {
    cudaFree(bp);
    return LATENTMOE_ERR_CUDA;
  }
  lmoe::GroupedArgs ga;
  memset(&ga, 0, sizeof(ga));
  ga.num_groups = static_cast<int>(G);
  ga.seg_offsets = offsets;
  ga.fblocks = mode == 2 ? static_cast<int>(N / 128) : ceil_div(N, 256);
  ga.kb = static_cast<int>(K / lmoe::kGBK8);
  ga.w_group_rows = static_cast<int>(N);
  ga.n_out = static_cast<int>(N);
  ga.out = C;
  ga.ldo = N;
  ga.out_rows = M;
  ga.status = status;
  ga.in_scale = scales;
  ga.out_scale = scales + 1;
  ga.w_scale0 = scales + 2;
  ga.w_scale1 = mode == 2 ? scales + 2 + G : scales + 2;
  ga.out_amax = amax;
  cudaError_t e;
  if (pair) {
    ga.fblocks = static_cast<int>(mode == 2 ? N / 256 : N / 512);
    e = lmoe::launch_gemm_grouped_pair(mode == 2 ? lmoe::kGrpSwiglu : lmoe::kGrpPlain, true, tok,
                                       w0, w1, ga, num_sms(), s);
  } else {
    e = lmoe::launch_gemm_grouped(mode == 2 ? lmoe::kGrpSwiglu : lmoe::kGrpPlain, true, tok, w0,
                                  w1, ga, num_sms(), s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFree(bp);
  return e == cudaSuccess ? LATENTMOE_OK : LATENTMOE_ERR_CUDA;
}

namespace {
// One thread waits, with the library's bounded wait, on an mbarrier that
// nothing ever arrives on; the wait gives up after limit_ns and records it.
__global__ void wait_timeout_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    lmoe::mbar_init(&bar, 1);
    abort_flag = 0;
    lmoe::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) lmoe::wait_bounded(&bar, 0, &abort_flag, status, limit_ns);
}
}  // namespace

int latentmoe_debug_wait_timeout(uint64_t limit_ns, uint32_t* device_status) {
  if (device_status == nullptr || limit_ns > 1000000000ull) return LATENTMOE_ERR_INVALID_ARG;
  unsigned* p = debug_status_word();
  if (p == nullptr) return LATENTMOE_ERR_CUDA;
  wait_timeout_kernel<<<1, 32>>>(p, limit_ns);
  if (cudaGetLastError() != cudaSuccess) return LATENTMOE_ERR_CUDA;
  return latentmoe_debug_status(device_status);
}

int latentmoe_debug_status(uint32_t* device_status) {
  if (device_status == nullptr) return LATENTMOE_ERR_INVALID_ARG;
  unsigned* p = debug_status_word();
  if (p == nullptr) return LATENTMOE_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return LATENTMOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LATENTMOE_ERR_CUDA;
  cudaMemset(p, 0, 4);
  *device_status = v;
  if (v & LATENTMOE_STATUS_TIMEOUT) return LATENTMOE_ERR_TIMEOUT;
  return v ? LATENTMOE_ERR_DEVICE_STATUS : LATENTMOE_OK;
}

}  // extern "C"
