// Grouped tcgen05 GEMM for the expert FFNs, weights on the M side.
//
// For each expert e with n_e slots, the product is computed transposed:
// D[feature, token] = W[feature, :] . Z[token, :], with M = 128 weight rows
// and N = the expert's tokens (a multiple of 16, at most 256 per tile). Token
// counts are only padded to 16, not to a 128-row tile, and one weight tile is
// read once for all tokens of an expert (n_e <= 256) or for each 256-token
// chunk (more tokens).
//
// Weights are read from the packed layout made by pack_weight_tiles: every
// 128-row x 64-column tile is one contiguous 16 KB block, so the weight
// stream reaches HBM as sequential reads instead of 128-byte pieces of rows
// 6-20 KB apart.
//
// Each tile uses two accumulators that share one token tile in shared
// memory: (gate, up) rows of the same 128 features for the SwiGLU GEMM, or
// two consecutive 128-row blocks of W_d for the down GEMM. Together they
// fill TMEM (2 x 256 columns), and a k-block moves 64 KB of shared memory for
// 2 x 128 x 256 x 64 MACs.
//
//   warp 0      TMA producer (one lane): two packed weight tiles, then the
//               token rows in 64-row boxes
//   warp 1      TMEM owner and MMA issuer (one lane)
//   warps 2..9  epilogue: warp w reads TMEM lanes [32*(w%4), +32) and every
//               other 32-token chunk; rows are transposed through shared
//               memory so each output row segment is one 64-byte store
//
// Accumulators are single-buffered: the MMA of the next tile waits for the
// epilogue, but the producer keeps filling the stage ring meanwhile, so the
// memory system stays busy; the kernel is bound by the weight stream.
//
// Tiles are enumerated on the device from the segment offsets: expert-major,
// then feature block, then token chunk, so chunks of one feature block run
// on neighbouring CTAs at the same time and share the weight tile in L2.
//
// E4M3 variant (F8 = true): weights and token rows are FP8 codes, a k-block
// is 128 elements (still one 128-byte swizzle row, so tiles, stages and
// descriptors are byte-for-byte the same) and the MMA is kind::f8f6f4 with
// K = 32 per instruction. The epilogue multiplies the accumulators by the
// token scale times the group's weight scale; the SwiGLU epilogue then
// records max |h| and writes h as E4M3 codes with the scale given for it
// ("The Training and RL Infrastructure Behind MAI-Thinking-1", section
// "2. Numerics": FP8 forward GEMMs with delayed scaling).
#pragma once

#include "fp8.cuh"
#include "ptx.cuh"

namespace lmoe {

enum GroupedMode : int { kGrpSwiglu = 0, kGrpPlain = 1 };

constexpr int kGBK = 64;                      // one 128-byte swizzle row
constexpr int kGBK8 = 128;                    // E4M3: one 128-byte swizzle row
constexpr int kGStages = 3;
constexpr int kGWeightTile = 128 * kGBK * 2;  // 16 KB
constexpr int kGTokenTile = 256 * kGBK * 2;   // 32 KB
constexpr int kGStageBytes = 2 * kGWeightTile + kGTokenTile;
constexpr int kGTokBox = 64;                  // token rows per TMA box
constexpr int kGTokBoxBytes = kGTokBox * kGBK * 2;
constexpr int kGMaxTok = 256;
constexpr int kGEpiWarps = 8;
constexpr int kGThreads = 64 + 32 * kGEpiWarps;
constexpr int kGBarrierBytes = 8 * (2 * kGStages + 3);
constexpr int kGStagePitch = 80;              // 64 B of bf16 + 16 B pad per token row
constexpr int kGStageWarpBytes = 32 * kGStagePitch;
constexpr int kGMaxGroups = 512;
// group table: first input row, first output row, rows, tile prefix
constexpr int kGTableBytes = (4 * kGMaxGroups + 1) * 4;
constexpr int kGSmemBytes = 1024 + kGStages * kGStageBytes + kGBarrierBytes + 16 + kGTableBytes +
                            16 /* staging alignment */ + kGEpiWarps * kGStageWarpBytes;

struct GroupedArgs {
  int num_groups;          // G <= kGMaxGroups
  const int* seg_offsets;  // [G+1] row offsets of the groups (input rows = output rows),
                           // used when seg_len is null
  const int* seg_len;      // [G] rows of each group, or null
  const int* in_start;     // [G] first token row of each group (with seg_len)
  const int* out_start;    // [G] first output row of each group (with seg_len)
  int fblocks;             // feature blocks per group (SwiGLU: F/128; plain: ceil(N/256))
  int kb;                  // k-blocks (K / 64)
  int w_group_rows;        // weight rows per group in the weight maps
  int n_out;               // output features (columns of out)
  void* out;               // bf16 [rows, n_out] (E4M3 SwiGLU: codes; plain with out_f32:
                           // fp32), rows in slot order
  long long ldo;
  long long out_rows;      // rows of the buffer out points to (bounds-checked build)
  int out_f32;             // plain: fp32 output
  unsigned* status;
  int* tile_counter;       // SM-pair kernel: [2] {tile counter, exit count}, both zero at
                           // launch and left zero by it; tiles past the first wave are
                           // taken from [0] (null: static round robin)
  // E4M3 variant only
  const float* w_scale0;   // [G] scale of the weights of accumulator 0, per group
  const float* w_scale1;   // [G] accumulator 1 (SwiGLU: the up rows)
  const float* in_scale;   // [1] scale of the token rows
  const float* out_scale;  // [1] SwiGLU: scale h is quantized with
  unsigned* out_amax;      // [1] SwiGLU: running max |h| (float bits)
};

struct GTile {
  int g;      // group
  int tok0;   // first token row
  int out0;   // first output row
  int len;    // valid tokens (<= 256)
  int n;      // MMA N: len rounded up to 16
  int f;      // feature block
  int wrow;   // first weight row of accumulator 0
};

__device__ __forceinline__ void group_chunks(int n, int& nch, int& cs) {
  nch = (n + kGMaxTok - 1) / kGMaxTok;
  const int per = (n + nch - 1) / nch;
  cs = (per + 15) & ~15;
}

// Group table in shared memory (kGTableBytes): per group its first input
// row, first output row and row count, then the exclusive prefix of tiles.
struct GroupTable {
  int* in;
  int* out;
  int* len;
  int* tp;
};

// The epilogue staging rows start on the next 16-byte boundary after the table.
__device__ __forceinline__ uint8_t* staging_after_table(void* table) {
  const uintptr_t p = reinterpret_cast<uintptr_t>(table) + kGTableBytes;
  return reinterpret_cast<uint8_t*>((p + 15) & ~static_cast<uintptr_t>(15));
}

__device__ __forceinline__ GroupTable group_table_at(void* p) {
  int* b = static_cast<int*>(p);
  return GroupTable{b, b + kGMaxGroups, b + 2 * kGMaxGroups, b + 3 * kGMaxGroups};
}

__device__ __forceinline__ void load_group_table(const GroupedArgs& a, const GroupTable& gt) {
  for (int i = threadIdx.x; i < a.num_groups; i += blockDim.x) {
    if (a.seg_len != nullptr) {
      gt.in[i] = a.in_start[i];
      gt.out[i] = a.out_start[i];
      gt.len[i] = a.seg_len[i];
    } else {
      const int s0 = a.seg_offsets[i];
      gt.in[i] = s0;
      gt.out[i] = s0;
      gt.len[i] = a.seg_offsets[i + 1] - s0;
    }
  }
}

// Exclusive prefix over groups of (token chunks x tiles per chunk), by one warp.
__device__ __forceinline__ void build_tile_prefix(const GroupedArgs& a, const GroupTable& gt,
                                                  int tiles_per_chunk) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  if (lane == 0) gt.tp[0] = 0;
  for (int base = 0; base < a.num_groups; base += 32) {
    const int g = base + lane;
    int v = 0;
    if (g < a.num_groups) {
      const int n = gt.len[g];
      if (n > 0) {
        int nch, cs;
        group_chunks(n, nch, cs);
        v = nch * tiles_per_chunk;
      }
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (g < a.num_groups) gt.tp[g + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
}

// The group of tile t: the largest g with tp[g] <= t (that group is non-empty).
__device__ __forceinline__ int tile_group(int t, const GroupedArgs& a, const GroupTable& gt) {
  int lo = 0, hi = a.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gt.tp[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int MODE>
__device__ __forceinline__ GTile decode_gtile(int t, const GroupedArgs& a, const GroupTable& gt) {
  const int g = tile_group(t, a, gt);
  const int n = gt.len[g];
  int nch, cs;
  group_chunks(n, nch, cs);
  const int local = t - gt.tp[g];
  const int f = local / nch;
  const int c = local - f * nch;
  GTile r;
  r.g = g;
  r.tok0 = gt.in[g] + c * cs;
  r.out0 = gt.out[g] + c * cs;
  r.len = min(cs, n - c * cs);
  r.n = (r.len + 15) & ~15;
  r.f = f;
  r.wrow = g * a.w_group_rows + f * (MODE == kGrpSwiglu ? 128 : 256);
  return r;
}

template <int MODE>
__device__ __forceinline__ bool second_acc_used(const GroupedArgs& a, int f) {
  return MODE == kGrpSwiglu || (f * 256 + 128 < a.n_out);
}

// Transpose one 32-token x 32-feature chunk (p: this lane's feature for 32
// tokens, bf16 pairs (token 2j, 2j+1) in p[j]) through the warp's staging rows
// and store 64 contiguous bytes per token row. Tokens at or past `tok_valid`
// are not stored.
// HINT: the stores carry the L2 eviction policy pol.
template <bool HINT = false>
__device__ __forceinline__ void gstore_chunk(const GroupedArgs& a, const uint32_t (&p)[16],
                                             uint8_t* stage, long long tok_row0, int tok_valid,
                                             int feat0, uint64_t pol = 0) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    *reinterpret_cast<uint16_t*>(stage + (2 * j) * kGStagePitch + lane * 2) =
        static_cast<uint16_t>(p[j] & 0xffffu);
    *reinterpret_cast<uint16_t*>(stage + (2 * j + 1) * kGStagePitch + lane * 2) =
        static_cast<uint16_t>(p[j] >> 16);
  }
  __syncwarp();
  const int piece = lane & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int rr = q * 8 + (lane >> 2);
    const uint4 w = *reinterpret_cast<const uint4*>(stage + rr * kGStagePitch + piece * 16);
    if (rr < tok_valid && in_bounds(tok_row0 + rr, a.out_rows, a.status)) {
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                            (tok_row0 + rr) * a.ldo + feat0 + piece * 8);
      if constexpr (HINT)
        st_global_u4_hint(dst, w, pol);
      else
        *dst = w;
    }
  }
  __syncwarp();
}

// E4M3 form of gstore_chunk: lane `lane` holds the codes of its feature for
// 32 tokens (token 4j+b in byte b of q[j]). Each token row segment is 32
// bytes; pieces are XOR-swizzled by (row / 4) so that both the byte writes
// and the 16-byte reads are free of bank conflicts.
// fp32 output of one 32-token chunk: for each token the warp's 32 lanes hold
// 32 consecutive features, one 128-byte store per token row.
__device__ __forceinline__ void gstore_chunk_f32(const GroupedArgs& a, const uint32_t (&v)[32],
                                                 float scale, long long tok_row0, int tok_valid,
                                                 int feat0) {
  const int lane = threadIdx.x & 31;
  float* out = static_cast<float*>(a.out) + feat0 + lane;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < tok_valid && in_bounds(tok_row0 + j, a.out_rows, a.status))
      out[(tok_row0 + j) * a.ldo] = __uint_as_float(v[j]) * scale;
}

template <bool HINT = false>
__device__ __forceinline__ void gstore_chunk_f8(const GroupedArgs& a, const uint32_t (&q)[8],
                                                uint8_t* stage, long long tok_row0,
                                                int tok_valid, int feat0, uint64_t pol = 0) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int sw = ((lane >> 4) ^ ((j >> 2) & 1)) * 16 + (lane & 15);
    stage[j * 32 + sw] = static_cast<uint8_t>(q[j >> 2] >> (8 * (j & 3)));
  }
  __syncwarp();
  const int piece = lane & 1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rr = h * 16 + (lane >> 1);
    const uint4 w =
        *reinterpret_cast<const uint4*>(stage + rr * 32 + ((piece ^ ((rr >> 2) & 1)) * 16));
    if (rr < tok_valid && in_bounds(tok_row0 + rr, a.out_rows, a.status)) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                            (tok_row0 + rr) * a.ldo + feat0 + piece * 16);
      if constexpr (HINT)
        st_global_u4_hint(dst, w, pol);
      else
        *dst = w;
    }
  }
  __syncwarp();
}

// One tile's epilogue for one epilogue warp, shared by the single-SM and the
// SM-pair kernels. The warp owns TMEM lanes [32 * quarter, +32) (lane_off)
// and the 32-token chunks half, half + 2, ... of the tile's len tokens
// (len <= 256, or <= 512 for a plain tile with one accumulator).
//   SwiGLU: h = SiLU(s_g acc0) * (s_u acc1) for output features
//           [feat0, +32), written as bf16 or (F8) E4M3 codes with max |h| of the
//           valid tokens folded into amax; TMEM is released before the stores.
//   plain:  acc0 and acc1 (when `two`) scaled by s_w and written to features
//           feat0 and feat1 (each only if below n_out), bf16 or fp32; TMEM is
//           released after the stores.
// release() hands TMEM back to the MMA issuer. HINT (SwiGLU): h is stored with
// the L2 eviction policy store_pol.
template <int MODE, bool F8, bool HINT = false, typename Release>
__device__ __forceinline__ void grouped_tile_epilogue(const GroupedArgs& a, uint32_t tmem_lanes,
                                                      int half, int g, int len, long long out0,
                                                      int feat0, int feat1, bool two,
                                                      float in_s, float out_inv, float& amax,
                                                      uint8_t* stage_w, Release release,
                                                      uint64_t store_pol = 0) {
  const int nchunks = (len + 31) / 32;
  if constexpr (MODE == kGrpSwiglu && F8) {
    // gate scale with SiLU's halving folded in (exact)
    const float sg_half = 0.5f * (in_s * a.w_scale0[g]), su = in_s * a.w_scale1[g];
    // the same 16-column software pipeline as the bf16 path below
    uint32_t hq[4][8];
    uint32_t gv[2][16], uv[2][16];
    tmem_ld_16cols(tmem_lanes + half * 32, gv[0]);
    tmem_ld_16cols(tmem_lanes + 256 + half * 32, uv[0]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = q >> 1, ch = half + 2 * i;
      if (ch >= nchunks) break;
      const int qn = q + 1, chn = half + 2 * (qn >> 1);
      if (qn < 8 && chn < nchunks) {
        const uint32_t col = chn * 32 + (qn & 1) * 16;
        tmem_ld_16cols(tmem_lanes + col, gv[qn & 1]);
        tmem_ld_16cols(tmem_lanes + 256 + col, uv[qn & 1]);
      }
      const int valid = len - ch * 32 - (q & 1) * 16;
      float hv[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        hv[j] = silu_from_half(__uint_as_float(gv[q & 1][j]) * sg_half) *
                (__uint_as_float(uv[q & 1][j]) * su);
        if (j < valid) amax = fmaxf(amax, fabsf(hv[j]));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        hq[i][(q & 1) * 4 + j] =
            quant4_e4m3(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3], out_inv);
      tmem_ld_wait();
    }
    release();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = half + 2 * i;
      if (ch < nchunks)
        gstore_chunk_f8<HINT>(a, hq[i], stage_w, out0 + ch * 32, len - ch * 32, feat0, store_pol);
    }
  } else if constexpr (MODE == kGrpSwiglu) {
    // h for this warp's chunks (at most 4) packed to bf16 in registers, then
    // TMEM goes back to the MMA before the slower transposing stores. The
    // chunks are read in 16-column halves, software-pipelined: the loads of
    // half q + 1 are in flight while half q's SiLU * up is formed, so the
    // TMEM reads and the arithmetic of the hold overlap.
    uint32_t hp[4][16];
    uint32_t gv[2][16], uv[2][16];
    tmem_ld_16cols(tmem_lanes + half * 32, gv[0]);
    tmem_ld_16cols(tmem_lanes + 256 + half * 32, uv[0]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = q >> 1, ch = half + 2 * i;
      if (ch >= nchunks) break;
      const int qn = q + 1, chn = half + 2 * (qn >> 1);
      if (qn < 8 && chn < nchunks) {
        const uint32_t col = chn * 32 + (qn & 1) * 16;
        tmem_ld_16cols(tmem_lanes + col, gv[qn & 1]);
        tmem_ld_16cols(tmem_lanes + 256 + col, uv[qn & 1]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        hp[i][(q & 1) * 8 + j] =
            pack_bf16x2(silu(__uint_as_float(gv[q & 1][2 * j])) * __uint_as_float(uv[q & 1][2 * j]),
                        silu(__uint_as_float(gv[q & 1][2 * j + 1])) *
                            __uint_as_float(uv[q & 1][2 * j + 1]));
      tmem_ld_wait();
    }
    release();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = half + 2 * i;
      if (ch < nchunks)
        gstore_chunk<HINT>(a, hp[i], stage_w, out0 + ch * 32, len - ch * 32, feat0, store_pol);
    }
  } else {
    const float so = F8 ? in_s * a.w_scale0[g] : 1.0f;
    for (int ch = half; ch < nchunks; ch += 2) {
      const long long row0 = out0 + ch * 32;
      const int valid = len - ch * 32;
#pragma unroll 1
      for (int acc = 0; acc < 2; ++acc) {
        if (acc == 1 && !two) break;
        const int feat = acc == 0 ? feat0 : feat1;
        if (feat >= a.n_out) continue;
        uint32_t v[32];
        tmem_ld_32cols(tmem_lanes + acc * 256 + ch * 32, v);
        tmem_ld_wait();
        if (a.out_f32) {
          gstore_chunk_f32(a, v, so, row0, valid, feat);
          continue;
        }
        uint32_t o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          o[j] =
              pack_bf16x2(__uint_as_float(v[2 * j]) * so, __uint_as_float(v[2 * j + 1]) * so);
        gstore_chunk(a, o, stage_w, row0, valid, feat);
      }
    }
    release();
  }
}

template <int MODE, bool F8>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_grouped_kernel(const __grid_constant__ CUtensorMap tmTok,
                        const __grid_constant__ CUtensorMap tmW0,
                        const __grid_constant__ CUtensorMap tmW1, const GroupedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kGStages * kGStageBytes);
  uint64_t* empty_bar = full_bar + kGStages;
  uint64_t* tfull_bar = empty_bar + kGStages;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* done_bar = tempty_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const GroupTable gt = group_table_at(tmem_slot + 4);
  uint8_t* stage_smem = staging_after_table(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 32 * kGEpiWarps);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmTok);
    tma_prefetch_desc(&tmW0);
    tma_prefetch_desc(&tmW1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // nothing above reads global memory: the set-up overlaps the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  load_group_table(a, gt);
  __syncthreads();
  if (warp == 2) build_tile_prefix(a, gt, a.fblocks);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = gt.tp[a.num_groups];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      // Weights come from the packed layout: tile (row tile rt, k-block kb)
      // is one contiguous 16 KB block at index rt * kb_count + kb.
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_t = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const GTile c = decode_gtile<MODE>(t, a, gt);
        const bool two = second_acc_used<MODE>(a, c.f);
        const int nbox = (c.n + kGTokBox - 1) / kGTokBox;
        const uint32_t bytes = kGWeightTile * (two ? 2 : 1) + nbox * kGTokBoxBytes;
        const int rt0 = c.wrow / 128;
        for (int kb = 0; kb < a.kb; ++kb) {
          if (!wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* sw0 = tiles + stage * kGStageBytes;
          uint8_t* sw1 = sw0 + kGWeightTile;
          uint8_t* stok = sw1 + kGWeightTile;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          tma_load_3d(&tmW0, &full_bar[stage], sw0, 0, 0, rt0 * a.kb + kb, pol_w);
          if (two) {
            if (MODE == kGrpSwiglu)
              tma_load_3d(&tmW1, &full_bar[stage], sw1, 0, 0, rt0 * a.kb + kb, pol_w);
            else
              tma_load_3d(&tmW0, &full_bar[stage], sw1, 0, 0, (rt0 + 1) * a.kb + kb, pol_w);
          }
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(&tmTok, &full_bar[stage], stok + b * kGTokBoxBytes,
                        kb * (F8 ? kGBK8 : kGBK), c.tok0 + b * kGTokBox, pol_t);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < kGStages; ++s)
        if (issued_mask & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const GTile c = decode_gtile<MODE>(t, a, gt);
        const bool two = second_acc_used<MODE>(a, c.f);
        const uint32_t idesc = F8 ? instr_desc_e4m3(128, c.n) : instr_desc_bf16(128, c.n);
        if (!wait_bounded(tempty_bar, acc_phase ^ 1u, abort_flag, a.status)) break;
        tc_fence_after_sync();
        for (int kb = 0; kb < a.kb; ++kb) {
          if (!wait_bounded(&full_bar[stage], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint8_t* sw0 = tiles + stage * kGStageBytes;
          const uint64_t d0 = smem_desc_sw128(sw0);
          const uint64_t d1 = smem_desc_sw128(sw0 + kGWeightTile);
          const uint64_t dt = smem_desc_sw128(sw0 + 2 * kGWeightTile);
          // 4 instructions per 128-byte row, each 32 bytes of K (+2 in addr >> 4)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
            if constexpr (F8) {
              tc_mma_f8(tmem_base, d0 + 2ull * k, dt + 2ull * k, idesc, accum);
              if (two) tc_mma_f8(tmem_base + 256, d1 + 2ull * k, dt + 2ull * k, idesc, accum);
            } else {
              tc_mma(tmem_base, d0 + 2ull * k, dt + 2ull * k, idesc, accum);
              if (two) tc_mma(tmem_base + 256, d1 + 2ull * k, dt + 2ull * k, idesc, accum);
            }
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar);
        acc_phase ^= 1u;
      }
      tc_commit(done_bar);
      wait_drain(done_bar, 0);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stage_w = stage_smem + (warp - 2) * kGStageWarpBytes;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc_phase = 0;
    const float in_s = F8 ? *a.in_scale : 1.0f;
    const float out_inv = (F8 && MODE == kGrpSwiglu) ? inv_scale(*a.out_scale) : 1.0f;
    float amax = 0.0f;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const GTile c = decode_gtile<MODE>(t, a, gt);
      const bool two = second_acc_used<MODE>(a, c.f);
      if (!warp_wait_bounded(tfull_bar, acc_phase, abort_flag, a.status)) break;
      tc_fence_after_sync();
      const int feat0 =
          MODE == kGrpSwiglu ? c.f * 128 + quarter * 32 : c.f * 256 + quarter * 32;
      grouped_tile_epilogue<MODE, F8>(a, tmem_base + lane_off, half, c.g, c.len, c.out0, feat0,
                                      feat0 + 128, two, in_s, out_inv, amax, stage_w, [&] {
                                        tc_fence_before_sync();
                                        mbar_arrive(tempty_bar);
                                      });
      acc_phase ^= 1u;
    }
    if constexpr (F8 && MODE == kGrpSwiglu) {
      amax = warp_max(amax);
      if (lane == 0) atomic_max_nonneg(a.out_amax, amax);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace lmoe
