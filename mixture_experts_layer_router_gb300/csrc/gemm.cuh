// Persistent tcgen05 GEMM, D = A B^T, for every matrix product of the layer.
//
// A [rows, K] and B [N, K] are bf16, K-major (nn.Linear layout), read by TMA
// into a ring of shared-memory stages with 128-byte swizzle (every map reads
// boxes of 128 rows; a 256-row B tile is two boxes). One thread
// issues tcgen05.mma (M = 128, N = 256, K = 16 per instruction) into one of
// two fp32 accumulators in tensor memory (2 x 256 columns); eight epilogue
// warps drain the other accumulator meanwhile, apply the epilogue and store.
//
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator and MMA issuer (one lane)
//   warps 2..9  epilogue; warp w reads TMEM lanes [32*(w%4), 32*(w%4)+32)
//               and every other 32-column chunk (warps 2..5 the even ones),
//               so two warps share the stores of each row quarter (the
//               scatter epilogue writes each row k times)
//
// Tiles: dense GEMMs walk (m, n) in bands of `group_m` m-tiles so that
// concurrent CTAs share A rows and B columns in L2. Grouped GEMMs (the
// expert FFNs) take the expert segments [seg[g], seg[g+1]) of A's rows from
// device memory; every CTA builds the prefix of m-tiles per group in shared
// memory and walks (group, n, m) with m fastest, so the CTAs working on the
// two or three m-tiles of one expert read each weight tile at about the same
// time. No host synchronisation is needed to know the segment sizes.
//
// Epilogues:
//   kEpiBf16     C[row, col] = bf16(acc)
//   kEpiF32      C[row, col] = acc (+ bias[col])
//   kEpiSwiglu   B holds 128 gate rows then 128 up rows of the same output
//                features; C[row, f] = bf16(SiLU(gate) * up)
//   kEpiScatter  token row t is written to rows pos[t*k + j], j < k, of C
//   kEpiScatterF8  the same with C as E4M3 codes of acc / out_scale, and the
//                running max |acc| of the valid rows recorded in out_amax
//   kEpiSwigluF8 the SwiGLU epilogue with C as E4M3 codes of h / out_scale
//                (max |h| of the valid rows recorded in out_amax)
//
// E4M3 operands (F8 = true): A and B are E4M3 codes, a k-block is 128 codes
// (still one 128-byte swizzle row), the MMA is kind::f8f6f4, and the
// accumulator is multiplied by a_scale * b_scale (SwiGLU: b_scale for the
// gate columns, b_scale2 for the up columns) before the epilogue. An fp32
// `addend` [rows, ld_add] is added to the scaled accumulator of kEpiBf16 /
// kEpiF32 before rounding (the shared expert's partial sum).
//
// Ragged edges: rows past a segment or past M are computed on whatever TMA
// brought in (zeros past the tensor) and never stored; columns past N are not
// stored either.
#pragma once

#include "fp8.cuh"
#include "ptx.cuh"

namespace lmoe {

enum EpiMode : int {
  kEpiBf16 = 0,
  kEpiF32 = 1,
  kEpiSwiglu = 2,
  kEpiScatter = 3,
  kEpiScatterF8 = 4,
  kEpiSwigluF8 = 5
};

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int kBK8 = 128;  // 128 E4M3 codes = one swizzle row
constexpr int kStages = 4;
constexpr int kATileBytes = kBM * kBK * 2;
constexpr int kBTileBytes = kBN * kBK * 2;
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kMaxGroups = 512;
constexpr int kGemmEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kGemmEpiWarps;
constexpr int kTmemCols = 2 * kBN;
constexpr int kBarrierBytes = 8 * (2 * kStages + 2 + 2 + 1);
// Epilogue staging: per epilogue warp, 32 rows x 64 bytes of bf16 output with
// a 16-byte pad per row (80-byte pitch keeps 16-byte accesses conflict-free).
constexpr int kStagePitch = 80;
constexpr int kStageWarpBytes = 32 * kStagePitch;
constexpr int kGemmSmemBytes =
    1024 /* alignment slack */ + kStages * kStageBytes + kBarrierBytes + 16 +
    2 * (kMaxGroups + 1) * 4 + kGemmEpiWarps * kStageWarpBytes;

struct GemmArgs {
  int grouped;             // 0: dense rows [0, M); 1: segments from seg_offsets
  int num_groups;          // G <= kMaxGroups (grouped)
  const int* seg_offsets;  // [G+1] row offsets of the segments (grouped)
  int M;                   // rows (dense)
  int N;                   // output columns (kEpiSwiglu: output features)
  int n_tiles;             // tiles along N
  int kb1;                 // k-blocks of the first (A, B) pair
  int kb2;                 // k-blocks of the second pair (dual-K only)
  int b_group_rows;        // rows of B per group (grouped)
  int group_m;             // dense raster band, in m-tiles
  void* out;
  long long ldo;           // row stride of out, elements
  long long out_rows;      // rows of the buffer out points to (bounds-checked build)
  const float* bias;       // kEpiF32, may be null
  const int* pos;          // kEpiScatter: [M * topk] destination rows (-1: skip)
  int topk;
  unsigned* status;        // device status word
  int hints;               // bit 0: A tiles evict_last in L2; bit 1: B tiles evict_first
  const float* out_scale;  // kEpiScatterF8 / kEpiSwigluF8: [1] scale the output is quantized with
  unsigned* out_amax;      // kEpiScatterF8 / kEpiSwigluF8: [1] running max (float bits)
  const float* a_scale;    // E4M3 operands: [1] scale of A
  const float* b_scale;    // E4M3 operands: [1] scale of B (SwiGLU: gate rows)
  const float* b_scale2;   // E4M3 SwiGLU: [1] scale of the up rows
  const float* addend;     // kEpiBf16 / kEpiF32: fp32 [rows, ld_add] added before rounding, or null
  long long ld_add;
};

struct TileCoord {
  int row0;  // first A row of the tile
  int rows;  // valid rows (<= kBM)
  int n;     // n-tile index
  int brow;  // first B row
};

__device__ __forceinline__ TileCoord decode_tile(int t, const GemmArgs& a, const int* seg_s,
                                                 const int* mt_s, int b_rows_per_tile) {
  TileCoord c;
  if (a.grouped) {
    // largest g with mt_s[g] * n_tiles <= t; that group is non-empty
    int lo = 0, hi = a.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mt_s[mid] * a.n_tiles <= t) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int mtg = mt_s[g + 1] - mt_s[g];
    const int local = t - mt_s[g] * a.n_tiles;
    const int n = local / mtg;
    const int m = local - n * mtg;
    const int seg0 = seg_s[g];
    const int len = seg_s[g + 1] - seg0;
    c.row0 = seg0 + m * kBM;
    c.rows = min(kBM, len - m * kBM);
    c.n = n;
    c.brow = g * a.b_group_rows + n * b_rows_per_tile;
  } else {
    const int mt = (a.M + kBM - 1) / kBM;
    const int per = a.group_m * a.n_tiles;
    const int band = t / per;
    const int first = band * a.group_m;
    const int gm = min(a.group_m, mt - first);
    const int local = t - band * per;
    const int m = first + local % gm;
    const int n = local / gm;
    c.row0 = m * kBM;
    c.rows = min(kBM, a.M - c.row0);
    c.n = n;
    c.brow = n * b_rows_per_tile;
  }
  return c;
}

// bf16 output of one 32-column chunk for the warp's 32 rows. Each lane packs
// its own row into the warp's staging rows, then the warp writes 8 rows per
// instruction with 4 lanes per row (64 contiguous bytes). Rows at or past
// `rows_valid` (relative to the warp's first row) are not stored; with
// kEpiScatter, row t goes to rows pos[t*k + j] of the output instead.
template <int MODE>
__device__ __forceinline__ void store_chunk_bf16_staged(const GemmArgs& a,
                                                        const uint32_t (&v)[32], uint8_t* stage,
                                                        long long warp_row0, int rows_valid,
                                                        int col) {
  const int lane = threadIdx.x & 31;
  uint4* mine = reinterpret_cast<uint4*>(stage + lane * kStagePitch);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
    w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
    w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
    w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
    mine[q] = w;
  }
  __syncwarp();
  const int piece = lane & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int rr = q * 8 + (lane >> 2);
    const uint4 w = *reinterpret_cast<const uint4*>(stage + rr * kStagePitch + piece * 16);
    if (rr < rows_valid) {
      const long long row = warp_row0 + rr;
      if constexpr (MODE == kEpiScatter) {
        for (int j = 0; j < a.topk; ++j) {
          const int dst_row = a.pos[row * a.topk + j];
          if (dst_row < 0 || !in_bounds(dst_row, a.out_rows, a.status)) continue;
          *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                    static_cast<long long>(dst_row) * a.ldo + col + piece * 8) = w;
        }
      } else if (in_bounds(row, a.out_rows, a.status)) {
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * a.ldo + col +
                                  piece * 8) = w;
      }
    }
  }
  __syncwarp();
}

// E4M3 output of one 32-column chunk, scattered like kEpiScatter (or to the
// lane's own row when a.pos is null): each lane
// quantizes its row to 32 bytes, the warp stages them (16-byte pieces
// XOR-swizzled by row / 4, conflict-free both ways) and writes 16 rows per
// instruction, 2 lanes per row.
__device__ __forceinline__ void store_chunk_f8_scatter(const GemmArgs& a, const uint32_t (&v)[32],
                                                       float inv, uint8_t* stage,
                                                       long long warp_row0, int rows_valid,
                                                       int col) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint4 w;
    const int b = 16 * p;
    w.x = quant4_e4m3(__uint_as_float(v[b + 0]), __uint_as_float(v[b + 1]),
                      __uint_as_float(v[b + 2]), __uint_as_float(v[b + 3]), inv);
    w.y = quant4_e4m3(__uint_as_float(v[b + 4]), __uint_as_float(v[b + 5]),
                      __uint_as_float(v[b + 6]), __uint_as_float(v[b + 7]), inv);
    w.z = quant4_e4m3(__uint_as_float(v[b + 8]), __uint_as_float(v[b + 9]),
                      __uint_as_float(v[b + 10]), __uint_as_float(v[b + 11]), inv);
    w.w = quant4_e4m3(__uint_as_float(v[b + 12]), __uint_as_float(v[b + 13]),
                      __uint_as_float(v[b + 14]), __uint_as_float(v[b + 15]), inv);
    *reinterpret_cast<uint4*>(stage + lane * 32 + ((p ^ ((lane >> 2) & 1)) * 16)) = w;
  }
  __syncwarp();
  const int piece = lane & 1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rr = h * 16 + (lane >> 1);
    const uint4 w =
        *reinterpret_cast<const uint4*>(stage + rr * 32 + ((piece ^ ((rr >> 2) & 1)) * 16));
    if (rr < rows_valid) {
      const long long row = warp_row0 + rr;
      if (a.pos == nullptr) {
        if (in_bounds(row, a.out_rows, a.status))
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + row * a.ldo + col +
                                    piece * 16) = w;
      } else {
        for (int j = 0; j < a.topk; ++j) {
          const int dst_row = a.pos[row * a.topk + j];
          if (dst_row < 0 || !in_bounds(dst_row, a.out_rows, a.status)) continue;
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                    static_cast<long long>(dst_row) * a.ldo + col + piece * 16) = w;
        }
      }
    }
  }
  __syncwarp();
}

template <int MODE>
__device__ __forceinline__ void store_chunk(const GemmArgs& a, const uint32_t (&v)[32],
                                            long long row, int col) {
  if (MODE != kEpiScatter && !in_bounds(row, a.out_rows, a.status)) return;
  if constexpr (MODE == kEpiF32) {
    float* dst = reinterpret_cast<float*>(a.out) + row * a.ldo + col;
    if (col + 32 <= a.N && (a.ldo & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 f;
        f.x = __uint_as_float(v[i + 0]);
        f.y = __uint_as_float(v[i + 1]);
        f.z = __uint_as_float(v[i + 2]);
        f.w = __uint_as_float(v[i + 3]);
        if (a.bias != nullptr) {
          f.x += a.bias[col + i + 0];
          f.y += a.bias[col + i + 1];
          f.z += a.bias[col + i + 2];
          f.w += a.bias[col + i + 3];
        }
        *reinterpret_cast<float4*>(dst + i) = f;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (col + i < a.N) {
          float f = __uint_as_float(v[i]);
          if (a.bias != nullptr) f += a.bias[col + i];
          dst[i] = f;
        }
      }
    }
  } else {
    uint4 p[4];
    uint32_t* pw = reinterpret_cast<uint32_t*>(p);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pw[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    if constexpr (MODE == kEpiScatter) {
      for (int j = 0; j < a.topk; ++j) {
        const int dst_row = a.pos[row * a.topk + j];
        if (dst_row < 0 || !in_bounds(dst_row, a.out_rows, a.status)) continue;
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                              static_cast<long long>(dst_row) * a.ldo + col);
        dst[0] = p[0]; dst[1] = p[1]; dst[2] = p[2]; dst[3] = p[3];
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                            row * a.ldo + col);
      dst[0] = p[0]; dst[1] = p[1]; dst[2] = p[2]; dst[3] = p[3];
    }
  }
}

// Scatter epilogues: bring the destination rows of the warp's rows of a tile
// (pos[row * topk ..], topk ints per row) into L1 before the epilogue waits
// for the accumulator. The epilogue reads them for every 32-column chunk; with
// them in L1 the first chunk's stores do not wait on a global load either,
// which shows where a CTA's only tile ends the kernel (one wave of tiles).
template <int MODE>
__device__ __forceinline__ void prefetch_scatter_rows(const GemmArgs& a, long long warp_row0,
                                                      int rows_valid) {
  if constexpr (MODE == kEpiScatter || MODE == kEpiScatterF8) {
    const int lane = threadIdx.x & 31;
    if (lane < rows_valid) {
      const int* p = a.pos + (warp_row0 + lane) * a.topk;
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p + a.topk - 1));
    }
  }
}

// The epilogue of one tile for the calling warp: TMEM lanes [32 * quarter,
// +32) of the accumulator at tbase hold rows row0 + 32 * quarter + lane of
// the tile (rows valid rows from row0; fewer, or none, at the ragged end),
// columns n_tile * 256 (SwiGLU: gate in the first 128 columns, up in the
// last 128, output features n_tile * 128). The warp takes the 32-column
// chunks ch = half, half + 2, ... Shared by the one-SM and the SM-pair
// kernels, which differ only in how they hand TMEM back.
template <int MODE, bool F8>
__device__ __forceinline__ void dense_tile_epilogue(const GemmArgs& a, uint32_t tbase, int row0,
                                                    int rows, int n_tile, int quarter, int half,
                                                    uint8_t* stage_w, float acc_s, float acc_s2,
                                                    float out_inv, float& amax) {
  constexpr bool kSwiglu = MODE == kEpiSwiglu || MODE == kEpiSwigluF8;
  const int lane = threadIdx.x & 31;
  const int r = quarter * 32 + lane;
  const bool row_ok = r < rows;
  const long long row = static_cast<long long>(row0) + r;
  const long long warp_row0 = static_cast<long long>(row0) + quarter * 32;
  const int warp_rows = rows - quarter * 32;
  if constexpr (kSwiglu) {
#pragma unroll 1
    for (int ch = half; ch < kBN / 64; ch += 2) {
      uint32_t g[32], u[32];
      tmem_ld_32cols(tbase + ch * 32, g);
      tmem_ld_32cols(tbase + kBN / 2 + ch * 32, u);
      tmem_ld_wait();
      const int col = n_tile * (kBN / 2) + ch * 32;
      if (col < a.N) {
        const float gs_half = 0.5f * acc_s;  // SiLU's halving folded into the gate scale
#pragma unroll
        for (int i = 0; i < 32; ++i)
          g[i] = __float_as_uint(silu_from_half(__uint_as_float(g[i]) * gs_half) *
                                 (__uint_as_float(u[i]) * acc_s2));
        if constexpr (MODE == kEpiSwigluF8) {
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(g[i])));
          }
          store_chunk_f8_scatter(a, g, out_inv, stage_w, warp_row0, warp_rows, col);
        } else {
          store_chunk_bf16_staged<kEpiBf16>(a, g, stage_w, warp_row0, warp_rows, col);
        }
      }
    }
  } else {
#pragma unroll 1
    for (int ch = half; ch < kBN / 32; ch += 2) {
      uint32_t v[32];
      tmem_ld_32cols(tbase + ch * 32, v);
      tmem_ld_wait();
      const int col = n_tile * kBN + ch * 32;
      if constexpr (F8) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * acc_s);
      }
      if constexpr (MODE == kEpiBf16 || MODE == kEpiF32) {
        if (a.addend != nullptr && row_ok && col < a.N) {
          // the lane's own row: 32 consecutive fp32 of the partial sum
          const float4* src = reinterpret_cast<const float4*>(a.addend + row * a.ld_add + col);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 f = src[q];
            v[4 * q + 0] = __float_as_uint(__uint_as_float(v[4 * q + 0]) + f.x);
            v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) + f.y);
            v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) + f.z);
            v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) + f.w);
          }
        }
      }
      if constexpr (MODE == kEpiF32) {
        if (row_ok && col < a.N) store_chunk<MODE>(a, v, row, col);
      } else if constexpr (MODE == kEpiScatterF8) {
        if (col < a.N) {
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(v[i])));
          }
          store_chunk_f8_scatter(a, v, out_inv, stage_w, warp_row0, warp_rows, col);
        }
      } else {
        if (col < a.N) store_chunk_bf16_staged<MODE>(a, v, stage_w, warp_row0, warp_rows, col);
      }
    }
  }
}

template <int MODE, bool DUAL, bool F8>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBu,
                   const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB2, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* tfull_bar = empty_bar + kStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* done_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* seg_s = reinterpret_cast<int*>(tmem_slot + 4);
  int* mt_s = seg_s + kMaxGroups + 1;
  uint8_t* stage_smem = reinterpret_cast<uint8_t*>(mt_s + kMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr bool kSwiglu = MODE == kEpiSwiglu || MODE == kEpiSwigluF8;
  constexpr int kBRowsPerTile = kSwiglu ? kBN / 2 : kBN;
  constexpr int kKB = F8 ? kBK8 : kBK;  // elements per k-block

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 32 * kGemmEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (kSwiglu) tma_prefetch_desc(&tmBu);
    if (DUAL) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // nothing above reads global memory: the set-up overlaps the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  if (a.grouped) {
    for (int i = threadIdx.x; i <= a.num_groups; i += blockDim.x) seg_s[i] = a.seg_offsets[i];
  }
  __syncthreads();
  if (a.grouped && warp == 2) {
    // exclusive prefix of ceil(n_g / kBM) over the groups
    int carry = 0;
    if (lane == 0) mt_s[0] = 0;
    for (int base = 0; base < a.num_groups; base += 32) {
      const int g = base + lane;
      int v = 0;
      if (g < a.num_groups) {
        const int len = seg_s[g + 1] - seg_s[g];
        v = len > 0 ? (len + kBM - 1) / kBM : 0;
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (g < a.num_groups) mt_s[g + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles =
      a.grouped ? mt_s[a.num_groups] * a.n_tiles : ((a.M + kBM - 1) / kBM) * a.n_tiles;
  const int kb_total = a.kb1 + (DUAL ? a.kb2 : 0);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol = (a.hints & 1) ? policy_evict_last() : policy_evict_normal();
      const uint64_t pol_b = (a.hints & 2) ? policy_evict_first() : policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0;
      uint32_t issued_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const TileCoord c = decode_tile(t, a, seg_s, mt_s, kBRowsPerTile);
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = tiles + stage * kStageBytes;
          uint8_t* sb = sa + kATileBytes;
          mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
          if (!DUAL || kb < a.kb1) {
            const int kc = kb * kKB;
            tma_load_2d(&tmA, &full_bar[stage], sa, kc, c.row0, pol);
            // B in two 128-row boxes: gate and up rows of the same features
            // (SwiGLU), or rows brow and brow + 128
            tma_load_2d(&tmB, &full_bar[stage], sb, kc, c.brow, pol_b);
            if (kSwiglu)
              tma_load_2d(&tmBu, &full_bar[stage], sb + kBTileBytes / 2, kc, c.brow, pol_b);
            else
              tma_load_2d(&tmB, &full_bar[stage], sb + kBTileBytes / 2, kc, c.brow + kBN / 2,
                          pol_b);
          } else {
            const int kc = (kb - a.kb1) * kKB;
            tma_load_2d(&tmA2, &full_bar[stage], sa, kc, c.row0, pol);
            tma_load_2d(&tmB2, &full_bar[stage], sb, kc, c.brow, pol_b);
            tma_load_2d(&tmB2, &full_bar[stage], sb + kBTileBytes / 2, kc, c.brow + kBN / 2, pol_b);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy this thread started lands before the CTA may exit
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = F8 ? instr_desc_e4m3(kBM, kBN) : instr_desc_bf16(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, a.status)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!wait_bounded(&full_bar[stage], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint8_t* sa = tiles + stage * kStageBytes;
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + kATileBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // +32 bytes along K inside the 128-byte swizzled row = +2 in addr>>4
            if constexpr (F8)
              tc_mma_f8(d_tmem, da + 2ull * k, db + 2ull * k, idesc, (kb | k) != 0 ? 1u : 0u);
            else
              tc_mma(d_tmem, da + 2ull * k, db + 2ull * k, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull_bar[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs issued by this thread complete before TMEM is released
      tc_commit(done_bar);
      wait_drain(done_bar, 0);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stage_w = stage_smem + (warp - 2) * kStageWarpBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    const float out_inv =
        (MODE == kEpiScatterF8 || MODE == kEpiSwigluF8) ? inv_scale(*a.out_scale) : 1.0f;
    // E4M3 operands: accumulator scale (SwiGLU: gate columns; up columns below)
    const float acc_s = F8 ? (*a.a_scale) * (*a.b_scale) : 1.0f;
    const float acc_s2 = (F8 && kSwiglu) ? (*a.a_scale) * (*a.b_scale2) : 1.0f;
    float amax = 0.0f;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const TileCoord c = decode_tile(t, a, seg_s, mt_s, kBRowsPerTile);
      prefetch_scatter_rows<MODE>(a, static_cast<long long>(c.row0) + quarter * 32,
                                  c.rows - quarter * 32);
      if (!warp_wait_bounded(&tfull_bar[acc], acc_phase, abort_flag, a.status)) break;
      tc_fence_after_sync();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      dense_tile_epilogue<MODE, F8>(a, tbase, c.row0, c.rows, c.n, quarter, half, stage_w, acc_s,
                                    acc_s2, out_inv, amax);
      tc_fence_before_sync();
      mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (MODE == kEpiScatterF8 || MODE == kEpiSwigluF8) {
      amax = warp_max(amax);
      if (lane == 0) atomic_max_nonneg(a.out_amax, amax);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace lmoe
