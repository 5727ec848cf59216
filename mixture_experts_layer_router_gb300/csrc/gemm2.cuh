// Dense GEMM on SM pairs: gemm_tc_kernel's product D = A B^T with tcgen05
// MMAs of cta_group::2 (M = 256 over two SMs, N = 256).
//
// A pair tile is 256 rows of A x 256 columns. CTA r of the pair holds A rows
// row0 + 128 r .. +128 and half of the B tile: B rows brow + 128 r .. +128
// (SwiGLU: the gate rows in CTA 0, the up rows of the same features in
// CTA 1). Each CTA receives its 128 rows x all 256 columns in its own TMEM,
// so its epilogue is the one-SM epilogue for those rows (gate columns first,
// then up). Per k-block a CTA takes in 16 KB of A and 16 KB of B (32 KB)
// for 128 x 256 x 64 MACs, against 48 KB for the same MACs on one SM: the
// operand feed per SM shrinks by a third. With 32 KB stages, six stages fit.
//
// Roles (both CTAs): warp 0 lane 0 loads its CTA's A and B halves
// (completing on the leader's full barrier, whose expected bytes the leader
// sets for both CTAs); warp 1 allocates TMEM (the leader's lane 0 issues the
// MMAs and commits to both CTAs); warps 2..9 drain this CTA's accumulator
// (two warps per TMEM lane quarter, alternate 32-column chunks) and arrive,
// one lane per warp, on the leader's TMEM-empty barrier.
// Accumulators are double-buffered (2 x 256 columns).
//
// Dense tiles only (GemmArgs::grouped == 0); the pair rules are those of
// ptx_pair.cuh.
#pragma once

#include "gemm.cuh"
#include "ptx_pair.cuh"

namespace lmoe {

constexpr int kPairBM = 2 * kBM;            // rows of A per pair tile
constexpr int kPairStages = 6;
constexpr int kPairBHalf = kBTileBytes / 2;  // 16 KB: this CTA's 128 rows of B
constexpr int kPairStageBytes = kATileBytes + kPairBHalf;
constexpr int kPairBarrierBytes = 8 * (2 * kPairStages + 2 + 2 + 1);
// layout: stage ring (1 KB aligned), epilogue staging (16-byte aligned for
// the 16-byte staging accesses), barriers, TMEM slot and abort flag
constexpr int kPairGemmSmemBytes =
    1024 + kPairStages * kPairStageBytes + kGemmEpiWarps * kStageWarpBytes + kPairBarrierBytes +
    16;
static_assert(kPairGemmSmemBytes <= 232448, "pair GEMM shared memory");

// Pair tile t of a dense GEMM: the raster of decode_tile with 256-row m-tiles
// (bands of max(1, group_m / 2) m-tiles).
__device__ __forceinline__ void decode_pair_tile(int t, const GemmArgs& a, int b_rows_per_tile,
                                                 int& row0, int& n, int& brow) {
  const int mt = (a.M + kPairBM - 1) / kPairBM;
  const int band_m = a.group_m > 1 ? a.group_m / 2 : 1;
  const int per = band_m * a.n_tiles;
  const int band = t / per;
  const int first = band * band_m;
  const int gm = min(band_m, mt - first);
  const int local = t - band * per;
  const int m = first + local % gm;
  n = local / gm;
  row0 = m * kPairBM;
  brow = n * b_rows_per_tile;
}

template <int MODE, bool DUAL, bool F8>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmBu,
                        const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB2, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint8_t* stage_smem = smem + kPairStages * kPairStageBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(stage_smem + kGemmEpiWarps * kStageWarpBytes);
  uint64_t* empty_bar = full_bar + kPairStages;
  uint64_t* tfull_bar = empty_bar + kPairStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* done_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const uint32_t peer_abort =
      mapa_shared(smem_addr(const_cast<int*>(abort_flag)), rank ^ 1u);
  constexpr bool kSwiglu = MODE == kEpiSwiglu || MODE == kEpiSwigluF8;
  constexpr int kBRowsPerTile = kSwiglu ? kBN / 2 : kBN;
  constexpr int kKB = F8 ? kBK8 : kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 2 * kGemmEpiWarps);  // one arrival per epilogue warp, both CTAs
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
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  // nothing above reads global memory: the set-up overlaps the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  // both CTAs' barriers are initialised before either touches the other's
  cluster_sync();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = ((a.M + kPairBM - 1) / kPairBM) * a.n_tiles;
  const int kb_total = a.kb1 + (DUAL ? a.kb2 : 0);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      const uint64_t pol = (a.hints & 1) ? policy_evict_last() : policy_evict_normal();
      const uint64_t pol_b = (a.hints & 2) ? policy_evict_first() : policy_evict_normal();
      const CUtensorMap* mapB = (kSwiglu && rank == 1) ? &tmBu : &tmB;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int t = pair; t < total_tiles && ok; t += npairs) {
        int row0, n, brow;
        decode_pair_tile(t, a, kBRowsPerTile, row0, n, brow);
        const int arow = row0 + static_cast<int>(rank) * kBM;
        // SwiGLU: both CTAs read rows brow (gate map in CTA 0, up map in CTA 1)
        const int brow_r = kSwiglu ? brow : brow + static_cast<int>(rank) * (kBN / 2);
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!wait_bounded_pair(&empty_bar[stage], phase ^ 1u, abort_flag, peer_abort,
                                 a.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = tiles + stage * kPairStageBytes;
          uint8_t* sb = sa + kATileBytes;
          const uint32_t fb = mapa_shared(smem_addr(&full_bar[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2u * kPairStageBytes);
          if (!DUAL || kb < a.kb1) {
            const int kc = kb * kKB;
            tma_load_2d_pair(&tmA, fb, sa, kc, arow, pol);
            tma_load_2d_pair(mapB, fb, sb, kc, brow_r, pol_b);
          } else {
            const int kc = (kb - a.kb1) * kKB;
            tma_load_2d_pair(&tmA2, fb, sa, kc, arow, pol);
            tma_load_2d_pair(&tmB2, fb, sb, kc, brow + static_cast<int>(rank) * (kBN / 2), pol_b);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the leader's full barriers count both CTAs' bytes: waiting on them
      // drains every copy of the pair still in flight
      if (leader)
        for (int s = 0; s < kPairStages; ++s)
          if (issued_mask & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (leader)
      constexpr uint32_t idesc =
          F8 ? instr_desc_e4m3(kPairBM, kBN) : instr_desc_bf16(kPairBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = pair; t < total_tiles && ok; t += npairs) {
        if (!wait_bounded_pair(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, peer_abort,
                               a.status))
          break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!wait_bounded_pair(&full_bar[stage], phase, abort_flag, peer_abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint8_t* sa = tiles + stage * kPairStageBytes;
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + kATileBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
            if constexpr (F8)
              tc_mma_pair_f8(d_tmem, da + 2ull * k, db + 2ull * k, idesc, accum);
            else
              tc_mma_pair(d_tmem, da + 2ull * k, db + 2ull * k, idesc, accum);
          }
          tc_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(&tfull_bar[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit_pair(done_bar, 0x3);
      wait_drain(done_bar, 0);
    }
  } else {
    // ------------------------------------------------ epilogue warps (both CTAs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stage_w = stage_smem + (warp - 2) * kStageWarpBytes;
    const uint32_t tempty0 = mapa_shared(smem_addr(&tempty_bar[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    const float out_inv =
        (MODE == kEpiScatterF8 || MODE == kEpiSwigluF8) ? inv_scale(*a.out_scale) : 1.0f;
    const float acc_s = F8 ? (*a.a_scale) * (*a.b_scale) : 1.0f;
    const float acc_s2 = (F8 && kSwiglu) ? (*a.a_scale) * (*a.b_scale2) : 1.0f;
    float amax = 0.0f;
    for (int t = pair; t < total_tiles; t += npairs) {
      int row0, n, brow;
      decode_pair_tile(t, a, kBRowsPerTile, row0, n, brow);
      const int crow0 = row0 + static_cast<int>(rank) * kBM;
      prefetch_scatter_rows<MODE>(a, static_cast<long long>(crow0) + quarter * 32,
                                  min(kBM, a.M - crow0) - quarter * 32);
      if (!warp_wait_bounded_pair(&tfull_bar[acc], acc_phase, abort_flag, peer_abort, a.status))
        break;
      tc_fence_after_sync();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      dense_tile_epilogue<MODE, F8>(a, tbase, crow0, min(kBM, a.M - crow0), n, quarter, half,
                                    stage_w, acc_s, acc_s2, out_inv, amax);
      // one arrival per warp on the leader's barrier
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * static_cast<uint32_t>(acc));
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
  // every MMA of the pair has completed (the leader waited on its last
  // commit) and both epilogues are done with TMEM
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace lmoe
