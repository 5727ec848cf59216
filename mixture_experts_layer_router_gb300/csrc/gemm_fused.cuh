// Both expert GEMMs in one persistent launch on SM pairs: the grouped
// gate+up GEMM with its SwiGLU epilogue (z -> h) and the grouped down GEMM
// (h -> o), as the tiles of one sequence taken from a global counter.
//
// The tiles are those of gemm_grouped_pair_kernel for the two GEMMs ("GU"
// tiles of the SwiGLU GEMM, "D" tiles of the down GEMM), and so are the
// stage ring, the TMEM use and the epilogues: every output element is formed
// by the same MMAs in the same order, so h and o are bitwise those of the
// two launches. What changes is the order and the hand-over of h:
//
// - Tile order. Blocks of tiles, one per (GEMM, expert): the GU blocks of
//   experts 0 .. lag-1, then GU(e) followed by D(e - lag) for e = lag ..
//   E-1, then the D blocks of the last lag experts. The down GEMM of an
//   expert thus comes about lag experts' worth of gate+up tiles after its
//   own gate+up tiles, and the SMs that finish the gate+up work early run
//   down tiles instead of idling in the first launch's tail.
// - Hand-over of h. Each GU tile, once its epilogue has stored its 256
//   features of h (128 per CTA) for its token chunk, adds one per epilogue
//   warp (16 per pair tile) to dep[e][pair feature block] after a GPU-scope
//   fence. Before a D tile's producers load h's k-blocks of a feature block,
//   they wait (acquire, bounded) until that count reaches 16 x the expert's
//   token chunks, then order the async-proxy loads after the acquire. h is
//   stored with an evict-last policy in the hope that the D tiles find it in
//   L2; measured, they mostly do not (the launch reads what the two launches
//   read from DRAM), so the gain is the second launch's tail, which matters
//   only for small layers.
//
// Progress: every tile, the first of each pair included, is taken from the
// global counter, so tiles are taken in sequence order and only by CTAs that
// are running. Every wait of a D tile is on tiles earlier in the sequence,
// which running CTAs took before it and whose loads their producers issued
// before moving on; so the earliest unfinished tile can always proceed, even
// if not every CTA of the grid is resident yet. Each wait is bounded anyway
// (kWaitLimitNs, then LATENTMOE_STATUS_TIMEOUT and the abort flags of both
// CTAs).
//
// The last CTA to exit sets the tile counter, the exit count and every dep
// count back to zero, so consecutive launches need no memset.
#pragma once

#include "gemm_grouped2.cuh"

namespace lmoe {

struct FusedExpertArgs {
  GroupedArgs gu;    // gate+up: seg_offsets, fblocks = F / 256, kb = l / BK, out = h
  GroupedArgs dn;    // down: the same seg_offsets, fblocks = l / 512, kb = F / BK, out = o
  int* dep;          // [E * gu.fblocks] completion counts, zero at launch and left zero
  int* tile_counter; // [2] {next tile, exit count}, zero at launch and left zero
  int lag;           // 1 <= lag <= E (see the tile order above)
};

// Block b of the tile order: GEMM (0: gate+up, 1: down) and expert.
__device__ __forceinline__ void fused_block(int b, int E, int lag, int& gemm, int& e) {
  if (b < lag) {
    gemm = 0;
    e = b;
  } else if (b < 2 * E - lag) {
    const int j = b - lag;
    gemm = j & 1;
    e = (j & 1) ? (j >> 1) : lag + (j >> 1);
  } else {
    gemm = 1;
    e = E - lag + (b - (2 * E - lag));
  }
}

// Group table of the fused kernel (kGTableBytes): first row and rows of each
// expert, then the exclusive prefix of tiles over the 2E blocks.
struct FusedTable {
  int* off;
  int* len;
  int* tp;  // [2E + 1]
};

__device__ __forceinline__ FusedTable fused_table_at(void* p) {
  int* b = static_cast<int*>(p);
  return FusedTable{b, b + kGMaxGroups, b + 2 * kGMaxGroups};
}

__device__ __forceinline__ int fused_block_tiles(const FusedExpertArgs& a, const FusedTable& ft,
                                                 int b) {
  int gemm, e;
  fused_block(b, a.gu.num_groups, a.lag, gemm, e);
  const int n = ft.len[e];
  return gemm == 0 ? pair_group_tiles<kGrpSwiglu>(n, a.gu.fblocks)
                   : pair_group_tiles<kGrpPlain>(n, a.dn.fblocks);
}

// Exclusive prefix of tiles over the blocks, by one warp.
__device__ __forceinline__ void build_fused_prefix(const FusedExpertArgs& a, const FusedTable& ft) {
  const int lane = threadIdx.x & 31;
  const int nb = 2 * a.gu.num_groups;
  int carry = 0;
  if (lane == 0) ft.tp[0] = 0;
  for (int base = 0; base < nb; base += 32) {
    const int b = base + lane;
    int v = b < nb ? fused_block_tiles(a, ft, b) : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (b < nb) ft.tp[b + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
}

struct FTile {
  int gemm;  // 0: gate+up, 1: down
  PTile c;
};

__device__ __forceinline__ FTile decode_ftile(int t, const FusedExpertArgs& a,
                                              const FusedTable& ft) {
  // the block of tile t: the largest b with tp[b] <= t (that block is non-empty)
  int lo = 0, hi = 2 * a.gu.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ft.tp[mid] <= t) lo = mid; else hi = mid - 1;
  }
  int gemm, e;
  fused_block(lo, a.gu.num_groups, a.lag, gemm, e);
  FTile r;
  r.gemm = gemm;
  const int local = t - ft.tp[lo];
  r.c = gemm == 0 ? ptile_of<kGrpSwiglu>(e, local, ft.len[e], ft.off[e], ft.off[e])
                  : ptile_of<kGrpPlain>(e, local, ft.len[e], ft.off[e], ft.off[e]);
  return r;
}

// Count of epilogue-warp arrivals that completes dep[e][p]: 16 per GU tile
// (8 warps in each CTA of the pair), one GU tile per token chunk.
__device__ __forceinline__ int dep_target(int n) {
  int nch, cs;
  group_chunks(n, nch, cs);
  return nch * 2 * kGEpiWarps;
}

// Bounded wait until *p >= target (acquire), then the proxy fence for the
// TMA loads that follow. On timeout: both CTAs' abort flags and the status.
__device__ __forceinline__ bool wait_count_pair(const int* p, int target, volatile int* abort_flag,
                                                uint32_t peer_abort, unsigned* status) {
  if (ld_acquire_gpu(p) >= target) {
    fence_proxy_async_global();
    return true;
  }
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    __nanosleep(200);
    if (ld_acquire_gpu(p) >= target) {
      fence_proxy_async_global();
      return true;
    }
    if ((++n & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1u) : "memory");
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

template <bool F8>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_expert_fused_kernel(const __grid_constant__ CUtensorMap tmZ,
                             const __grid_constant__ CUtensorMap tmWg,
                             const __grid_constant__ CUtensorMap tmWu,
                             const __grid_constant__ CUtensorMap tmH,
                             const __grid_constant__ CUtensorMap tmWd, const FusedExpertArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kPStages * kPStageBytes);
  uint64_t* empty_bar = full_bar + kPStages;
  uint64_t* tfull_bar = empty_bar + kPStages;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* done_bar = tempty_bar + 1;
  uint64_t* tr_full = done_bar + 1;             // [kTileRing], both CTAs
  uint64_t* tr_empty = tr_full + kTileRing;     // [kTileRing], the leader's is used
  int* tile_ring = reinterpret_cast<int*>(tr_empty + kTileRing);  // [kTileRing]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_ring + kTileRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* last_flag = const_cast<int*>(abort_flag) + 1;
  const FusedTable ft = fused_table_at(tmem_slot + 4);
  uint8_t* stage_smem = staging_after_table(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int E = a.gu.num_groups;
  const uint32_t peer_abort =
      mapa_shared(smem_addr(const_cast<int*>(abort_flag)), rank ^ 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * kGEpiWarps);
    mbar_init(done_bar, 1);
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(&tr_full[i], 1);
      mbar_init(&tr_empty[i], kTileConsumers);
    }
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmZ);
    tma_prefetch_desc(&tmWg);
    tma_prefetch_desc(&tmWu);
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmWd);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  // nothing above reads global memory: the set-up overlaps the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const int s0 = a.gu.seg_offsets[i];
    ft.off[i] = s0;
    ft.len[i] = a.gu.seg_offsets[i + 1] - s0;
  }
  __syncthreads();
  if (warp == 2) build_fused_prefix(a, ft);
  tc_fence_before_sync();
  __syncthreads();
  // both CTAs' barriers are initialised before either touches the other's
  cluster_sync();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = ft.tp[2 * E];

  // Tile sequence: the leader's producer takes every index from the counter
  // (the next one while the current tile's loads are issued) and publishes
  // each to the other roles of both CTAs through the ring (as the dynamic
  // order of gemm_grouped_pair_kernel).
  const uint32_t tr_empty_leader = mapa_shared(smem_addr(&tr_empty[0]), 0);
  auto read_tile = [&](int& slot, uint32_t& ph) -> int {
    if (!wait_bounded_pair(&tr_full[slot], ph, abort_flag, peer_abort, a.gu.status)) return -2;
    const int t = *reinterpret_cast<volatile int*>(&tile_ring[slot]);
    mbar_arrive_cluster(tr_empty_leader + 8u * static_cast<uint32_t>(slot));
    if (++slot == kTileRing) {
      slot = 0;
      ph ^= 1u;
    }
    return t;
  };

  // k-blocks of h per pair feature block of the gate+up GEMM (256 features)
  constexpr int kKbPerBlock = 256 / (F8 ? kGBK8 : kGBK);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      const uint64_t pol_w = policy_evict_normal();
      const uint64_t pol_t = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      int ring_slot = 0;
      uint32_t ring_ph = 0;
      int t_next = leader ? atomicAdd(a.tile_counter, 1) : 0;
      const uint32_t ring_peer = mapa_shared(smem_addr(&tile_ring[0]), 1);
      const uint32_t full_peer = mapa_shared(smem_addr(&tr_full[0]), 1);
      while (ok) {
        int t;
        if (leader) {
          t = t_next < total_tiles ? t_next : -1;
          if (!wait_bounded_pair(&tr_empty[ring_slot], ring_ph ^ 1u, abort_flag, peer_abort,
                                 a.gu.status)) {
            ok = false;
            break;
          }
          tile_ring[ring_slot] = t;
          st_cluster_s32(ring_peer + 4u * static_cast<uint32_t>(ring_slot), t);
          mbar_arrive(&tr_full[ring_slot]);
          mbar_arrive_cluster(full_peer + 8u * static_cast<uint32_t>(ring_slot));
          if (++ring_slot == kTileRing) {
            ring_slot = 0;
            ring_ph ^= 1u;
          }
          if (t >= 0) t_next = atomicAdd(a.tile_counter, 1);
        } else {
          t = read_tile(ring_slot, ring_ph);
        }
        if (t < 0) break;
        const FTile f = decode_ftile(t, a, ft);
        const PTile& c = f.c;
        const GroupedArgs& g = f.gemm == 0 ? a.gu : a.dn;
        const int half = c.n >> 1, half2 = c.n2 >> 1;
        const int nbox = (half + kGTokBox - 1) / kGTokBox;
        const int nbox2 = (half2 + kGTokBox - 1) / kGTokBox;
        const uint32_t bytes =
            c.wide ? 2u * (kGWeightTile + (nbox + nbox2) * kGTokBoxBytes)
                   : 2u * (2 * kGWeightTile + nbox * kGTokBoxBytes);
        int rt0, rt1;
        const CUtensorMap* m_w0;
        const CUtensorMap* m_w1;
        const CUtensorMap* m_tok;
        if (f.gemm == 0) {
          rt0 = rt1 = (c.g * g.w_group_rows) / 128 + 2 * c.p + static_cast<int>(rank);
          m_w0 = &tmWg;
          m_w1 = &tmWu;
          m_tok = &tmZ;
        } else {
          if (c.wide) {
            rt0 = rt1 = (c.g * g.w_group_rows) / 128 + 2 * c.p + static_cast<int>(rank);
          } else {
            rt0 = (c.g * g.w_group_rows) / 128 + 4 * c.p + static_cast<int>(rank);
            rt1 = rt0 + 2;
          }
          m_w0 = m_w1 = &tmWd;
          m_tok = &tmH;
        }
        const int tok_row = c.tok0 + static_cast<int>(rank) * half;
        const int tok_row2 = c.tok0 + kGMaxTok + static_cast<int>(rank) * half2;
        const int* dep_e = a.dep + c.g * a.gu.fblocks;
        const int dep_n = f.gemm == 1 ? dep_target(ft.len[c.g]) : 0;
        for (int kb = 0; kb < g.kb; ++kb) {
          // a down tile reads h's k-blocks of a feature block once every gate+up
          // tile of that feature block of the expert has stored them
          if (f.gemm == 1 && kb % kKbPerBlock == 0 &&
              !wait_count_pair(dep_e + kb / kKbPerBlock, dep_n, abort_flag, peer_abort,
                               a.gu.status)) {
            ok = false;
            break;
          }
          if (!wait_bounded_pair(&empty_bar[stage], phase ^ 1u, abort_flag, peer_abort,
                                 a.gu.status)) {
            ok = false;
            break;
          }
          uint8_t* sw0 = tiles + stage * kPStageBytes;
          uint8_t* sw1 = sw0 + kGWeightTile;
          uint8_t* stok = sw1 + kGWeightTile;
          const uint32_t fb = mapa_shared(smem_addr(&full_bar[stage]), 0);
          const int kc = kb * (F8 ? kGBK8 : kGBK);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], bytes);
          tma_load_3d_pair(m_w0, fb, sw0, 0, 0, rt0 * g.kb + kb, pol_w);
          if (c.wide) {
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_pair(m_tok, fb, sw1 + b * kGTokBoxBytes, kc, tok_row + b * kGTokBox,
                               pol_t);
            for (int b = 0; b < nbox2; ++b)
              tma_load_2d_pair(m_tok, fb, stok + b * kGTokBoxBytes, kc, tok_row2 + b * kGTokBox,
                               pol_t);
          } else {
            tma_load_3d_pair(m_w1, fb, sw1, 0, 0, rt1 * g.kb + kb, pol_w);
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_pair(m_tok, fb, stok + b * kGTokBoxBytes, kc, tok_row + b * kGTokBox,
                               pol_t);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the leader's full barriers count both CTAs' bytes: waiting on them
      // drains every copy of the pair still in flight
      if (leader)
        for (int s = 0; s < kPStages; ++s)
          if (issued_mask & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (leader)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int ring_slot = 0;
      uint32_t ring_ph = 0;
      while (ok) {
        const int t = read_tile(ring_slot, ring_ph);
        if (t < 0) break;
        const FTile f = decode_ftile(t, a, ft);
        const PTile& c = f.c;
        const int kbn = f.gemm == 0 ? a.gu.kb : a.dn.kb;
        const uint32_t idesc = F8 ? instr_desc_e4m3(256, c.n) : instr_desc_bf16(256, c.n);
        const uint32_t idesc2 = F8 ? instr_desc_e4m3(256, c.n2 > 0 ? c.n2 : 16)
                                   : instr_desc_bf16(256, c.n2 > 0 ? c.n2 : 16);
        if (!wait_bounded_pair(tempty_bar, acc_phase ^ 1u, abort_flag, peer_abort, a.gu.status))
          break;
        tc_fence_after_sync();
        for (int kb = 0; kb < kbn; ++kb) {
          if (!wait_bounded_pair(&full_bar[stage], phase, abort_flag, peer_abort, a.gu.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint8_t* sw0 = tiles + stage * kPStageBytes;
          const uint64_t d0 = smem_desc_sw128(sw0);
          const uint64_t d1 = smem_desc_sw128(sw0 + kGWeightTile);
          const uint64_t dt = smem_desc_sw128(sw0 + 2 * kGWeightTile);
          if (c.wide) {
            // one weight tile; tokens [0, 256) into columns [0, 256), the
            // rest of the chunk into columns [256, 512)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
              if constexpr (F8) {
                tc_mma_pair_f8(tmem_base, d0 + 2ull * k, d1 + 2ull * k, idesc, accum);
                if (c.n2 > 0)
                  tc_mma_pair_f8(tmem_base + 256, d0 + 2ull * k, dt + 2ull * k, idesc2, accum);
              } else {
                tc_mma_pair(tmem_base, d0 + 2ull * k, d1 + 2ull * k, idesc, accum);
                if (c.n2 > 0)
                  tc_mma_pair(tmem_base + 256, d0 + 2ull * k, dt + 2ull * k, idesc2, accum);
              }
            }
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
              if constexpr (F8) {
                tc_mma_pair_f8(tmem_base, d0 + 2ull * k, dt + 2ull * k, idesc, accum);
                tc_mma_pair_f8(tmem_base + 256, d1 + 2ull * k, dt + 2ull * k, idesc, accum);
              } else {
                tc_mma_pair(tmem_base, d0 + 2ull * k, dt + 2ull * k, idesc, accum);
                tc_mma_pair(tmem_base + 256, d1 + 2ull * k, dt + 2ull * k, idesc, accum);
              }
            }
          }
          tc_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(tfull_bar, 0x3);
        acc_phase ^= 1u;
      }
      tc_commit_pair(done_bar, 0x3);
      wait_drain(done_bar, 0);
    }
  } else {
    // ------------------------------------------------ epilogue warps (both CTAs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stage_w = stage_smem + (warp - 2) * kGStageWarpBytes;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tempty_leader = mapa_shared(smem_addr(tempty_bar), 0);
    uint32_t acc_phase = 0;
    const float in_gu = F8 ? *a.gu.in_scale : 1.0f;
    const float in_dn = F8 ? *a.dn.in_scale : 1.0f;
    const float out_inv = F8 ? inv_scale(*a.gu.out_scale) : 1.0f;
    float amax = 0.0f, amax_dn = 0.0f;
    // h stays in L2 until the down tiles read it
    const uint64_t pol_h = policy_evict_last();
    int ring_slot = 0;
    uint32_t ring_ph = 0;
    auto release = [&] {
      // one arrival per warp on the leader's barrier
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);
    };
    while (true) {
      int t = 0;
      if (lane == 0) t = read_tile(ring_slot, ring_ph);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0) break;
      const FTile f = decode_ftile(t, a, ft);
      const PTile& c = f.c;
      if (!warp_wait_bounded_pair(tfull_bar, acc_phase, abort_flag, peer_abort, a.gu.status))
        break;
      tc_fence_after_sync();
      const int r = static_cast<int>(rank);
      if (f.gemm == 0) {
        const int feat0 = (2 * c.p + r) * 128 + quarter * 32;
        grouped_tile_epilogue<kGrpSwiglu, F8, true>(a.gu, tmem_base + lane_off, half, c.g,
                                                    c.len, c.out0, feat0, feat0 + 256, true,
                                                    in_gu, out_inv, amax, stage_w, release,
                                                    pol_h);
        // this warp's part of h is stored: count it for the down tiles
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(a.dep + c.g * a.gu.fblocks + c.p, 1);
        }
      } else {
        const int feat0 = c.wide ? c.p * 256 + r * 128 + quarter * 32
                                 : c.p * 512 + r * 128 + quarter * 32;
        grouped_tile_epilogue<kGrpPlain, F8>(a.dn, tmem_base + lane_off, half, c.g, c.len,
                                             c.out0, feat0, feat0 + 256, !c.wide, in_dn, 1.0f,
                                             amax_dn, stage_w, release);
      }
      acc_phase ^= 1u;
    }
    if constexpr (F8) {
      amax = warp_max(amax);
      if (lane == 0) atomic_max_nonneg(a.gu.out_amax, amax);
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
    tmem_dealloc_pair(tmem_base, 512);
  }
  // the last CTA out sets the tile counter, the exit count and the dep counts
  // back to zero: every CTA has passed its last wait and its last arrival
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned* exits = reinterpret_cast<unsigned*>(a.tile_counter) + 1;
    *last_flag = atomicAdd(exits, 1u) == gridDim.x - 1u ? 1 : 0;
  }
  __syncthreads();
  if (*last_flag) {
    __threadfence();
    for (int i = threadIdx.x; i < E * a.gu.fblocks; i += blockDim.x) a.dep[i] = 0;
    if (threadIdx.x == 0) {
      a.tile_counter[0] = 0;
      a.tile_counter[1] = 0;
    }
    __threadfence();
  }
}

}  // namespace lmoe
