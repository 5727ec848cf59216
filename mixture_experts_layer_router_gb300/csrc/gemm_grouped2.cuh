// Grouped expert GEMM on SM pairs: the grouped kernel of gemm_grouped.cuh
// with tcgen05 MMAs of cta_group::2 (M = 256 over two SMs).
//
// A pair tile is 256 weight rows per accumulator x the expert's tokens of one
// chunk (N <= 256, a multiple of 16). Each CTA of the pair holds its 128
// weight rows of both accumulators and half of the token rows (N/2), and
// receives its 128 rows of both accumulators in its own TMEM. Per k-block a
// CTA therefore takes in 32 KB of weights + 16 KB of tokens (against 32 + 32
// on one SM) and its tensor core reads 64 KB of shared memory (against 96),
// for the same MACs per SM: the operand feed that bounds the one-SM kernel
// shrinks by about 1.4x.
//
//   SwiGLU: CTA r holds feature block 2p + r (gate rows in accumulator 0, up
//           rows in accumulator 1) of pair tile p; its epilogue is the one-SM
//           SwiGLU epilogue for those 128 features.
//   plain:  accumulator a covers rows 512p + 256a .. +256 of W_d; CTA r holds
//           rows 512p + 256a + 128r .. +128. An expert of more than 256 slots
//           runs "wide" tiles instead (one accumulator of rows 256p + 128r ..
//           +128 per CTA for up to 512 tokens; see wide_chunks below).
//
// Roles (both CTAs): warp 0 lane 0 loads its CTA's tiles (completing on the
// leader's full barrier), warp 1 allocates TMEM (the leader's lane 0 also
// issues the MMAs and commits to both CTAs), warps 2..9 drain this CTA's
// accumulators and arrive, one lane per warp, on the leader's TMEM-empty
// barrier. Pair rules are listed in ptx_pair.cuh.
//
// Tile order: without GroupedArgs::tile_counter, every role walks the tiles
// round robin itself (pair, pair + npairs, ...). With it, each pair's first
// tile is its own index and the leader's producer takes the later ones from
// that global counter (zero at launch; the last CTA to exit sets it back to
// zero, so no memset sits between two launches), so pairs whose tiles ran
// faster take more of them and the last wave ends together; the indices then
// reach the other roles of both CTAs through a ring in shared memory
// (tile_ring, tr_full, tr_empty). The down GEMM, with few long tiles per
// pair, uses the counter (the round robin left its slowest pair ~4 % behind
// the mean); the gate+up GEMM, with many short tiles, keeps the round robin,
// whose tiles need no hand-off (with the ring it measured ~1.5 % slower).
//
// Shapes: SwiGLU needs F % 256 == 0, plain needs l % 512 == 0 (otherwise the
// one-SM kernel runs).
#pragma once

#include "gemm_grouped.cuh"
#include "ptx_pair.cuh"

namespace lmoe {

constexpr int kPStages = 4;
constexpr int kPTokenTile = 128 * 128;  // up to 128 token rows of 128 bytes
constexpr int kPStageBytes = 2 * kGWeightTile + kPTokenTile;  // 48 KB
// The tile sequence ring: the leader's producer publishes each tile index to
// the consumers of both CTAs (peer producer, MMA issuer, 2 x 8 epilogue warps)
constexpr int kTileRing = 8;
constexpr int kTileConsumers = 2 + 2 * kGEpiWarps;
constexpr int kPBarrierBytes = 8 * (2 * kPStages + 3 + 2 * kTileRing) + 4 * kTileRing;
constexpr int kPSmemBytes = 1024 + kPStages * kPStageBytes + kPBarrierBytes + 16 + kGTableBytes +
                            16 /* staging alignment */ + kGEpiWarps * kGStageWarpBytes;
static_assert(kPSmemBytes <= 232448, "pair kernel shared memory");

struct PTile {
  int g;      // group
  int tok0;   // first token row of the chunk
  int out0;   // first output row of the chunk
  int len;    // valid tokens (<= 256; wide tiles <= 512)
  int n;      // MMA N of the first MMA: len (wide: its first 256 tokens) rounded up to 16
  int n2;     // wide tiles: MMA N of the second MMA (tokens 256.. of the chunk), else 0
  int p;      // pair feature block (wide tiles: of 256 rows)
  int wide;   // plain GEMM, expert of more than 256 slots: one accumulator, up to 512 tokens
};

// Plain (down) GEMM on SM pairs. An expert of n <= 256 slots takes fblocks
// tiles of two accumulators (512 rows of W_d over the pair x its n tokens).
// An expert of more slots takes ceil(n / 512) token chunks, split evenly, of
// 2 * fblocks "wide" tiles: one accumulator (256 rows of W_d over the pair,
// 128 per CTA) x all tokens of the chunk, in two MMAs whose results land at
// TMEM columns [0, 256) and [256, 512), so that a token's column is its
// index in the chunk. A wide tile moves one weight tile per k-block for up
// to 512 tokens, where two chunk tiles of two accumulators would move the
// weights twice for the same MACs.
__device__ __forceinline__ void wide_chunks(int n, int& nch, int& cs) {
  nch = (n + 2 * kGMaxTok - 1) / (2 * kGMaxTok);
  const int per = (n + nch - 1) / nch;
  cs = (per + 15) & ~15;
}

template <int MODE>
__device__ __forceinline__ int pair_group_tiles(int n, int fblocks) {
  if (n <= 0) return 0;
  int nch, cs;
  if (MODE == kGrpPlain && n > kGMaxTok) {
    wide_chunks(n, nch, cs);
    return nch * 2 * fblocks;
  }
  group_chunks(n, nch, cs);
  return nch * fblocks;
}

// Exclusive prefix over groups of pair_group_tiles, by one warp.
template <int MODE>
__device__ __forceinline__ void build_pair_tile_prefix(const GroupedArgs& a, const GroupTable& gt) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  if (lane == 0) gt.tp[0] = 0;
  for (int base = 0; base < a.num_groups; base += 32) {
    const int g = base + lane;
    int v = g < a.num_groups ? pair_group_tiles<MODE>(gt.len[g], a.fblocks) : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (g < a.num_groups) gt.tp[g + 1] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
}

// Tile `local` of a group of n rows starting at input row in0 and output row
// out0 (group index g), in the order of pair_group_tiles: feature block
// major, then token chunk.
template <int MODE>
__device__ __forceinline__ PTile ptile_of(int g, int local, int n, int in0, int out0) {
  const bool wide = MODE == kGrpPlain && n > kGMaxTok;
  int nch, cs;
  if (wide)
    wide_chunks(n, nch, cs);
  else
    group_chunks(n, nch, cs);
  const int p = local / nch;
  const int c = local - p * nch;
  PTile r;
  r.g = g;
  r.tok0 = in0 + c * cs;
  r.out0 = out0 + c * cs;
  r.len = min(cs, n - c * cs);
  r.wide = wide ? 1 : 0;
  if (wide) {
    r.n = r.len >= kGMaxTok ? kGMaxTok : (r.len + 15) & ~15;
    r.n2 = r.len > kGMaxTok ? (r.len - kGMaxTok + 15) & ~15 : 0;
  } else {
    r.n = (r.len + 15) & ~15;
    r.n2 = 0;
  }
  r.p = p;
  return r;
}

template <int MODE>
__device__ __forceinline__ PTile decode_ptile(int t, const GroupedArgs& a, const GroupTable& gt) {
  const int g = tile_group(t, a, gt);
  return ptile_of<MODE>(g, t - gt.tp[g], gt.len[g], gt.in[g], gt.out[g]);
}

// a.fblocks = pair feature blocks per group (SwiGLU F/256, plain l/512).
template <int MODE, bool F8>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_grouped_pair_kernel(const __grid_constant__ CUtensorMap tmTok,
                             const __grid_constant__ CUtensorMap tmW0,
                             const __grid_constant__ CUtensorMap tmW1, const GroupedArgs a) {
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
  const GroupTable gt = group_table_at(tmem_slot + 4);
  uint8_t* stage_smem = staging_after_table(tmem_slot + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
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
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmTok);
    tma_prefetch_desc(&tmW0);
    tma_prefetch_desc(&tmW1);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  // nothing above reads global memory: the set-up overlaps the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  load_group_table(a, gt);
  __syncthreads();
  if (warp == 2) build_pair_tile_prefix<MODE>(a, gt);
  tc_fence_before_sync();
  __syncthreads();
  // both CTAs' barriers are initialised before either touches the other's
  cluster_sync();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = gt.tp[a.num_groups];

  // Tile sequence. The leader's producer walks the tiles: the first is `pair`,
  // later ones come from a.tile_counter (so pairs that run ahead take more
  // tiles and the last wave ends together), or pair + i * npairs without a
  // counter; -1 ends the walk. Every other role reads the same sequence from
  // the ring: wait on tr_full[slot] of its own CTA, read tile_ring[slot],
  // arrive on the leader's tr_empty[slot]. Returns -2 if a wait gave up.
  // Without a counter no role touches the ring: each one walks
  // pair, pair + npairs, ... itself (next_static).
  const bool dynamic = a.tile_counter != nullptr;
  auto next_static = [&](int& cur) -> int {
    const int t = cur;
    cur += npairs;
    return t < total_tiles ? t : -1;
  };
  const uint32_t tr_empty_leader = mapa_shared(smem_addr(&tr_empty[0]), 0);
  auto read_tile = [&](int& slot, uint32_t& ph) -> int {
    if (!wait_bounded_pair(&tr_full[slot], ph, abort_flag, peer_abort, a.status)) return -2;
    const int t = *reinterpret_cast<volatile int*>(&tile_ring[slot]);
    mbar_arrive_cluster(tr_empty_leader + 8u * static_cast<uint32_t>(slot));
    if (++slot == kTileRing) {
      slot = 0;
      ph ^= 1u;
    }
    return t;
  };

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
      int t_next = pair;
      const uint32_t ring_peer = mapa_shared(smem_addr(&tile_ring[0]), 1);
      const uint32_t full_peer = mapa_shared(smem_addr(&tr_full[0]), 1);
      int t_static = pair;
      while (ok) {
        int t;
        if (!dynamic) {
          t = next_static(t_static);
        } else if (leader) {
          t = t_next < total_tiles ? t_next : -1;
          // publish t to both CTAs
          if (!wait_bounded_pair(&tr_empty[ring_slot], ring_ph ^ 1u, abort_flag, peer_abort,
                                 a.status)) {
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
          if (t >= 0) t_next = npairs + atomicAdd(a.tile_counter, 1);
        } else {
          t = read_tile(ring_slot, ring_ph);
        }
        if (t < 0) break;
        const PTile c = decode_ptile<MODE>(t, a, gt);
        // this CTA's token rows: half of the (first) MMA's N, and for a wide
        // tile half of the second MMA's, from token 256 of the chunk on
        const int half = c.n >> 1, half2 = c.n2 >> 1;
        const int nbox = (half + kGTokBox - 1) / kGTokBox;
        const int nbox2 = (half2 + kGTokBox - 1) / kGTokBox;
        const uint32_t bytes =
            c.wide ? 2u * (kGWeightTile + (nbox + nbox2) * kGTokBoxBytes)
                   : 2u * (2 * kGWeightTile + nbox * kGTokBoxBytes);
        int rt0, rt1;
        if (MODE == kGrpSwiglu) {
          rt0 = rt1 = (c.g * a.w_group_rows) / 128 + 2 * c.p + static_cast<int>(rank);
        } else if (c.wide) {
          rt0 = rt1 = (c.g * a.w_group_rows) / 128 + 2 * c.p + static_cast<int>(rank);
        } else {
          rt0 = (c.g * a.w_group_rows) / 128 + 4 * c.p + static_cast<int>(rank);
          rt1 = rt0 + 2;
        }
        const int tok_row = c.tok0 + static_cast<int>(rank) * half;
        const int tok_row2 = c.tok0 + kGMaxTok + static_cast<int>(rank) * half2;
        for (int kb = 0; kb < a.kb; ++kb) {
          if (!wait_bounded_pair(&empty_bar[stage], phase ^ 1u, abort_flag, peer_abort,
                                 a.status)) {
            ok = false;
            break;
          }
          // stage: [weights 0 | weights 1 | tokens], or for a wide tile
          // [weights | tokens of the first MMA | tokens of the second]
          uint8_t* sw0 = tiles + stage * kPStageBytes;
          uint8_t* sw1 = sw0 + kGWeightTile;
          uint8_t* stok = sw1 + kGWeightTile;
          const uint32_t fb = mapa_shared(smem_addr(&full_bar[stage]), 0);
          const int kc = kb * (F8 ? kGBK8 : kGBK);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], bytes);
          tma_load_3d_pair(&tmW0, fb, sw0, 0, 0, rt0 * a.kb + kb, pol_w);
          if (c.wide) {
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_pair(&tmTok, fb, sw1 + b * kGTokBoxBytes, kc, tok_row + b * kGTokBox,
                               pol_t);
            for (int b = 0; b < nbox2; ++b)
              tma_load_2d_pair(&tmTok, fb, stok + b * kGTokBoxBytes, kc, tok_row2 + b * kGTokBox,
                               pol_t);
          } else {
            tma_load_3d_pair(MODE == kGrpSwiglu ? &tmW1 : &tmW0, fb, sw1, 0, 0,
                             rt1 * a.kb + kb, pol_w);
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_pair(&tmTok, fb, stok + b * kGTokBoxBytes, kc, tok_row + b * kGTokBox,
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
      int t_static = pair;
      while (ok) {
        const int t = dynamic ? read_tile(ring_slot, ring_ph) : next_static(t_static);
        if (t < 0) break;
        const PTile c = decode_ptile<MODE>(t, a, gt);
        const uint32_t idesc = F8 ? instr_desc_e4m3(256, c.n) : instr_desc_bf16(256, c.n);
        const uint32_t idesc2 =
            F8 ? instr_desc_e4m3(256, c.n2 > 0 ? c.n2 : 16) : instr_desc_bf16(256, c.n2 > 0 ? c.n2 : 16);
        if (!wait_bounded_pair(tempty_bar, acc_phase ^ 1u, abort_flag, peer_abort, a.status))
          break;
        tc_fence_after_sync();
        for (int kb = 0; kb < a.kb; ++kb) {
          if (!wait_bounded_pair(&full_bar[stage], phase, abort_flag, peer_abort, a.status)) {
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
    const float in_s = F8 ? *a.in_scale : 1.0f;
    const float out_inv = (F8 && MODE == kGrpSwiglu) ? inv_scale(*a.out_scale) : 1.0f;
    float amax = 0.0f;
    int ring_slot = 0;
    uint32_t ring_ph = 0;
    int t_static = pair;
    while (true) {
      int t;
      if (dynamic) {
        t = 0;
        if (lane == 0) t = read_tile(ring_slot, ring_ph);
        t = __shfl_sync(0xffffffffu, t, 0);
      } else {
        t = next_static(t_static);
      }
      if (t < 0) break;
      const PTile c = decode_ptile<MODE>(t, a, gt);
      if (!warp_wait_bounded_pair(tfull_bar, acc_phase, abort_flag, peer_abort, a.status)) break;
      tc_fence_after_sync();
      const int r = static_cast<int>(rank);
      // a wide tile's one accumulator holds rows 256p + 128r .. of W_d for
      // all len (<= 512) tokens, token j at column j
      const int feat0 = MODE == kGrpSwiglu ? (2 * c.p + r) * 128 + quarter * 32
                        : c.wide           ? c.p * 256 + r * 128 + quarter * 32
                                           : c.p * 512 + r * 128 + quarter * 32;
      grouped_tile_epilogue<MODE, F8>(a, tmem_base + lane_off, half, c.g, c.len, c.out0, feat0,
                                      feat0 + 256, !c.wide, in_s, out_inv, amax, stage_w, [&] {
                                        // one arrival per warp on the leader's barrier
                                        tc_fence_before_sync();
                                        __syncwarp();
                                        if (lane == 0) mbar_arrive_cluster(tempty_leader);
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
  // every MMA of the pair has completed (the leader waited on its last
  // commit) and both epilogues are done with TMEM
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, 512);
  }
  // the last CTA out sets the tile counter and the exit count back to zero
  // (every producer has taken its last tile before its CTA gets here)
  if (dynamic && threadIdx.x == 0) {
    __threadfence();
    unsigned* exits = reinterpret_cast<unsigned*>(a.tile_counter) + 1;
    if (atomicAdd(exits, 1u) == gridDim.x - 1u) {
      a.tile_counter[0] = 0;
      *exits = 0u;
      __threadfence();
    }
  }
}

}  // namespace lmoe
