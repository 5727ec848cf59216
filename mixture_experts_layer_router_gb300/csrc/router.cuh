// Router GEMM fused with softmax gating and stable top-k.
//
// "The Training and RL Infrastructure Behind MAI-Thinking-1": the router reads
// the full hidden state and gates with a softmax over all experts (section
// "The model the systems run"); router logits stay in FP32 (section
// "2. Numerics"); top-k uses a stable sort, so equal logits resolve to the
// lower expert index (section "Bitwise determinism").
//
// One CTA owns 128 token rows and all E <= 512 experts: L = x W_r^T (+ b)
// accumulates in TMEM (128 lanes x E columns, fp32) from TMA-fed tcgen05 MMAs
// (M = 128 tokens, N = up to 256 experts per instruction). The x map reads
// 128 rows x router_box_cols(E) columns per box, the W_r map
// router_w_box_rows(E) rows x router_box_cols(E) columns.
//
// Epilogue: 16 warps, four per TMEM lane quarter (32 rows); the four warps
// of a quarter split each row's experts.
//   phase A: warp s of the quarter takes the 32-expert chunks c = s, s+4, ...:
//            logits (+ bias) are stored for export, and each thread keeps its
//            row's maximum and a ranked list of its largest logits (larger
//            value first, lower expert id on equal values): each group of 8
//            logits is sorted by a fixed compare-and-swap network and merged
//            into the list by a bitonic merge (short dependency chains; the
//            same list as inserting the logits one by one). The four partial
//            maxima and lists meet in shared memory.
//   phase B: with the row maximum m, warp s forms partial sums
//            p[i] = sum over c of exp(L[32c + i] - m) for i in [8s, 8s + 8),
//            c ascending. The first warp of the quarter folds p[0..31] in the
//            order of a 32-lane butterfly, merges the four sets, and writes
//            idx and gates = exp(L - m) / sum (divided by their sum with
//            renorm). The sum and the gates are therefore bitwise identical
//            to the warp-per-token kernels of route.cu on the same logits.
#pragma once

#include "ptx.cuh"

namespace lmoe {

// k-blocks: 32 columns (64-byte swizzle) for E > 256, where a stage holds
// 512 rows of W_r (40 KB; four stages fit); 64 columns (128-byte swizzle) for
// E <= 256: the TMA then reads 128-byte row pieces of x and W_r instead of
// 64-byte ones, half the requests for the same bytes; and for E <= 128, 128
// columns as two 128-byte-swizzled atoms side by side, loaded by two TMA
// copies issued back to back, so that each x row is read as 256 contiguous
// bytes at a time (at E = 64, four 48 KB stages). The ring takes all the
// shared memory the exchange leaves.
__host__ __device__ constexpr int router_bk(int E) { return E <= 128 ? 128 : E <= 256 ? 64 : 32; }
// Columns of one TMA box of x and W_r (one swizzle atom wide).
__host__ __device__ constexpr int router_box_cols(int E) {
  return router_bk(E) < 64 ? router_bk(E) : 64;
}
constexpr int kRMaxStages = 16;
constexpr int kREpiWarps = 16;
constexpr int kRThreads = 64 + 32 * kREpiWarps;  // producer, MMA, 16 epilogue warps
constexpr int kRMaxSmem = 232448;                 // the most a CTA may have (227 KB)

// Shared-memory exchange between the four warps of a lane quarter.
template <int KMAX>
struct RouterExchange {
  float v[4][4][KMAX][32];  // [quarter][warp][slot][row]: partial top-k values
  int i[4][4][KMAX][32];    // and their expert ids
  float m[4][4][32];        // partial maxima
  float p[4][32][32];       // [quarter][partial i][row]
};

struct RouterArgs {
  int T, E, k, renorm;
  int kb;                  // d / router_bk(E)
  int stages;              // shared-memory stages (set by the launcher)
  const float* bias;       // [E] or null
  int bias_select;         // 0: bias is part of the logits; 1: it only moves the top-k choice
  float* logits;           // [T, E] fp32 out
  int* idx;                // [T, k]
  float* gates;            // [T, k]
  unsigned* status;
};

// Rows of the W_r box: the experts rounded up to 16 up to 256 experts (so a
// small router moves no zero rows), else two boxes of 256 rows.
__host__ __device__ constexpr int router_w_box_rows(int E) {
  return E <= 256 ? ((E + 15) & ~15) : 256;
}

// x tile (128 rows) plus the W_r boxes, for k-blocks of router_bk(E) columns
__host__ __device__ constexpr int router_stage_bytes(int E) {
  return 128 * router_bk(E) * 2 +
         (E <= 256 ? router_w_box_rows(E) * router_bk(E) * 2 : 2 * 256 * router_bk(E) * 2);
}

template <int KMAX>
__host__ __device__ constexpr int router_fixed_smem() {
  return 1024 + static_cast<int>(sizeof(RouterExchange<KMAX>)) + 8 * (2 * kRMaxStages + 3) + 16;
}

// (x, e) ranks before (v, i): larger value first, lower expert id on equal values.
__device__ __forceinline__ bool ranks_before(float x, int e, float v, int i) {
  return x > v || (x == v && e < i);
}

// Insert (x, e) into the list sv/si kept in ranking order (slot 0 first);
// the last slot drops out. A fixed, branch-free compare-and-shift network:
// the list stays in registers and the 32 rows of a warp never diverge.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&sv)[KMAX], int (&si)[KMAX], float x, int e) {
#pragma unroll
  for (int j = KMAX - 1; j > 0; --j) {
    const bool up = ranks_before(x, e, sv[j - 1], si[j - 1]);
    const bool here = ranks_before(x, e, sv[j], si[j]);
    const float nv = up ? sv[j - 1] : (here ? x : sv[j]);
    const int ni = up ? si[j - 1] : (here ? e : si[j]);
    sv[j] = nv;
    si[j] = ni;
  }
  if (ranks_before(x, e, sv[0], si[0])) {
    sv[0] = x;
    si[0] = e;
  }
}

// Compare-and-swap in ranking order: afterwards (va, ia) ranks before (vb, ib).
__device__ __forceinline__ void rank_cswap(float& va, int& ia, float& vb, int& ib) {
  const bool sw = ranks_before(vb, ib, va, ia);
  const float tv = sw ? vb : va;
  const int ti = sw ? ib : ia;
  vb = sw ? va : vb;
  ib = sw ? ia : ib;
  va = tv;
  ia = ti;
}

// Sorts 8 (value, expert) pairs into ranking order with a fixed network of 19
// compare-and-swaps in 6 layers (it sorts every 0-1 input, hence every input).
__device__ __forceinline__ void rank_sort8(float (&v)[8], int (&i)[8]) {
  constexpr int kNet[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6},
                               {3, 7}, {0, 1}, {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5},
                               {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) rank_cswap(v[kNet[c][0]], i[kNet[c][0]], v[kNet[c][1]], i[kNet[c][1]]);
}

// The first K of two lists in ranking order (sv/si of K, gv/gi of at least
// K), into sv/si, in ranking order: element j of the list against element
// K-1-j of the other keeps the better, which leaves a bitonic sequence
// holding the best K; log2(K) half-cleaning layers sort it. Equal to
// inserting the other list's elements one by one, for any K in {2, 4, 8}.
template <int K, int N>
__device__ __forceinline__ void rank_merge(float (&sv)[K], int (&si)[K], const float (&gv)[N],
                                           const int (&gi)[N]) {
  static_assert(K <= N && (K & (K - 1)) == 0, "merge of a power-of-two list");
#pragma unroll
  for (int j = 0; j < K; ++j) {
    if (ranks_before(gv[K - 1 - j], gi[K - 1 - j], sv[j], si[j])) {
      sv[j] = gv[K - 1 - j];
      si[j] = gi[K - 1 - j];
    }
  }
#pragma unroll
  for (int st = K / 2; st >= 1; st >>= 1)
#pragma unroll
    for (int j = 0; j < K; ++j)
      if ((j & st) == 0) rank_cswap(sv[j], si[j], sv[j + st], si[j + st]);
}

// BK = router_bk(E): the k-block width; the tensor maps' boxes are
// router_box_cols(E) columns wide (BK / 64 atoms per k-block for BK = 128).
template <int KMAX, int BK>
__global__ void __launch_bounds__(kRThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kATile = 128 * BK * 2;  // x
  constexpr int kAtoms = BK > 64 ? BK / 64 : 1;
  constexpr int kAtomCols = BK / kAtoms;
  constexpr int kXAtom = 128 * kAtomCols * 2;
  constexpr int kKPerAtom = kAtomCols / 16;
  const int stage_bytes = router_stage_bytes(a.E);
  // W_r atom (box b, atom j at sb + (b * kAtoms + j) * w_atom)
  const int w_atom = (a.E <= 256 ? router_w_box_rows(a.E) : 256) * kAtomCols * 2;
  RouterExchange<KMAX>* xch = reinterpret_cast<RouterExchange<KMAX>*>(smem);
  uint8_t* tiles = smem + ((sizeof(RouterExchange<KMAX>) + 1023) & ~static_cast<size_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(tiles + a.stages * stage_bytes);
  uint64_t* empty_bar = full_bar + a.stages;
  uint64_t* tfull_bar = empty_bar + a.stages;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* done_bar = tempty_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e_pad = (a.E + 15) & ~15;
  const int nbox = (a.E + 255) / 256;
  const uint32_t tmem_cols = e_pad <= 32 ? 32 : e_pad <= 64 ? 64 : e_pad <= 128 ? 128
                           : e_pad <= 256 ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 32 * kREpiWarps);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  // nothing above reads global memory: the set-up overlaps the previous kernel
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int m_tiles = (a.T + 127) / 128;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_x = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      // CTAs start their k walk at different k-blocks so that they do not all
      // read the same W_r slice at the same moment; the order is fixed per
      // CTA, so results stay deterministic
      const int kb0 = static_cast<int>((static_cast<unsigned>(blockIdx.x) * 37u) % a.kb);
      for (int t = blockIdx.x; t < m_tiles && ok; t += gridDim.x) {
        for (int i = 0; i < a.kb; ++i) {
          const int kb = (kb0 + i) % a.kb;
          if (!wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = tiles + stage * stage_bytes;
          uint8_t* sb = sa + kATile;
          mbar_arrive_expect_tx(&full_bar[stage], stage_bytes);
#pragma unroll
          for (int j = 0; j < kAtoms; ++j)
            tma_load_2d(&tmX, &full_bar[stage], sa + j * kXAtom, kb * BK + j * kAtomCols, t * 128,
                        pol_x);
          for (int b = 0; b < nbox; ++b)
#pragma unroll
            for (int j = 0; j < kAtoms; ++j)
              tma_load_2d(&tmW, &full_bar[stage], sb + (b * kAtoms + j) * w_atom,
                          kb * BK + j * kAtomCols, b * 256, pol_w);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < a.stages; ++s)
        if (issued_mask & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const int n0 = e_pad < 256 ? e_pad : 256;
      const int n1 = e_pad - n0;
      const uint32_t id0 = instr_desc_bf16(128, n0);
      const uint32_t id1 = instr_desc_bf16(128, n1 > 0 ? n1 : 16);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < m_tiles && ok; t += gridDim.x) {
        if (!wait_bounded(tempty_bar, acc_phase ^ 1u, abort_flag, a.status)) break;
        tc_fence_after_sync();
        for (int kb = 0; kb < a.kb; ++kb) {
          if (!wait_bounded(&full_bar[stage], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint8_t* sa = tiles + stage * stage_bytes;
          const uint8_t* sb = sa + kATile;
#pragma unroll
          for (int j = 0; j < kAtoms; ++j) {
            const uint8_t* xa = sa + j * kXAtom;
            const uint8_t* w0 = sb + j * w_atom;
            const uint8_t* w1 = sb + (kAtoms + j) * w_atom;  // second 256 experts (E > 256)
            const uint64_t da = kAtomCols == 64 ? smem_desc_sw128(xa) : smem_desc_sw64(xa);
            const uint64_t db0 = kAtomCols == 64 ? smem_desc_sw128(w0) : smem_desc_sw64(w0);
            const uint64_t db1 = kAtomCols == 64 ? smem_desc_sw128(w1) : smem_desc_sw64(w1);
#pragma unroll
            for (int k = 0; k < kKPerAtom; ++k) {
              const uint32_t accum = (kb | j | k) != 0 ? 1u : 0u;
              tc_mma(tmem_base, da + 2ull * k, db0 + 2ull * k, id0, accum);
              if (n1 > 0) tc_mma(tmem_base + 256, da + 2ull * k, db1 + 2ull * k, id1, accum);
            }
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == a.stages) {
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
    // ------------------------------------------------ epilogue: 4 warps per lane quarter
    const int quarter = warp & 3;
    const int sub = (warp - 2) >> 2;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const int nchunks = (a.E + 31) / 32;
    const int ngroups = (a.E + 7) / 8;
    const int k = a.k;
    const int bar_id = 1 + quarter;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < m_tiles; t += gridDim.x) {
      const int row = t * 128 + quarter * 32 + lane;
      const bool row_ok = row < a.T;
      if (!warp_wait_bounded(tfull_bar, acc_phase, abort_flag, a.status)) break;
      tc_fence_after_sync();

      // phase A: this warp's chunks: export, max, local top-k set
      float m = -INFINITY;
      float sv[KMAX];
      int si[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        sv[j] = -INFINITY;
        si[j] = 0x7fffffff;
      }
      float* lrow = a.logits + static_cast<long long>(row) * a.E;
      {
#pragma unroll 1
        for (int g8 = sub; g8 < ngroups; g8 += 4) {
          const int e0 = g8 * 8;
          uint32_t v[8];
          tmem_ld_8cols(lane_base + e0, v);
          tmem_ld_wait();
          float xv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x = __uint_as_float(v[i]);
            if (e0 + i < a.E && a.bias != nullptr && !a.bias_select) x += a.bias[e0 + i];
            xv[i] = x;
          }
          if (row_ok) {
            if (e0 + 8 <= a.E && (a.E & 3) == 0) {
              *reinterpret_cast<float4*>(lrow + e0) = make_float4(xv[0], xv[1], xv[2], xv[3]);
              *reinterpret_cast<float4*>(lrow + e0 + 4) = make_float4(xv[4], xv[5], xv[6], xv[7]);
            } else {
              for (int i = 0; i < 8; ++i)
                if (e0 + i < a.E) lrow[e0 + i] = xv[i];
            }
          }
          // ranking keys (the logit, or logit + bias for a selection-only
          // bias); columns past E get a key that never ranks
          float gv[8];
          int gi[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = e0 + i;
            const bool in = e < a.E;
            float x = xv[i];
            x = (x != x || !in) ? -INFINITY : x;
            m = fmaxf(m, x);
            gv[i] = (in && a.bias_select) ? x + a.bias[e] : x;
            gi[i] = in ? e : 0x7fffffff;
          }
          if constexpr (KMAX <= 8) {
            // sort the 8 and merge them into the running list
            rank_sort8(gv, gi);
            rank_merge<KMAX, 8>(sv, si, gv, gi);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) topk_insert<KMAX>(sv, si, gv[i], gi[i]);
          }
        }
      }
      xch->m[quarter][sub][lane] = m;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        xch->v[quarter][sub][j][lane] = sv[j];
        xch->i[quarter][sub][j][lane] = si[j];
      }
      named_barrier(bar_id, 128);

      // phase B: row maximum, then this warp's 8 of the 32 exp partials
      m = fmaxf(fmaxf(xch->m[quarter][0][lane], xch->m[quarter][1][lane]),
                fmaxf(xch->m[quarter][2][lane], xch->m[quarter][3][lane]));
      float p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) p[j] = 0.0f;
      for (int c0 = 0; c0 < nchunks; c0 += 2) {
        // two chunks' 8 columns per TMEM wait; the sums still run over the
        // chunks in ascending order
        uint32_t v[2][8];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (c0 + q < nchunks) tmem_ld_8cols(lane_base + (c0 + q) * 32 + sub * 8, v[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int c = c0 + q;
          if (c >= nchunks) break;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int e = c * 32 + sub * 8 + j;
            if (e < a.E) {
              float x = __uint_as_float(v[q][j]);
              if (a.bias != nullptr && !a.bias_select) x += a.bias[e];
              x = (x != x) ? -INFINITY : x;
              p[j] += expf(x - m);
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(tempty_bar);  // this warp is done with the tile's TMEM
#pragma unroll
      for (int j = 0; j < 8; ++j) xch->p[quarter][sub * 8 + j][lane] = p[j];
      named_barrier(bar_id, 128);

      if (sub == 0 && row_ok) {
        // fold the 32 partials as a butterfly would (lane 0's result)
        float q[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) q[i] = xch->p[quarter][i][lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int i = 0; i < off; ++i) q[i] = q[i] + q[i + off];
        const float ssum = q[0];
        // merge the other warps' lists into this one; the result is in
        // ranking order already
#pragma unroll 1
        for (int s2 = 1; s2 < 4; ++s2) {
          if constexpr (KMAX <= 8) {
            float ov[KMAX];
            int oi[KMAX];
#pragma unroll
            for (int j2 = 0; j2 < KMAX; ++j2) {
              ov[j2] = xch->v[quarter][s2][j2][lane];
              oi[j2] = xch->i[quarter][s2][j2][lane];
            }
            rank_merge<KMAX, KMAX>(sv, si, ov, oi);
          } else {
#pragma unroll
            for (int j2 = 0; j2 < KMAX; ++j2) {
              if (j2 >= k) break;
              topk_insert<KMAX>(sv, si, xch->v[quarter][s2][j2][lane],
                                xch->i[quarter][s2][j2][lane]);
            }
          }
        }
        float g[KMAX];
        float gsum = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          g[j] = 0.0f;
          if (j < k) {
            // with a selection-only bias the list holds biased keys: take the
            // logit itself from the row this CTA exported
            float lx = sv[j];
            if (a.bias_select) {
              lx = lrow[si[j]];
              lx = (lx != lx) ? -INFINITY : lx;
            }
            g[j] = expf(lx - m) / ssum;
            gsum += g[j];
          }
        }
        const float scale = a.renorm ? 1.0f / gsum : 1.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) {
            a.idx[static_cast<long long>(row) * k + j] = si[j];
            a.gates[static_cast<long long>(row) * k + j] = a.renorm ? g[j] * scale : g[j];
          }
      }
      // the exchange buffers are reused by the next tile
      named_barrier(bar_id, 128);
      acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace lmoe
