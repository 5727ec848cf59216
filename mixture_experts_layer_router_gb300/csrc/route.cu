// Routing: softmax gating with stable top-k, and the counting sort of the
// (token, choice) slots by expert.
//
// "The Training and RL Infrastructure Behind MAI-Thinking-1": the router
// reads the full hidden state and gates with a softmax (section "The model
// the systems run"); top-k uses a stable sort so equal logits always resolve
// to the lower expert index (section "Bitwise determinism"); dropless routing
// with token metadata kept on the device (sections "Sharding and
// parallelism" and, in "Frontier Pre-training at Microsoft AI", "Reducing
// per-expert overhead").
//
// Everything here is integer or fixed-order: no floating-point atomics, so
// the outputs are bitwise reproducible.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lmoe {

// One warp per token. Lane i holds logits of experts i, i+32, ... (VPL of
// them). Softmax: max and sum of exp by warp butterflies (fixed order).
// Selection: k rounds of a warp arg-max under the order (value desc, index
// asc); the winner is marked taken. NaN logits are treated as -inf.
template <int VPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int renorm,
                                                         const float* __restrict__ sel_bias,
                                                         int* __restrict__ idx,
                                                         float* __restrict__ gates) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + static_cast<long long>(t) * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? row[e] : -INFINITY;
    v[i] = (x != x) ? -INFINITY : x;
  }
  float m = v[0];
#pragma unroll
  for (int i = 1; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);

  // ranking keys: the logits, or logits + bias for a selection-only bias
  float key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = (sel_bias != nullptr && e < E) ? v[i] + sel_bias[e] : v[i];
  }
  uint32_t taken = 0;
  float gsel[16];
  int isel[16];
  float gsum = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      float bl = -INFINITY;  // the logit of the best key
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (key[i] > bv || (key[i] == bv && e < bi))) {
          bv = key[i];
          bi = e;
          bl = v[i];
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        const float ol = __shfl_xor_sync(0xffffffffu, bl, off);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
          bl = ol;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      const float g = expf(bl - m) / s;
      gsel[j] = g;
      isel[j] = bi;
      gsum += g;
    }
  }
  if (lane == 0) {
    const float scale = renorm ? 1.0f / gsum : 1.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < k) {
        idx[static_cast<long long>(t) * k + j] = isel[j];
        gates[static_cast<long long>(t) * k + j] = renorm ? gsel[j] * scale : gsel[j];
      }
    }
  }
}

// Router replay without gates: the softmax probabilities (over all E, same
// reductions as route_topk_kernel) of given expert choices. Ids outside
// [0, E) get gate 0 (the counting sort drops them and flags the status).
template <int VPL>
__global__ void __launch_bounds__(256) replay_gates_kernel(const float* __restrict__ logits, int T,
                                                           int E, const int* __restrict__ idx,
                                                           int k, int renorm,
                                                           float* __restrict__ gates) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + static_cast<long long>(t) * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? row[e] : -INFINITY;
    v[i] = (x != x) ? -INFINITY : x;
  }
  float m = v[0];
#pragma unroll
  for (int i = 1; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    float g[16];
    float gsum = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      g[j] = 0.0f;
      if (j < k) {
        const int e = idx[static_cast<long long>(t) * k + j];
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
          float x = row[e];
          x = (x != x) ? -INFINITY : x;
          g[j] = expf(x - m) / s;
        }
        gsum += g[j];
      }
    }
    const float scale = (renorm && gsum > 0.0f) ? 1.0f / gsum : 1.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < k) gates[static_cast<long long>(t) * k + j] = renorm ? g[j] * scale : g[j];
  }
}

cudaError_t launch_replay_gates(const float* logits, int T, int E, const int* idx, int k,
                                int renorm, float* gates, cudaStream_t s) {
  const int blocks = (T + 7) / 8;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    replay_gates_kernel<1><<<blocks, 256, 0, s>>>(logits, T, E, idx, k, renorm, gates);
  else if (vpl <= 2)
    replay_gates_kernel<2><<<blocks, 256, 0, s>>>(logits, T, E, idx, k, renorm, gates);
  else if (vpl <= 4)
    replay_gates_kernel<4><<<blocks, 256, 0, s>>>(logits, T, E, idx, k, renorm, gates);
  else if (vpl <= 8)
    replay_gates_kernel<8><<<blocks, 256, 0, s>>>(logits, T, E, idx, k, renorm, gates);
  else
    replay_gates_kernel<16><<<blocks, 256, 0, s>>>(logits, T, E, idx, k, renorm, gates);
  return cudaGetLastError();
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renorm,
                              const float* sel_bias, int* idx, float* gates, cudaStream_t s) {
  const int blocks = (T + 7) / 8;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    route_topk_kernel<1><<<blocks, 256, 0, s>>>(logits, T, E, k, renorm, sel_bias, idx, gates);
  else if (vpl <= 2)
    route_topk_kernel<2><<<blocks, 256, 0, s>>>(logits, T, E, k, renorm, sel_bias, idx, gates);
  else if (vpl <= 4)
    route_topk_kernel<4><<<blocks, 256, 0, s>>>(logits, T, E, k, renorm, sel_bias, idx, gates);
  else if (vpl <= 8)
    route_topk_kernel<8><<<blocks, 256, 0, s>>>(logits, T, E, k, renorm, sel_bias, idx, gates);
  else
    route_topk_kernel<16><<<blocks, 256, 0, s>>>(logits, T, E, k, renorm, sel_bias, idx, gates);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Load-balancing statistics: prob_sum[e] = sum over tokens of softmax(L_t)_e,
// with the softmax of route_topk_kernel (same max and sum reductions). Block b
// takes kLblTokens tokens, 32 per warp in token order; each lane accumulates
// its experts over its warp's tokens, the warps' partials are added in warp
// order, and a second kernel adds the blocks' partials in block order, so the
// result does not depend on scheduling.
template <int VPL>
__global__ void __launch_bounds__(256) lbl_partial_kernel(const float* __restrict__ logits, int T,
                                                          int E, float* __restrict__ partial) {
  __shared__ float wsum[8][512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.0f;
  const int t0 = blockIdx.x * kLblTokens + warp * (kLblTokens / 8);
  for (int tt = 0; tt < kLblTokens / 8; ++tt) {
    const int t = t0 + tt;
    if (t >= T) break;
    const float* row = logits + static_cast<long long>(t) * E;
    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      float x = (e < E) ? row[e] : -INFINITY;
      v[i] = (x != x) ? -INFINITY : x;
    }
    float m = v[0];
#pragma unroll
    for (int i = 1; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E) acc[i] += expf(v[i] - m) / s;
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) wsum[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float tot = 0.0f;
    for (int w = 0; w < 8; ++w) tot += wsum[w][e];
    partial[static_cast<long long>(blockIdx.x) * E + e] = tot;
  }
}

__global__ void lbl_reduce_kernel(const float* __restrict__ partial, int nb, int E,
                                  float* __restrict__ out) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  float tot = 0.0f;
  for (int b = 0; b < nb; ++b) tot += partial[static_cast<long long>(b) * E + e];
  out[e] = tot;
}

cudaError_t launch_lbl_prob_sum(const float* logits, int T, int E, float* partial, float* out,
                                cudaStream_t s) {
  const int nb = (T + kLblTokens - 1) / kLblTokens;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    lbl_partial_kernel<1><<<nb, 256, 0, s>>>(logits, T, E, partial);
  else if (vpl <= 2)
    lbl_partial_kernel<2><<<nb, 256, 0, s>>>(logits, T, E, partial);
  else if (vpl <= 4)
    lbl_partial_kernel<4><<<nb, 256, 0, s>>>(logits, T, E, partial);
  else if (vpl <= 8)
    lbl_partial_kernel<8><<<nb, 256, 0, s>>>(logits, T, E, partial);
  else
    lbl_partial_kernel<16><<<nb, 256, 0, s>>>(logits, T, E, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  lbl_reduce_kernel<<<(E + 127) / 128, 128, 0, s>>>(partial, nb, E, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Counting sort. The S = T*k slots s (flattened [T, k], token t = s / k) are
// cut into chunks of kSortChunk. (1) Each chunk counts its experts into row
// b of cnt [chunks, E]. (2) For each expert, an exclusive scan over chunks
// gives cbase[b, e]; counts[e] is the total, offsets the exclusive scan over
// experts. (3) Each chunk walks its slots in order, 32 at a time; lanes with
// the same expert get consecutive ranks in lane order, so slot order inside
// an expert follows s, i.e. token order (a token never picks an expert
// twice). Expert ids outside [0, E) set kStatusBadExpert and get pos = -1.

__global__ void __launch_bounds__(256) sort_hist_kernel(const int* __restrict__ idx, int S, int E,
                                                        int* __restrict__ cnt, unsigned* status) {
  extern __shared__ int hist[];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * kSortChunk;
  bool bad = false;
  for (int i = threadIdx.x; i < kSortChunk; i += blockDim.x) {
    const int s = base + i;
    if (s < S) {
      const int e = idx[s];
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
        atomicAdd(&hist[e], 1);
      else
        bad = true;
    }
  }
  if (bad) atomicOr(status, kStatusBadExpert);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    cnt[static_cast<long long>(blockIdx.x) * E + i] = hist[i];
}

// One block of 512 threads; thread e owns expert e (E <= 512).
__global__ void __launch_bounds__(512) sort_scan_kernel(const int* __restrict__ cnt, int nb, int E,
                                                        int* __restrict__ cbase,
                                                        int* __restrict__ counts,
                                                        int* __restrict__ offsets) {
  __shared__ int warp_tot[16];
  const int e = threadIdx.x;
  const int lane = e & 31, w = e >> 5;
  int run = 0;
  if (e < E) {
    int b = 0;
    for (; b + 8 <= nb; b += 8) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = cnt[static_cast<long long>(b + i) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cbase[static_cast<long long>(b + i) * E + e] = run;
        run += v[i];
      }
    }
    for (; b < nb; ++b) {
      const int v = cnt[static_cast<long long>(b) * E + e];
      cbase[static_cast<long long>(b) * E + e] = run;
      run += v;
    }
  }
  // exclusive scan of run over e
  int incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int wbase = 0;
  for (int i = 0; i < w; ++i) wbase += warp_tot[i];
  if (e < E) {
    counts[e] = run;
    offsets[e] = wbase + incl - run;
    if (e == E - 1) offsets[E] = wbase + incl;
  }
}

// One warp per chunk.
__global__ void __launch_bounds__(32) sort_scatter_kernel(const int* __restrict__ idx, int S, int k,
                                                          int E, const int* __restrict__ cbase,
                                                          const int* __restrict__ offsets,
                                                          int* __restrict__ perm,
                                                          int* __restrict__ pos,
                                                          unsigned* status) {
  extern __shared__ int run[];
  const int lane = threadIdx.x;
  for (int i = lane; i < E; i += 32)
    run[i] = offsets[i] + cbase[static_cast<long long>(blockIdx.x) * E + i];
  const int base = blockIdx.x * kSortChunk;
  int ev[kSortChunk / 32];
#pragma unroll
  for (int st = 0; st < kSortChunk / 32; ++st) {
    const int s = base + st * 32 + lane;
    ev[st] = (s < S) ? idx[s] : -1;
  }
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int st = 0; st < kSortChunk / 32; ++st) {
    const int s = base + st * 32 + lane;
    const int e = ev[st];
    const bool valid = s < S && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const int key = valid ? e : (0x40000000 | lane);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & lt);
    if (valid) {
      const int slot = run[e] + rank;
      if (in_bounds(slot, S, status)) {
        perm[slot] = s / k;
        pos[s] = slot;
      }
    } else if (s < S) {
      pos[s] = -1;
    }
    __syncwarp();
    if (valid && rank == 0) run[e] += __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// The same counting sort in one cooperative launch (every CTA resident at
// once). CTA b owns chunk b (kSortChunk slots); warp w of it owns the 128
// slots [b * kSortChunk + 128 w, +128). Three phases, two grid barriers:
//   1. per-warp expert histograms in shared memory; the CTA's sum is row b
//      of cnt [chunks, E];
//   2. expert e is scanned over the chunks by one warp of the grid (warp
//      b * 8 + w takes experts e = b * 8 + w, + 8 * chunks, ...): cbase[b, e]
//      is the exclusive prefix over chunks and counts[e] the total;
//   3. every CTA forms offsets from counts (exclusive scan over experts; CTA 0
//      writes them), turns its warp histograms into starting slots
//      offsets[e] + cbase[b, e] + (slots of e in earlier warps of the chunk),
//      and each warp ranks its slots in order, 32 at a time, exactly as
//      sort_scatter_kernel does, so perm and pos are the three-kernel sort's.
// The barrier counters (sync[0]: arrivals, sync[1]: exits) start at zero and
// the last CTA to leave sets them back to zero for the next launch. A barrier
// wait gives up after kWaitLimitNs and sets kStatusTimeout.
constexpr int kFSortWarps = kSortChunk / 128;  // 8

__device__ __forceinline__ bool grid_barrier(unsigned* arrivals, unsigned target,
                                             unsigned* status, int* ok_smem) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(arrivals, 1u);
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    while (*reinterpret_cast<volatile unsigned*>(arrivals) < target) {
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(status, kStatusTimeout);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *ok_smem = ok;
  }
  __syncthreads();
  return *ok_smem != 0;
}

__global__ void __launch_bounds__(256) sort_fused_kernel(
    const int* __restrict__ idx, int S, int k, int E, int* __restrict__ cnt,
    int* __restrict__ cbase, int* __restrict__ counts, int* __restrict__ offsets,
    int* __restrict__ perm, int* __restrict__ pos, unsigned* status, unsigned* sync) {
  extern __shared__ int whist[];  // [kFSortWarps][E], later the warps' starting slots
  __shared__ int ok_smem;
  __shared__ int wtot[kFSortWarps];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  for (int i = threadIdx.x; i < kFSortWarps * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();

  // 1. histograms: each distinct expert of a 32-slot step is added by its
  // lowest lane (match_any), so a warp's row needs no atomics
  const unsigned lt = (1u << lane) - 1u;
  const int base = b * kSortChunk + warp * 128;
  int ev[4];
  bool bad = false;
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int sl = base + st * 32 + lane;
    const int e = sl < S ? idx[sl] : -1;
    ev[st] = e;
    const bool valid = sl < S && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    if (sl < S && !valid) bad = true;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : (0x40000000 | lane));
    if (valid && (peers & lt) == 0) whist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (bad) atomicOr(status, kStatusBadExpert);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kFSortWarps; ++w) c += whist[w * E + e];
    cnt[static_cast<long long>(b) * E + e] = c;
  }
  if (!grid_barrier(&sync[0], static_cast<unsigned>(nb), status, &ok_smem)) return;

  // 2. per-expert exclusive scan over the chunks, one warp per expert
  for (int e = b * kFSortWarps + warp; e < E; e += nb * kFSortWarps) {
    int carry = 0;
    for (int c0 = 0; c0 < nb; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nb ? cnt[static_cast<long long>(c) * E + e] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < nb) cbase[static_cast<long long>(c) * E + e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[e] = carry;
  }
  if (!grid_barrier(&sync[0], 2u * static_cast<unsigned>(nb), status, &ok_smem)) return;

  // 3a. offsets: exclusive scan of counts over the experts (every CTA)
  __shared__ int off_s[kMaxGroups + 1];
  {
    // thread i holds experts 2i, 2i + 1 (E <= 512)
    const int e0 = 2 * threadIdx.x;
    const int c0 = e0 < E ? counts[e0] : 0, c1 = e0 + 1 < E ? counts[e0 + 1] : 0;
    int incl = c0 + c1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    int wb = 0;
    for (int w = 0; w < warp; ++w) wb += wtot[w];
    const int ex = wb + incl - c0 - c1;
    if (e0 < E) off_s[e0] = ex;
    if (e0 + 1 < E) off_s[e0 + 1] = ex + c0;
    if (e0 + 1 == E) off_s[E] = ex + c0;
    if (e0 + 2 == E) off_s[E] = ex + c0 + c1;
    __syncthreads();
    if (b == 0)
      for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off_s[e];
  }
  // 3b. starting slot of each expert for each warp of this chunk
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = off_s[e] + cbase[static_cast<long long>(b) * E + e];
#pragma unroll
    for (int w = 0; w < kFSortWarps; ++w) {
      const int c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // 3c. stable scatter of this warp's slots
  int* run = whist + warp * E;
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int sl = base + st * 32 + lane;
    const int e = ev[st];
    const bool valid = sl < S && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : (0x40000000 | lane));
    const int rank = __popc(peers & lt);
    if (valid) {
      const int slot = run[e] + rank;
      if (in_bounds(slot, S, status)) {
        perm[slot] = sl / k;
        pos[sl] = slot;
      }
    } else if (sl < S) {
      pos[sl] = -1;
    }
    __syncwarp();
    if (valid && rank == 0) run[e] += __popc(peers);
    __syncwarp();
  }

  // the last CTA out resets the barrier counters for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sync[1], 1u) == static_cast<unsigned>(nb) - 1u) {
      sync[0] = 0u;
      sync[1] = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// The same counting sort in one CTA of 1024 threads, for up to
// kBlockSortMaxSlots slots: the grid barriers of sort_fused_kernel become
// block barriers. At T = 128, k = 2 it takes 8 us against 12 us for the
// cooperative launch; at 16384 slots it took 37 against 14 us (each warp then
// ranks 16 steps of 32 slots, where the 16 CTAs of the cooperative sort give
// each warp 4), hence the small limit. Warp w owns the slots [w L, (w + 1) L), L = ceil(S / 32)
// rounded up to 32, so the warps' ranges follow slot order:
//   1. per-warp expert histograms in shared memory (lowest lane of each
//      match_any group adds its size);
//   2. thread e (< E) sums expert e over the warps (counts), the block scans
//      the counts over the experts (offsets), and thread e turns the warps'
//      counts into their starting slots offsets[e] + (slots of e in earlier
//      warps);
//   3. each warp ranks its slots in order, 32 at a time, as
//      sort_scatter_kernel does.
// perm and pos are those of the other two sorts (a stable counting sort has
// one result).
__global__ void __launch_bounds__(1024) sort_block_kernel(const int* __restrict__ idx, int S, int k,
                                                          int E, int* __restrict__ counts,
                                                          int* __restrict__ offsets,
                                                          int* __restrict__ perm,
                                                          int* __restrict__ pos,
                                                          unsigned* status) {
  extern __shared__ int whist[];  // [32][E]: counts, then starting slots
  __shared__ int wtot[32];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  const int L = ((S + 31) / 32 + 31) & ~31;  // slots per warp, a multiple of 32
  const int base = warp * L;
  const unsigned lt = (1u << lane) - 1u;
  // the warp's expert ids, read once (all loads in flight together)
  constexpr int kSteps = kBlockSortMaxSlots / 1024;
  int ev[kSteps];
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int sl = base + i * 32 + lane;
    ev[i] = (i * 32 < L && sl < S) ? idx[sl] : -1;
  }

  // 1. histograms
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    if (i * 32 >= L) break;
    const int sl = base + i * 32 + lane;
    const int e = ev[i];
    const bool valid = sl < S && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    if (sl < S && !valid) bad = true;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : (0x40000000 | lane));
    if (valid && (peers & lt) == 0) whist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (bad) atomicOr(status, kStatusBadExpert);
  __syncthreads();

  // 2. counts, offsets (exclusive scan over the experts, E <= 1024), starting slots
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int w = 0; w < 32; ++w) c += whist[w * E + e];
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  int wb = 0;
  for (int w = 0; w < warp; ++w) wb += wtot[w];
  const int ex = wb + incl - c;
  if (e < E) {
    counts[e] = c;
    offsets[e] = ex;
    if (e == E - 1) offsets[E] = ex + c;
    int run = ex;
    for (int w = 0; w < 32; ++w) {
      const int cw = whist[w * E + e];
      whist[w * E + e] = run;
      run += cw;
    }
  }
  __syncthreads();

  // 3. stable scatter of this warp's slots
  int* run = whist + warp * E;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    if (i * 32 >= L) break;
    const int sl = base + i * 32 + lane;
    const int e = ev[i];
    const bool valid = sl < S && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : (0x40000000 | lane));
    const int rank = __popc(peers & lt);
    if (valid) {
      const int slot = run[e] + rank;
      if (in_bounds(slot, S, status)) {
        perm[slot] = sl / k;
        pos[sl] = slot;
      }
    } else if (sl < S) {
      pos[sl] = -1;
    }
    __syncwarp();
    if (valid && rank == 0) run[e] += __popc(peers);
    __syncwarp();
  }
}

cudaError_t launch_sort_block(const int* idx, int S, int k, int E, int* counts, int* offsets,
                              int* perm, int* pos, unsigned* status, cudaStream_t s) {
  if (S > kBlockSortMaxSlots || E > kMaxGroups) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(32) * E * sizeof(int);
  static bool attr_set[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        sort_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(static_cast<size_t>(32) * kMaxGroups * sizeof(int)));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  return launch_kernel(sort_block_kernel, dim3(1), dim3(1024), smem, s, 1, false, idx, S, k, E,
                       counts, offsets, perm, pos, status);
}

bool sort_fused_fits(int S, int E) {
  static int max_blocks_of[kMaxDevices] = {};
  const int dev = current_device_index();
  if (dev < 0 || E > kMaxGroups) return false;
  int& mb = max_blocks_of[dev];
  if (mb == 0) {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, sort_fused_kernel, 256, static_cast<size_t>(kFSortWarps) * kMaxGroups * 4) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    mb = per_sm * sms;
  }
  const int nb = (S + kSortChunk - 1) / kSortChunk;
  return nb <= mb;
}

cudaError_t launch_sort_fused(const int* idx, int S, int k, int E, int* cnt, int* cbase,
                              int* counts, int* offsets, int* perm, int* pos, unsigned* status,
                              unsigned* sync, cudaStream_t s) {
  const int nb = (S + kSortChunk - 1) / kSortChunk;
  const size_t smem = static_cast<size_t>(kFSortWarps) * E * sizeof(int);
  return launch_kernel(sort_fused_kernel, dim3(nb), dim3(256), smem, s, 1, true, idx, S, k, E,
                       cnt, cbase, counts, offsets, perm, pos, status, sync);
}

cudaError_t launch_sort(const int* idx, int S, int k, int E, int* cnt, int* cbase, int* counts,
                        int* offsets, int* perm, int* pos, unsigned* status, cudaStream_t s) {
  const int nb = (S + kSortChunk - 1) / kSortChunk;
  const size_t smem = static_cast<size_t>(E) * sizeof(int);
  sort_hist_kernel<<<nb, 256, smem, s>>>(idx, S, E, cnt, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sort_scan_kernel<<<1, 512, 0, s>>>(cnt, nb, E, cbase, counts, offsets);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sort_scatter_kernel<<<nb, 32, smem, s>>>(idx, S, k, E, cbase, offsets, perm, pos, status);
  return cudaGetLastError();
}

}  // namespace lmoe
