// Multi-round fixed-capacity schedule of the expert GEMMs.
//
// "Frontier Pre-training at Microsoft AI", section "Dropless MoE with
// tunable, fixed-size memory usage": experts are put into groups; each group
// runs rounds with a fixed per-expert token capacity; an overloaded expert
// first uses capacity its group leaves unused in the round, and only its
// remaining slots wait for another round; the round count is global. No slot
// is dropped.
//
// Round r, group of experts [e0, e1): every expert first takes
// min(remaining, C) of its slots; the group's unused capacity is then lent to
// experts with slots left, lowest index first. Expert e's slots keep their
// order: round r runs slots [start, start + take) of e's segment. The round's
// slots are packed expert after expert into a buffer of E * C rows.
//
// One block of up to 512 threads (E <= 512): thread g < groups decides the
// takes of its group, then the block writes, per round r,
//   len[r][e]  = take,   in[r][e] = offsets[e] + start (row of the expert-sorted slots),
//   out[r][e]  = exclusive prefix of take over e (row in the round buffer), out[r][E] = total,
// and info = {rounds used, slots left after max_rounds}.
#include "kernels.h"

namespace lmoe {

namespace {

// Exclusive prefix sum over the block (blockDim.x <= 1024, multiple of 32);
// returns this thread's prefix and writes the total to *total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += o;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    if (lane < nwarps) warp_sums[lane] = w;  // inclusive prefix of warp totals
    if (lane == nwarps - 1) *total = w;
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  const int r = before + x - v;
  __syncthreads();
  return r;
}

}  // namespace

__global__ void __launch_bounds__(512) round_schedule_kernel(const int* __restrict__ counts,
                                                             const int* __restrict__ offsets, int E,
                                                             int C, int G, int max_rounds,
                                                             int* __restrict__ rin,
                                                             int* __restrict__ rout,
                                                             int* __restrict__ rlen,
                                                             int* __restrict__ info,
                                                             unsigned* __restrict__ status) {
  __shared__ int rem[kGMaxGroups];
  __shared__ int used[kGMaxGroups];
  __shared__ int take[kGMaxGroups];
  __shared__ int warp_sums[32];
  __shared__ int total;
  __shared__ int rounds;
  const int tid = threadIdx.x;
  if (tid < E) {
    rem[tid] = counts[tid];
    used[tid] = 0;
  }
  if (tid == 0) rounds = 0;
  __syncthreads();
  const int ngroups = (E + G - 1) / G;
  for (int r = 0; r < max_rounds; ++r) {
    if (tid < ngroups) {
      const int e0 = tid * G, e1 = min(e0 + G, E);
      int pool = C * (e1 - e0);
      bool any = false;
      for (int e = e0; e < e1; ++e) {
        const int own = min(rem[e], C);
        take[e] = own;
        pool -= own;
      }
      for (int e = e0; e < e1; ++e) {
        const int extra = min(rem[e] - take[e], pool);
        take[e] += extra;
        pool -= extra;
        any |= take[e] > 0;
      }
      if (any) atomicMax(&rounds, r + 1);
    }
    __syncthreads();
    const int t = tid < E ? take[tid] : 0;
    const int pre = block_exclusive_scan(t, warp_sums, &total);
    if (tid < E) {
      rlen[r * E + tid] = t;
      rin[r * E + tid] = offsets[tid] + used[tid];
      rout[r * (E + 1) + tid] = pre;
      used[tid] += t;
      rem[tid] -= t;
    }
    if (tid == 0) rout[r * (E + 1) + E] = total;
    __syncthreads();
  }
  // slots that did not fit in max_rounds rounds
  const int left = tid < E ? rem[tid] : 0;
  const int pre = block_exclusive_scan(left, warp_sums, &total);
  (void)pre;
  if (tid == 0) {
    info[0] = rounds;
    info[1] = total;
    if (total > 0) atomicOr(status, kStatusRounds);
  }
}

cudaError_t launch_round_schedule(const int* counts, const int* offsets, int E, int C, int G,
                                  int max_rounds, int* rin, int* rout, int* rlen, int* info,
                                  unsigned* status, cudaStream_t s) {
  if (E < 1 || E > kGMaxGroups || C < 1 || G < 1 || max_rounds < 1) return cudaErrorInvalidValue;
  const int threads = ((E + 31) / 32) * 32;
  round_schedule_kernel<<<1, threads, 0, s>>>(counts, offsets, E, C, G, max_rounds, rin, rout, rlen,
                                              info, status);
  return cudaGetLastError();
}

}  // namespace lmoe
