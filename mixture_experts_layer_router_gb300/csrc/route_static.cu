// Allocation-free routing: the same softmax / stable top-k / counting sort as
// latentmoe_route_from_logits, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: an application whose memory pool owns
// the whole device (an out-of-band allocation would fail, or break the pool's
// accounting), or a latency-critical loop that cannot afford cudaFree's
// implicit device synchronisation. This entry needs no handle and no
// workspace. The sort's scratch (per-chunk expert counts and their prefix
// sums, plus a status word) lives in one file-scope device array of fixed
// size, which every GPU that loads this library keeps until the process exits.
//
// Host code may not pass the array's name to a kernel: on the host that name
// is a stand-in, not a device address. The device address is looked up once
// per device with cudaGetSymbolAddress, on the first call made while that
// device is current, and cached by device ordinal. The cache does not follow
// a cudaDeviceReset (the module, and so the array, is then loaded again at
// another address), which is why the header rules out calls after a reset.
#include <mutex>

#include "kernels.h"
#include "latentmoe.h"

namespace {

// Per table (chunk counts, chunk prefix sums): ceil(T*k / 1024) * E ints.
constexpr long long kStaticTableInts = 131072;  // 512 KiB per table
constexpr int kStatusInts = 64;                  // 256 bytes; word 0 is the status

// [status | chunk counts | chunk prefix sums], 1 MiB + 256 B in total.
static __device__ __align__(256) int g_route_scratch[kStatusInts + 2 * kStaticTableInts];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
int* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_route_scratch on the current device (looked up once).
int scratch_on_current_device(int** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return LATENTMOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return LATENTMOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int*>(p);
  }
  *out = g_scratch_addr[dev];
  return LATENTMOE_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" int latentmoe_route_from_logits_static(const float* logits, int64_t T, int64_t E,
                                                  int top_k, uint32_t flags, int32_t* idx,
                                                  float* gates, int32_t* counts,
                                                  int32_t* offsets, int32_t* perm, int32_t* pos,
                                                  latentmoe_stream_t stream) {
  if (!logits || !idx || !gates || !counts || !offsets || !perm || !pos)
    return LATENTMOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || top_k < 1 || top_k > 16 || top_k > E) return LATENTMOE_ERR_INVALID_ARG;
  if (flags & ~static_cast<uint32_t>(LATENTMOE_RENORM)) return LATENTMOE_ERR_INVALID_ARG;
  if (E > lmoe::kMaxGroups) return LATENTMOE_ERR_UNSUPPORTED;
  const void* ptrs[] = {logits, idx, gates, counts, offsets, perm, pos};
  for (const void* p : ptrs)
    if (!aligned4(p)) return LATENTMOE_ERR_UNSUPPORTED;
  const long long S = static_cast<long long>(T) * top_k;
  if (S > (1ll << 30)) return LATENTMOE_ERR_UNSUPPORTED;
  // the fixed scratch holds ceil(S / 1024) * E ints per table, no more
  if (lmoe::sort_scratch_ints(S, E) > kStaticTableInts) return LATENTMOE_ERR_UNSUPPORTED;

  int* scratch = nullptr;
  const int r = scratch_on_current_device(&scratch);
  if (r != LATENTMOE_OK) return r;
  unsigned* status = reinterpret_cast<unsigned*>(scratch);
  int* cnt = scratch + kStatusInts;
  int* cbase = cnt + kStaticTableInts;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the count tables are fully rewritten by every call; only the status word
  // has to start at zero
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return LATENTMOE_ERR_CUDA;
  if (lmoe::launch_route_topk(logits, static_cast<int>(T), static_cast<int>(E), top_k,
                              (flags & LATENTMOE_RENORM) ? 1 : 0, nullptr, idx, gates,
                              s) != cudaSuccess)
    return LATENTMOE_ERR_CUDA;
  if (lmoe::launch_sort(idx, static_cast<int>(S), top_k, static_cast<int>(E), cnt, cbase, counts,
                        offsets, perm, pos, status, s) != cudaSuccess)
    return LATENTMOE_ERR_CUDA;
  return LATENTMOE_OK;
}
