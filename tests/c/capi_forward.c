/* The whole forward from C through the C ABI: device memory from the CUDA
 * runtime, seeded bf16 weights and tokens made on the host, two forwards on
 * the default stream. Checks: every call returns LATENTMOE_OK, the device
 * status word stays 0, the output is finite and not all zero, and the two
 * forwards are bitwise equal. Prints "ok" and exits 0, or names the failed
 * check and exits 1. Needs a GPU. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "latentmoe.h"

#define CHECK(call)                                                  \
  do {                                                               \
    int rc_ = (call);                                                \
    if (rc_ != 0) {                                                  \
      printf("FAILED: %s -> %d (%s)\n", #call, rc_,                  \
             latentmoe_strerror(rc_) ? latentmoe_strerror(rc_) : ""); \
      return 1;                                                      \
    }                                                                \
  } while (0)

#define CUDA(call)                                                            \
  do {                                                                        \
    cudaError_t e_ = (call);                                                  \
    if (e_ != cudaSuccess) {                                                  \
      printf("FAILED: %s -> %s\n", #call, cudaGetErrorString(e_));            \
      return 1;                                                               \
    }                                                                         \
  } while (0)

static uint64_t rng_state = 0x9e3779b97f4a7c15ull;

/* xorshift64*: a uniform double in [-1, 1) */
static double uniform(void) {
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  const uint64_t r = rng_state * 0x2545f4914f6cdd1dull;
  return (double)(r >> 11) / 9007199254740992.0 * 2.0 - 1.0;
}

/* round-to-nearest-even float -> bf16 bits (finite inputs only) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* a device bf16 array of n values, uniform in [-scale, scale) */
static void* device_bf16(size_t n, double scale) {
  uint16_t* h = (uint16_t*)malloc(n * 2);
  void* d = NULL;
  if (h == NULL) return NULL;
  for (size_t i = 0; i < n; ++i) h[i] = to_bf16((float)(uniform() * scale));
  if (cudaMalloc(&d, n * 2) != cudaSuccess || cudaMemcpy(d, h, n * 2, cudaMemcpyHostToDevice) != cudaSuccess)
    d = NULL;
  free(h);
  return d;
}

int main(void) {
  const int64_t T = 300, d = 256, l = 128, E = 16, F = 256, Fs = 256;
  const int k = 2;
  latentmoe_dims dims;
  dims.hidden = d;
  dims.latent = l;
  dims.num_experts = E;
  dims.ffn = F;
  dims.shared_ffn = Fs;
  dims.max_tokens = T;

  latentmoe_weights w;
  memset(&w, 0, sizeof(w));
  w.w_r = device_bf16((size_t)(E * d), 1.0 / sqrt((double)d));
  w.w_dn = device_bf16((size_t)(l * d), 1.0 / sqrt((double)d));
  w.w_g = device_bf16((size_t)(E * F * l), 1.0 / sqrt((double)l));
  w.w_u = device_bf16((size_t)(E * F * l), 1.0 / sqrt((double)l));
  w.w_d = device_bf16((size_t)(E * l * F), 1.0 / sqrt((double)F));
  w.w_up = device_bf16((size_t)(d * l), 1.0 / sqrt((double)l));
  w.w_gs = device_bf16((size_t)(Fs * d), 1.0 / sqrt((double)d));
  w.w_us = device_bf16((size_t)(Fs * d), 1.0 / sqrt((double)d));
  w.w_ds = device_bf16((size_t)(d * Fs), 1.0 / sqrt((double)Fs));
  void* x = device_bf16((size_t)(T * d), 1.0);
  if (!w.w_r || !w.w_dn || !w.w_g || !w.w_u || !w.w_d || !w.w_up || !w.w_gs || !w.w_us ||
      !w.w_ds || !x) {
    printf("FAILED: device allocation\n");
    return 1;
  }
  void* y1 = NULL;
  void* y2 = NULL;
  CUDA(cudaMalloc(&y1, (size_t)(T * d) * 2));
  CUDA(cudaMalloc(&y2, (size_t)(T * d) * 2));

  latentmoe_t h = NULL;
  CHECK(latentmoe_create(&dims, k, 0, &h));
  CHECK(latentmoe_load_weights(h, &w, NULL));
  CHECK(latentmoe_forward(h, x, y1, T, NULL));
  CHECK(latentmoe_forward(h, x, y2, T, NULL));
  uint32_t status = 1;
  CHECK(latentmoe_get_status(h, &status));
  if (status != 0) {
    printf("FAILED: device status %u\n", status);
    return 1;
  }

  uint16_t* a = (uint16_t*)malloc((size_t)(T * d) * 2);
  uint16_t* b = (uint16_t*)malloc((size_t)(T * d) * 2);
  if (a == NULL || b == NULL) return 1;
  CUDA(cudaMemcpy(a, y1, (size_t)(T * d) * 2, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(b, y2, (size_t)(T * d) * 2, cudaMemcpyDeviceToHost));
  double norm = 0.0;
  for (int64_t i = 0; i < T * d; ++i) {
    const float v = from_bf16(a[i]);
    if (!isfinite(v)) {
      printf("FAILED: non-finite output at %lld\n", (long long)i);
      return 1;
    }
    norm += (double)v * v;
  }
  if (!(norm > 0.0)) {
    printf("FAILED: output is all zero\n");
    return 1;
  }
  if (memcmp(a, b, (size_t)(T * d) * 2) != 0) {
    printf("FAILED: two forwards differ\n");
    return 1;
  }
  CHECK(latentmoe_destroy(h));
  printf("ok %.6e\n", sqrt(norm));
  return 0;
}
