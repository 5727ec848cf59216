/* The C ABI from C: include/latentmoe.h compiles as C99 and the library's
 * host-side checks answer as documented, with no GPU touched (argument
 * validation happens before any CUDA call). Prints "ok" and exits 0, or
 * names the first failed check and exits 1. */
#include <stdio.h>
#include <string.h>

#include "latentmoe.h"

static int failures = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    printf("FAILED: %s\n", what);
    ++failures;
  }
}

static latentmoe_dims dims(int64_t d, int64_t l, int64_t E, int64_t F, int64_t Fs, int64_t T) {
  latentmoe_dims x;
  x.hidden = d;
  x.latent = l;
  x.num_experts = E;
  x.ffn = F;
  x.shared_ffn = Fs;
  x.max_tokens = T;
  return x;
}

int main(void) {
  latentmoe_t h = (latentmoe_t)0x1;
  latentmoe_dims ok = dims(256, 128, 16, 256, 0, 128);
  latentmoe_dims bad_d = dims(200, 128, 16, 256, 0, 128);
  latentmoe_dims bad_e = dims(256, 128, 513, 256, 0, 128);

  expect(latentmoe_create(&ok, 0, 0, &h) == LATENTMOE_ERR_INVALID_ARG, "k = 0 rejected");
  expect(h == NULL, "handle cleared on error");
  h = (latentmoe_t)0x1;
  expect(latentmoe_create(&ok, 17, 0, &h) == LATENTMOE_ERR_INVALID_ARG, "k = 17 rejected");
  expect(latentmoe_create(&bad_d, 2, 0, &h) == LATENTMOE_ERR_UNSUPPORTED, "d % 128 != 0");
  expect(latentmoe_create(&bad_e, 2, 0, &h) == LATENTMOE_ERR_UNSUPPORTED, "E > 512");
  expect(latentmoe_create(NULL, 2, 0, &h) == LATENTMOE_ERR_INVALID_ARG, "null dims");
  expect(latentmoe_create(&ok, 2, 0, NULL) == LATENTMOE_ERR_INVALID_ARG, "null out");
  expect(latentmoe_destroy(NULL) == LATENTMOE_OK, "destroy(NULL) is a no-op");
  expect(latentmoe_forward(NULL, NULL, NULL, 1, NULL) == LATENTMOE_ERR_INVALID_ARG,
         "forward(NULL)");
  expect(latentmoe_load_weights(NULL, NULL, NULL) == LATENTMOE_ERR_INVALID_ARG, "load(NULL)");
  expect(strcmp(latentmoe_strerror(LATENTMOE_ERR_TIMEOUT), "a bounded device wait timed out") == 0,
         "strerror(TIMEOUT)");
  expect(latentmoe_num_stages() == 10, "ten stages");
  expect(strcmp(latentmoe_stage_name(0), "router") == 0, "stage 0 is the router");
  expect(latentmoe_stage_name(latentmoe_num_stages()) == NULL, "past the last stage");
  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
