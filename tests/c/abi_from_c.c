/* The C ABI used from plain C99: the header compiles without C++, the
 * library links, and the host-only calls behave as documented.  No call here
 * reaches the GPU. */
#include <stdio.h>
#include <string.h>

#include "spec_verify.h"

static int fails = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, #cond); \
      ++fails;                                                   \
    }                                                            \
  } while (0)

int main(void) {
  spec_model_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_layers = 32;
  cfg.d_model = 4096;
  cfg.n_heads = 32;
  cfg.n_kv_heads = 8;
  cfg.d_ffn = 14336;
  cfg.vocab = 128256;
  cfg.rms_eps = 1e-5f;
  cfg.rope_theta = 500000.0f;

  CHECK(spec_model_weight_bytes(&cfg) > (size_t)15000000000ull);
  CHECK(spec_kv_bytes(&cfg, 1, 2048) == (size_t)32 * 1 * 8 * 2048 * 128 * 2);
  CHECK(spec_workspace_bytes(&cfg, 1, 4, 4096) > 0);
  CHECK(spec_workspace_bytes(&cfg, 2, 4, 4096) > spec_workspace_bytes(&cfg, 1, 4, 4096));
  CHECK(spec_accept_workspace_bytes(1, 4, 128256) > 0);

  CHECK(strlen(spec_status_string(SPEC_OK)) > 0);
  CHECK(strlen(spec_status_string(SPEC_EINVAL)) > 0);
  CHECK(strlen(spec_status_string(SPEC_ETIMEOUT)) > 0);

  /* argument validation returns before any CUDA call */
  CHECK(spec_verify_forward(NULL, NULL, 1, 4, NULL, NULL, NULL, 0, NULL) == SPEC_EINVAL);
  CHECK(spec_accept(NULL, NULL, NULL, NULL, 1, 4, 10, 1.0f, 1.0f, NULL, NULL, NULL, 0, NULL) ==
        SPEC_EINVAL);
  CHECK(spec_wait_selftest(NULL, 1, 50.0, NULL, 4, NULL) == SPEC_EINVAL);
  CHECK(spec_device_status(NULL, NULL, NULL) == SPEC_EINVAL);
  CHECK(spec_model_destroy(NULL) == SPEC_OK);

  /* host-only parts: the depth rule and the page pool */
  {
    int32_t g = -1;
    CHECK(spec_gamma_optimal(0.8, 2, 8, 2.0, 20.0, &g) == SPEC_OK);
    CHECK(g >= 2 && g <= 8);
  }
  {
    spec_page_pool* pool = NULL;
    CHECK(spec_page_pool_create(8, 2, 4, &pool) == SPEC_OK);
    CHECK(spec_page_pool_reserve(pool, 0, 130) == SPEC_OK); /* 3 pages of 64 slots */
    CHECK(spec_page_pool_free_pages(pool) == 5);
    CHECK(spec_page_pool_release(pool, 0, 64) == SPEC_OK);  /* keeps 1 page */
    CHECK(spec_page_pool_free_pages(pool) == 7);
    CHECK(spec_page_pool_destroy(pool) == SPEC_OK);
  }

  if (fails) {
    fprintf(stderr, "%d check(s) failed\n", fails);
    return 1;
  }
  printf("ok\n");
  return 0;
}
