/* c_abi_host.c — the C ABI from plain C (C99, no CUDA header): includes
 * okc_attn.h, links libokc_attn.so and calls the host-only entry points with
 * the SM count and occupancy given in the options (no GPU needed): status
 * strings, config validation, sizes, the work list and the size bounds.
 * Prints "ok" and returns 0 when every check holds. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "okc_attn.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      printf("FAIL line %d: %s\n", __LINE__, #c);             \
      return 1;                                               \
    }                                                         \
  } while (0)

int main(void) {
  okc_attn_config cfg;
  okc_plan_options opts;
  okc_attn_sizes sizes, bound;
  int32_t seq[4] = {100, 3000, 0, 2047};
  int32_t count = -1, b, i;
  int32_t* items;
  int64_t covered[4] = {0, 0, 0, 0};

  CHECK(strcmp(okc_status_string(OKC_OK), "ok") == 0);
  CHECK(okc_status_string(OKC_ERR_WORKSPACE) != NULL);

  memset(&cfg, 0, sizeof cfg);
  cfg.batch = 4;
  cfg.q_len = 8;
  cfg.num_q_heads = 16;
  cfg.num_kv_heads = 2;
  cfg.head_dim = 64;
  cfg.page_size = 64;
  cfg.window = 2048;
  cfg.max_pages = 64;
  cfg.num_pages = 256;
  cfg.rope_theta = 5e5f;
  cfg.qk_scale_factor = 5.473f;
  cfg.sm_scale = 0.125f;
  cfg.kv_scale = 0.5f;
  memset(&opts, 0, sizeof opts);
  opts.sm_count = 152;
  opts.ctas_per_sm = 1;

  CHECK(okc_attn_plan_sizes(&cfg, seq, &opts, &sizes) == OKC_OK);
  CHECK(sizes.num_tokens == 32 && sizes.num_work >= 4 && sizes.step_kernels == 3);
  CHECK(sizes.workspace_bytes % 256 == 0 && sizes.o_partial_bytes % 256 == 0);
  CHECK(sizes.q_fp8_bytes == 32 * 16 * 64);

  /* the work list covers every request's visible keys exactly once */
  CHECK(okc_attn_plan_items(&cfg, seq, &opts, NULL, 0, &count) == OKC_OK && count == sizes.num_work);
  items = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)count);
  CHECK(items != NULL);
  CHECK(okc_attn_plan_items(&cfg, seq, &opts, items, count, &count) == OKC_OK);
  for (i = 0; i < count; i++) {
    b = items[3 * i];
    CHECK(b >= 0 && b < 4 && items[3 * i + 2] > items[3 * i + 1]);
    covered[b] += items[3 * i + 2] - items[3 * i + 1];
  }
  for (b = 0; b < 4; b++) {
    const int64_t hi = (int64_t)seq[b] + cfg.q_len;
    const int64_t lo = seq[b] - cfg.window + 1 > 0 ? seq[b] - cfg.window + 1 : 0;
    CHECK(covered[b] == hi - lo);
  }
  free(items);

  /* bounds over every step up to the longest context */
  CHECK(okc_attn_plan_max_sizes(&cfg, 3008, &opts, &bound) == OKC_OK);
  CHECK(bound.workspace_bytes >= sizes.workspace_bytes && bound.num_work >= sizes.num_work);
  CHECK(okc_attn_plan_max_sizes(&cfg, 7, &opts, &bound) == OKC_ERR_INVALID); /* below q_len */

  /* validation before any GPU work */
  cfg.head_dim = 128;
  CHECK(okc_attn_plan_sizes(&cfg, seq, &opts, &sizes) == OKC_ERR_UNSUPPORTED);
  cfg.head_dim = 64;
  cfg.q_len = 0;
  CHECK(okc_attn_plan_sizes(&cfg, seq, &opts, &sizes) == OKC_ERR_INVALID);
  cfg.q_len = 8;
  seq[1] = 64 * 64; /* + q_len runs past the page table */
  CHECK(okc_attn_plan_sizes(&cfg, seq, &opts, &sizes) == OKC_ERR_INVALID);
  CHECK(okc_attn_plan_destroy(NULL) == OKC_OK);
  CHECK(okc_selftest_bounded_wait(NULL, 1000, NULL) == OKC_ERR_INVALID);

  printf("ok\n");
  return 0;
}
