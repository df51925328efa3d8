/* A plain C99 client of include/kvc.h: it must compile as C (no C++, no torch
 * types) and link against libkvc.so. It makes only host-side calls, so it runs
 * without a GPU:
 *   budgets <L> <avg> <depth> <n> <alpha>   pyramid budgets, one per line
 *   checks                                  validation and null-handle statuses
 * Used by tests/test_c_abi.py. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvc.h"

static kvc_dims make_dims(int L, int n, int alpha) {
  kvc_dims d;
  memset(&d, 0, sizeof d);
  d.n_layers = L;
  d.batch = 1;
  d.n_q_heads = 32;
  d.n_kv_heads = 8;
  d.head_dim = 128;
  d.prompt_len = n;
  d.obs_window = alpha;
  d.pool_kernel = 7;
  d.bits = 2;
  d.group_size = 32;
  d.window_len = 128;
  d.max_new_tokens = 16;
  return d;
}

int main(int argc, char** argv) {
  if (argc >= 7 && strcmp(argv[1], "budgets") == 0) {
    const int L = atoi(argv[2]), avg = atoi(argv[3]), depth = atoi(argv[4]);
    kvc_dims d = make_dims(L, atoi(argv[5]), atoi(argv[6]));
    int32_t* b = (int32_t*)calloc((size_t)L, sizeof(int32_t));
    kvc_status st = kvc_plan_budgets(&d, KVC_SCHED_PYRAMID, avg, depth, b);
    if (st != KVC_OK) {
      printf("error %d %s\n", (int)st, kvc_status_string(st));
      free(b);
      return 1;
    }
    for (int l = 0; l < L; ++l) printf("%d\n", (int)b[l]);
    free(b);
    return 0;
  }
  if (argc >= 2 && strcmp(argv[1], "checks") == 0) {
    kvc_dims d = make_dims(4, 4096, 32);
    int32_t b[4];
    kvc_dims bad = d;
    bad.head_dim = 96;
    printf("bad_head_dim %d\n", (int)kvc_plan_budgets(&bad, KVC_SCHED_UNIFORM, 64, 0, b));
    bad = d;
    bad.max_new_tokens = KVC_MAX_NEW_TOKENS + 1;
    printf("too_many_new_tokens %d\n", (int)kvc_plan_budgets(&bad, KVC_SCHED_UNIFORM, 64, 0, b));
    printf("uneven_budget %d\n", (int)kvc_plan_budgets(&d, KVC_SCHED_UNIFORM, 48, 0, b));
    printf("null_out %d\n", (int)kvc_plan_budgets(&d, KVC_SCHED_UNIFORM, 64, 0, NULL));
    printf("append_null %d\n", (int)kvc_append(NULL, 0, NULL, NULL, NULL));
    printf("decode_null %d\n", (int)kvc_decode_attn(NULL, 0, 1, NULL, NULL, NULL));
    printf("free_null %d\n", (int)kvc_free(NULL));
    printf("checked_build %d\n", (int)kvc_build_checked());
    printf("launches %llu\n", (unsigned long long)kvc_launch_count());
    printf("status_capacity %s\n", kvc_status_string(KVC_E_CAPACITY));
    return 0;
  }
  fprintf(stderr, "usage: %s budgets L avg depth n alpha | checks\n", argv[0]);
  return 2;
}
