/*
 * A plain C caller of the library (no Python, no torch): builds host-only
 * plans (device = -1, no GPU needed) for a small fused model through
 * include/wt.h and prints what the plan compiler decided, one "key value"
 * pair per line, for tests/test_c_abi.py to check.
 *
 * The model: q (256x256, shards 128/128), k and v (128x256, shards 64/64)
 * fused into an FP8 qkv sent whole to ranks 0 and 1; an FP8 gate_up fused
 * from gate and up (512x256 each, shards 256/256) sliced by rows between
 * ranks 0 and 1; a BF16 norm (256x1, shards 200/56) on rank 1.
 */
#include <stdio.h>
#include <string.h>

#include "wt.h"

#define CHECK(call)                                                              \
  do {                                                                           \
    wt_status s_ = (call);                                                       \
    if (s_ != WT_OK) {                                                           \
      printf("error %s %s: %s\n", #call, wt_status_string(s_), wt_last_error()); \
      return 1;                                                                  \
    }                                                                            \
  } while (0)

static int run(uint32_t flags, int32_t local_shard, const char* tag) {
  const int64_t q_sh[2] = {128, 128}, kv_sh[2] = {64, 64}, gu_sh[2] = {256, 256}, n_sh[2] = {200, 56};
  wt_param_desc params[6];
  memset(params, 0, sizeof(params));
  params[0] = (wt_param_desc){"q", 256, 256, 2, q_sh};
  params[1] = (wt_param_desc){"k", 128, 256, 2, kv_sh};
  params[2] = (wt_param_desc){"v", 128, 256, 2, kv_sh};
  params[3] = (wt_param_desc){"gate", 512, 256, 2, gu_sh};
  params[4] = (wt_param_desc){"up", 512, 256, 2, gu_sh};
  params[5] = (wt_param_desc){"norm", 256, 1, 2, n_sh};

  const int32_t qkv_parts[3] = {0, 1, 2}, gu_parts[2] = {3, 4}, n_parts[1] = {5};
  const int32_t both[2] = {0, 1}, one[1] = {1};
  /* gate_up: rank 0 takes fused rows [0, 512), rank 1 rows [512, 1024) */
  const int64_t b0[1] = {0}, b1[1] = {512}, len[1] = {512};
  wt_slice_desc gu_slices[2] = {{0, 1, b0, len}, {0, 1, b1, len}};

  wt_output_desc outs[3];
  memset(outs, 0, sizeof(outs));
  outs[0] = (wt_output_desc){"qkv", 3, qkv_parts, WT_OUT_FP8_E4M3_B128, 2, both, NULL, NULL, NULL};
  outs[1] = (wt_output_desc){"gate_up", 2, gu_parts, WT_OUT_FP8_E4M3_B128, 2, both, NULL, NULL, gu_slices};
  outs[2] = (wt_output_desc){"norm", 1, n_parts, WT_OUT_BF16, 1, one, NULL, NULL, NULL};

  wt_plan_desc d;
  memset(&d, 0, sizeof(d));
  d.num_params = 6;
  d.params = params;
  d.num_outputs = 3;
  d.outputs = outs;
  d.num_ranks = 2;
  d.flags = flags;
  d.local_shard = local_shard;

  wt_plan* p = NULL;
  CHECK(wt_plan_create(&d, -1, &p));
  wt_plan_stats st;
  CHECK(wt_plan_get_stats(p, &st));
  printf("%s.units %lld\n", tag, (long long)st.num_units);
  printf("%s.bytes_read %llu\n", tag, (unsigned long long)st.bytes_read);
  printf("%s.bytes_written %llu\n", tag, (unsigned long long)st.bytes_written);
  printf("%s.slots %d\n", tag, st.num_slots);
  for (int32_t r = 0; r < 2; ++r) {
    uint64_t pool = 0, cnt = 0;
    CHECK(wt_plan_pool_bytes(p, r, &pool));
    CHECK(wt_plan_expected_count(p, r, &cnt));
    printf("%s.pool%d %llu\n", tag, r, (unsigned long long)pool);
    printf("%s.count%d %llu\n", tag, r, (unsigned long long)cnt);
  }
  for (int32_t o = 0; o < 3; ++o)
    for (int32_t k = 0; k < outs[o].num_dsts; ++k) {
      int32_t rank = -1;
      uint64_t doff = 0, soff = 0;
      CHECK(wt_plan_output_layout(p, o, k, &rank, &doff, &soff));
      printf("%s.layout%d.%d %d %llu %llu\n", tag, o, k, rank, (unsigned long long)doff,
             (unsigned long long)soff);
    }
  for (int32_t i = 0; i < 6; ++i)
    for (int32_t s = 0; s < 2; ++s) {
      int64_t rows = 0;
      CHECK(wt_plan_shard_rows_read(p, i, s, &rows));
      printf("%s.read%d.%d %lld\n", tag, i, s, (long long)rows);
    }
  /* a host-only plan refuses to run */
  const void* shards[10] = {0};
  void* pools[2] = {0};
  printf("%s.prepare %s\n", tag, wt_status_string(wt_prepare(p, shards, pools, NULL)));
  CHECK(wt_plan_destroy(p));
  return 0;
}

int main(void) {
  if (run(0, 0, "full")) return 1;
  for (int32_t s = 0; s < 2; ++s) {
    char tag[16];
    snprintf(tag, sizeof(tag), "halo%d", s);
    if (run(WT_FLAG_SHARD_LOCAL | WT_FLAG_SHARD_HALO, s, tag)) return 1;
  }
  printf("null %s\n", wt_status_string(wt_plan_create(NULL, -1, NULL)));
  /* without halos the 64-row k and v shards put a block row across shards:
     the plan is refused (the run prints the error and returns 1) */
  return run(WT_FLAG_SHARD_LOCAL, 0, "strict") == 1 ? 0 : 1;
}
