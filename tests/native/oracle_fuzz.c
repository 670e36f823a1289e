/* The CPU checker under AddressSanitizer / UBSan: the planners, casts, the
 * array-driven step (plain, clipped, sharded subsets, micro-batches), the
 * generator-driven step (with worker threads) and the unit gather on small
 * random inputs. Built and run by tests/test_sanitizers.py (CPU only). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

static uint64_t g_state = 0x2545F4914F6CDD1Dull;
static uint64_t next_u64(void) {
  g_state ^= g_state >> 12;
  g_state ^= g_state << 25;
  g_state ^= g_state >> 27;
  return g_state * 2685821657736338717ull;
}

#define CHECK(c)                                                            \
  do {                                                                      \
    if (!(c)) {                                                             \
      fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__);        \
      return 1;                                                             \
    }                                                                       \
  } while (0)

static int step_case(int clip, int micro) {
  const int32_t n = 1 + (int32_t)(next_u64() % 8);
  const int32_t nt = 1 + (int32_t)(next_u64() % 4);
  int64_t numels[4];
  for (int k = 0; k < nt; ++k) numels[k] = (int64_t)(next_u64() % 3000);
  const int64_t bucket = (next_u64() & 1) ? 0 : 1 + (int64_t)(next_u64() % 2000);
  orc_plan p;
  orc_segment segs[4096];
  CHECK(orc_plan_make(numels, nt, n, bucket, &p, NULL, segs, 4096) == 0);
  const int64_t m = p.psi_pad;
  const int32_t bf = (int32_t)(next_u64() & 1);
  uint16_t** reps = malloc(sizeof(uint16_t*) * n);
  float** acc = malloc(sizeof(float*) * n);
  for (int r = 0; r < n; ++r) {
    reps[r] = malloc(sizeof(uint16_t) * (size_t)(m > 0 ? m : 1));
    acc[r] = malloc(sizeof(float) * (size_t)(m > 0 ? m : 1));
    for (int64_t j = 0; j < m; ++j) {
      const float x = j < p.psi ? (float)((int64_t)(next_u64() % 2001) - 1000) * 1e-4f : 0.0f;
      reps[r][j] = bf ? orc_f32_to_bf16(x) : orc_f32_to_f16(x);
    }
    orc_accumulate(reps[r], acc[r], m, bf, 1);
    if (micro) orc_accumulate(reps[r], acc[r], m, bf, 0);
  }
  float* master = calloc((size_t)(m > 0 ? m : 1), sizeof(float));
  float* mm = calloc((size_t)(m > 0 ? m : 1), sizeof(float));
  float* vv = calloc((size_t)(m > 0 ? m : 1), sizeof(float));
  float* ghat = calloc((size_t)(m > 0 ? m : 1), sizeof(float));
  uint16_t* params = calloc((size_t)(m > 0 ? m : 1), sizeof(uint16_t));
  uint32_t flags[4096] = {0};
  orc_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01, clip ? 0.5 : 0.0, 1, 2000};
  orc_scaler sc = {1.0f, 0, 0, 0, 0.0, 0.0, 1.0f, 0};
  /* a subset of owners, as the sharded drivers run them */
  const int32_t lo = (int32_t)(next_u64() % (uint64_t)n);
  const int32_t hi = lo + 1 + (int32_t)(next_u64() % (uint64_t)(n - lo));
  int rc;
  if (micro)
    rc = orc_step_arrays_f32(&p, lo, hi, bf, (const float* const*)acc, 2, 0, master, mm, vv,
                             params, ghat, flags, &hp, &sc);
  else
    rc = orc_step_arrays(&p, lo, hi, bf, (const uint16_t* const*)reps, 0, master, mm, vv,
                         params, ghat, flags, &hp, &sc);
  CHECK(rc == 0);
  CHECK(sc.t == 1);
  for (int r = 0; r < n; ++r) {
    free(reps[r]);
    free(acc[r]);
  }
  free(reps);
  free(acc);
  free(master);
  free(mm);
  free(vv);
  free(ghat);
  free(params);
  return 0;
}

static int gen_case(void) {
  const int64_t numels[1] = {(int64_t)(1 + next_u64() % 300000)};
  const int32_t n = 1 + (int32_t)(next_u64() % 8);
  orc_plan p;
  CHECK(orc_plan_make(numels, 1, n, 0, &p, NULL, NULL, 0) == 0);
  orc_gen g;
  memset(&g, 0, sizeof(g));
  g.spec.seed = next_u64();
  g.spec.sigma = 1e-3f;
  g.spec.loss_scale = 1.0f;
  g.spec.psi = p.psi;
  g.is_bf16 = 1;
  g.inject_step = -1;
  int64_t elems[3] = {0, p.psi_pad / 2, p.psi_pad - 1};
  float master[3] = {0.01f, -0.02f, 0.0f}, mm[3] = {0}, vv[3] = {0};
  uint16_t params[3] = {0};
  uint32_t flags[1] = {0};
  orc_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 0, 2000};
  orc_scaler sc = {1.0f, 0, 0, 0, 0.0, 0.0, 1.0f, 0};
  CHECK(orc_gen_step(&p, 0, n, &g, 1, 3, elems, 3, master, mm, vv, params, flags, &hp, &sc) == 0);
  float gh[3];
  CHECK(orc_gen_ghat(&p, &g, 1, 1.0f, elems, 3, gh) == 0);
  return 0;
}

static int unit_case(void) {
  const int32_t nt = 1 + (int32_t)(next_u64() % 8);
  const int32_t nu = 1 + (int32_t)(next_u64() % (uint64_t)nt);
  int64_t numels[8];
  int32_t uot[8];
  for (int k = 0; k < nt; ++k) {
    numels[k] = (int64_t)(next_u64() % 5000);
    uot[k] = k < nu ? k : (int32_t)(next_u64() % (uint64_t)nu);
  }
  const int32_t n = 1 + (int32_t)(next_u64() % 16);
  const int32_t al = (next_u64() & 1) ? 1 : 8;
  orc_unit_plan p;
  orc_unit units[8];
  int32_t slots[8];
  int64_t toff[8];
  CHECK(orc_unit_plan_make(numels, nt, uot, nu, n, al, &p, units, slots, toff) == 0);
  uint16_t** shards = malloc(sizeof(uint16_t*) * n);
  for (int r = 0; r < n; ++r) {
    shards[r] = malloc(sizeof(uint16_t) * (size_t)(p.shard > 0 ? p.shard : 1));
    for (int64_t j = 0; j < p.shard; ++j) shards[r][j] = (uint16_t)next_u64();
  }
  for (int u = 0; u < nu; ++u) {
    uint16_t* full = malloc(sizeof(uint16_t) * (size_t)(units[u].psi_pad > 0 ? units[u].psi_pad : 1));
    orc_gather_unit(&units[u], n, (const uint16_t* const*)shards, full);
    orc_shard_unit(&units[u], n, full, shards);
    free(full);
  }
  for (int s = 0; s < 5; ++s) {
    orc_strategy_cost c;
    CHECK(orc_strategy_cost_make(&p, s, 1, &c) == 0);
  }
  for (int r = 0; r < n; ++r) free(shards[r]);
  free(shards);
  return 0;
}

int main(int argc, char** argv) {
  const int iters = argc > 1 ? atoi(argv[1]) : 200;
  for (int i = 0; i < iters; ++i) {
    if (step_case(i & 1, (i >> 1) & 1)) return 1;
    if (unit_case()) return 1;
    if (i % 20 == 0 && gen_case()) return 1;
  }
  for (uint32_t b = 0; b < 65536; b += 7) {
    volatile float a = orc_f16_to_f32((uint16_t)b), c = orc_bf16_to_f32((uint16_t)b);
    (void)orc_f32_to_f16(a);
    (void)orc_f32_to_bf16(c);
  }
  printf("oracle_fuzz ok %d\n", iters);
  return 0;
}
