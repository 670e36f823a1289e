// Host planner under AddressSanitizer / UBSan: random tensor lists, rank
// counts, bucket sizes and unit layouts through every host entry point of
// zero.h and zero_units.h, with the layout invariants checked on the way.
// Built and run by tests/test_sanitizers.py (CPU only).
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "zero.h"
#include "zero_units.h"

static uint64_t g_state = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64() {  // xorshift64*
  g_state ^= g_state >> 12;
  g_state ^= g_state << 25;
  g_state ^= g_state >> 27;
  return g_state * 2685821657736338717ull;
}
static int64_t pick(const int64_t* v, int n) { return v[next_u64() % n]; }

#define CHECK(c)                                                     \
  do {                                                               \
    if (!(c)) {                                                      \
      std::fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
      return 1;                                                      \
    }                                                                \
  } while (0)

static int flat_case() {
  const int64_t sizes[] = {0, 1, 2, 7, 31, 4096, 10007, 65536};
  const int64_t buckets[] = {0, 1, 3, 64, 1000, 4096, 99991};
  const int64_t ranks[] = {1, 2, 3, 4, 7, 8, 16, 63, 64};
  const int nt = static_cast<int>(next_u64() % 9);
  std::vector<int64_t> numels(nt);
  for (auto& x : numels) x = pick(sizes, 8);
  const int32_t n = static_cast<int32_t>(pick(ranks, 9));
  const int64_t b = pick(buckets, 7);
  const zero_dtype dt = (next_u64() & 1) ? ZERO_BF16 : ZERO_FP16;
  zero_plan* p = nullptr;
  CHECK(zero_plan_create(numels.data(), nt, n, b, dt, &p) == ZERO_OK && p);
  zero_plan_info info;
  CHECK(zero_plan_get_info(p, &info) == ZERO_OK);
  CHECK(info.psi_pad % n == 0 && info.pad < n && info.shard_elems * n == info.psi_pad);
  std::vector<int64_t> offs(nt > 0 ? nt : 1);
  CHECK(zero_plan_tensor_offsets(p, offs.data()) == ZERO_OK);
  std::vector<zero_segment> segs(info.n_segments > 0 ? info.n_segments : 1);
  CHECK(zero_plan_segments(p, segs.data(), info.n_segments) == ZERO_OK);
  int64_t at = 0;
  for (int32_t i = 0; i < info.n_segments; ++i) {  // segments tile [0, psi_pad) in order
    CHECK(segs[i].lo == at && segs[i].hi > segs[i].lo);
    CHECK(segs[i].lo / info.shard_elems == segs[i].rank);
    at = segs[i].hi;
  }
  CHECK(at == info.psi_pad);
  for (int32_t k = 0; k < info.n_buckets; ++k) {
    int64_t lo = -1, hi = -1;
    CHECK(zero_plan_bucket_range(p, k, &lo, &hi) == ZERO_OK && lo < hi);
  }
  int64_t lo = 0, hi = 0;
  CHECK(zero_plan_bucket_range(p, info.n_buckets, &lo, &hi) != ZERO_OK);
  if (info.n_segments > 0) CHECK(zero_plan_segments(p, segs.data(), info.n_segments - 1) != ZERO_OK);
  CHECK(zero_workspace_bytes(p, 1) >=
        static_cast<size_t>(info.n_tiles + static_cast<int64_t>(n) * ZERO_NORM_OWNER_BLOCKS) * 16);
  CHECK(zero_workspace_bytes(p, 0) == 0);
  // all buckets and segments at once: each bucket's segments are one run
  // that tiles its range
  std::vector<zero_bucket> bk(info.n_buckets > 0 ? info.n_buckets : 1);
  std::vector<zero_segment> segs2(info.n_segments > 0 ? info.n_segments : 1);
  CHECK(zero_plan_buckets(p, bk.data(), segs2.data()) == ZERO_OK);
  CHECK(zero_plan_buckets(p, nullptr, nullptr) == ZERO_OK);
  for (int32_t k = 0; k < info.n_buckets; ++k) {
    int64_t covered = 0;
    for (int32_t s = bk[k].seg_first; s < bk[k].seg_first + bk[k].seg_count; ++s) {
      CHECK(s >= 0 && s < info.n_segments && segs2[s].bucket == k);
      covered += segs2[s].hi - segs2[s].lo;
    }
    CHECK(covered == bk[k].hi - bk[k].lo);
  }
  zero_plan_info alias;
  CHECK(zero_plan_info_get(p, &alias) == ZERO_OK && alias.psi == info.psi);
  zero_plan_destroy(p);
  return 0;
}

static int unit_case() {
  const int64_t sizes[] = {0, 1, 3, 8, 255, 4096, 10007};
  const int64_t ranks[] = {1, 2, 3, 8, 13, 64};
  const int64_t aligns[] = {1, 2, 8, 64};
  const int nt = 1 + static_cast<int>(next_u64() % 9);
  const int nu = 1 + static_cast<int>(next_u64() % nt);
  std::vector<int64_t> numels(nt);
  std::vector<int32_t> uot(nt);
  for (int k = 0; k < nt; ++k) {
    numels[k] = pick(sizes, 7);
    uot[k] = k < nu ? k : static_cast<int32_t>(next_u64() % nu);
  }
  const int32_t n = static_cast<int32_t>(pick(ranks, 6));
  const int32_t al = static_cast<int32_t>(pick(aligns, 4));
  zero_unit_plan* p = nullptr;
  CHECK(zero_unit_plan_create(numels.data(), nt, uot.data(), nu, n, al, &p) == ZERO_OK && p);
  zero_unit_plan_info info;
  CHECK(zero_unit_plan_get_info(p, &info) == ZERO_OK);
  std::vector<zero_unit> units(nu);
  CHECK(zero_unit_plan_units(p, units.data(), nu) == ZERO_OK);
  CHECK(zero_unit_plan_units(p, units.data(), nu - 1) != ZERO_OK);
  std::vector<int32_t> slots(nt);
  std::vector<int64_t> toff(nt);
  CHECK(zero_unit_plan_tensors(p, slots.data(), toff.data(), nt) == ZERO_OK);
  int64_t held = 0, flat = 0;
  for (int u = 0; u < nu; ++u) {
    CHECK(units[u].psi_pad % (static_cast<int64_t>(n) * al) == 0);
    CHECK(units[u].shard_offset == held && units[u].flat_offset == flat);
    held += units[u].shard_elems;
    flat += units[u].psi_pad;
  }
  CHECK(held == info.shard_elems && flat == info.psi_pad);
  for (int s = 0; s < 5; ++s) {
    zero_strategy_cost c;
    CHECK(zero_unit_plan_strategy_cost(p, s, 1, &c) == ZERO_OK);
    CHECK(c.persistent_bytes >= 0 && c.peak_bytes >= c.persistent_bytes);
  }
  zero_strategy_cost c;
  CHECK(zero_unit_plan_strategy_cost(p, ZERO_HYBRID_SHARD, 3, &c) == ZERO_OK);
  CHECK(zero_unit_plan_strategy_cost(p, 9, 1, &c) != ZERO_OK);
  zero_unit_plan_destroy(p);
  return 0;
}

static int bad_arguments() {
  const int64_t ok[] = {10, 20};
  const int64_t neg[] = {10, -1};
  const int32_t uot_bad[] = {0, 5};
  zero_plan* p = nullptr;
  CHECK(zero_plan_create(ok, 2, 0, 0, ZERO_BF16, &p) != ZERO_OK && !p);
  CHECK(zero_plan_create(neg, 2, 2, 0, ZERO_BF16, &p) != ZERO_OK && !p);
  CHECK(zero_plan_create(ok, 2, 65, 0, ZERO_BF16, &p) != ZERO_OK && !p);
  zero_unit_plan* u = nullptr;
  CHECK(zero_unit_plan_create(ok, 2, uot_bad, 2, 2, 1, &u) != ZERO_OK && !u);
  zero_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 1, 0, 1.0};
  zero_scaler s;
  CHECK(zero_scaler_init(&hp, &s) != ZERO_OK);
  hp.growth_interval = 2000;
  CHECK(zero_scaler_init(&hp, &s) == ZERO_OK && s.scale == 1.0f);
  for (int st = -8; st <= 1; ++st) CHECK(zero_strerror(st) != nullptr);
  return 0;
}

int main(int argc, char** argv) {
  const int iters = argc > 1 ? std::atoi(argv[1]) : 2000;
  for (int i = 0; i < iters; ++i) {
    if (flat_case()) return 1;
    if (unit_case()) return 1;
  }
  if (bad_arguments()) return 1;
  std::printf("planner_fuzz ok %d\n", iters);
  return 0;
}
