// checked.cuh -- range tests of the checked build (-DZERO_CHECKED).
//
// In libzero_checked.so every kernel tests the global and shared-memory
// ranges it is about to touch against the extents the plan gives (window,
// shard, records, stage slot, unit slices). A failing test skips the access,
// counts the violation and keeps the first one (site << 48 | low 48 bits of
// the index); nothing traps. Each translation unit keeps its own counters
// (device code is not linked across units); zero_checked_status collects
// them. The release build compiles every test away.
#ifndef ZERO_CHECKED_CUH
#define ZERO_CHECKED_CUH

#include <cuda_runtime.h>

#include <cstdint>

enum CheckSite : int {
  kSiteSelftest = 1,
  kSiteScalar = 2,
  kSiteVector = 3,
  kSiteRepCopy = 4,
  kSiteAccCopy = 5,
  kSiteStateCopy = 6,
  kSiteStageBytes = 7,
  kSiteStore = 8,
  kSiteRecord = 9,
  kSiteAccumulate = 10,
  kSiteGather = 11,
  kSiteLoad = 12,
};

#ifdef ZERO_CHECKED
static __device__ unsigned long long g_check_first;
static __device__ unsigned int g_check_count;

static __device__ __noinline__ bool check_failed(int site, int64_t where) {
  atomicAdd(&g_check_count, 1u);
  atomicCAS(&g_check_first, 0ull,
            (static_cast<unsigned long long>(site) << 48) |
                (static_cast<unsigned long long>(where) & 0xFFFFFFFFFFFFull));
  return false;
}
#define ZCHECK(cond, site, where) ((cond) ? true : check_failed((site), (where)))

// this unit's counters: add them to *count, keep the first code if *first
// is still 0, then clear them
static inline int collect_checks(unsigned long long* count, unsigned long long* first) {
  unsigned int c = 0;
  unsigned long long f = 0;
  const unsigned int zc = 0;
  const unsigned long long zf = 0;
  if (cudaMemcpyFromSymbol(&c, g_check_count, sizeof(c)) != cudaSuccess ||
      cudaMemcpyFromSymbol(&f, g_check_first, sizeof(f)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_check_count, &zc, sizeof(zc)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_check_first, &zf, sizeof(zf)) != cudaSuccess)
    return -1;
  *count += c;
  if (*first == 0) *first = f;
  return 0;
}
#else
#define ZCHECK(cond, site, where) true
#endif

#endif
