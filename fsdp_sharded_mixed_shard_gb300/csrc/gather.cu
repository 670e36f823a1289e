/*
 * gather.cu -- the just-in-time all-gather of stage-3 FSDP units and its
 * inverse, as one HBM-bound copy kernel on sm_103a.
 *
 * "ZeRO Stage 3 Math", "Just-in-time all-gather: how the weights reappear":
 * immediately before a unit runs, the N ranks all-gather so that every rank
 * holds the unit's full parameters; "Training models too big for one GPU:
 * ZeRO & FSDP", "FSDP: the same idea, one unit at a time": the unit's
 * flattened parameters are sharded across the GPUs, gathered, used, freed.
 * With the N ranks' shard buffers resident on one GPU, the all-gather of a
 * window of units is a set of N * units copies ("pieces"), rank r's slice of
 * unit u to offset r * S_u of the unit's buffer, done by one launch per 256
 * pieces.
 *
 * Work is cut into 32 KB tiles of destination bytes, numbered across the
 * pieces; one CTA per tile. A tile is a run of 16-byte aligned
 * destination vectors; each thread issues its eight vectors' loads before its
 * stores (about 96 KB in flight per SM). A window larger than half of L2 is
 * stored evict-first. A slice need not start on a 16-byte boundary (units padded to a
 * multiple of N only), so the source of an aligned destination vector sits
 * at a fixed byte offset d in [0, 16) inside its 16-byte blocks for the whole
 * piece: d = 0 is one 16-byte load; otherwise each source block is loaded
 * once, the next block comes from the neighbouring lane by warp shuffle, and
 * a word select and funnel shift cut out the 16 bytes -- chosen at run time,
 * so that pieces of every phase share a launch. The one or two partial
 * vectors at a piece's ends are copied element by element.
 */
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>

#include "checked.cuh"
#include "pdl.cuh"
#include "zero_internal.h"
#include "zero_units_internal.h"

namespace zg {

constexpr int kMaxPieces = 256;  // copies per launch (8 KB of kernel parameters)
constexpr int kThreads = 256;
constexpr int kVecs = 8;         // 16-byte destination vectors per thread per tile
constexpr int64_t kTileBytes = static_cast<int64_t>(kThreads) * kVecs * 16;
constexpr int64_t kMaxGrid = 1 << 30;

struct Piece {
  const uint8_t* src;
  uint8_t* dst;
  int64_t bytes;  // even, > 0
  int64_t tile0;  // first tile of the piece in the launch's numbering
};

struct Args {
  Piece piece[kMaxPieces];
  int32_t n_pieces;
  int32_t stream_stores;  // 1: evict-first stores (the window is larger than half of L2)
  int64_t n_tiles;
};

// The 16 bytes that start d bytes (d even, 0 < d < 16) into block x and run
// on into block y, the block after it.
__device__ __forceinline__ uint4 bytes_at(const uint4& x, const uint4& y, int d) {
  const uint32_t c[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
  const int q = d >> 2;  // whole words to skip, picked in two select steps
  uint32_t t[6], w[5];
#pragma unroll
  for (int j = 0; j < 6; ++j) t[j] = (q & 2) ? c[j + 2] : c[j];
#pragma unroll
  for (int j = 0; j < 5; ++j) w[j] = (q & 1) ? t[j + 1] : t[j];
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = (d & 2) ? __funnelshift_r(w[k], w[k + 1], 16) : w[k];
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One tile of one piece. Lanes of a warp hold consecutive destination
// vectors, so with d != 0 the source blocks they need are consecutive too:
// each lane loads the one block under its vector's first byte, takes the
// next block from the next lane by shuffle (lane 31 loads its own), and
// every source block is read once. All lanes take part in the shuffles; a
// lane loads only a block that holds at least one byte of the piece's
// source.
__device__ __forceinline__ void copy_tile(const uint8_t* src, int64_t bytes, uintptr_t d0,
                                          int64_t tile, bool stream_stores) {
  const uintptr_t end = d0 + static_cast<uintptr_t>(bytes);
  const uintptr_t s_lo = reinterpret_cast<uintptr_t>(src);
  const uintptr_t s_hi = s_lo + static_cast<uintptr_t>(bytes);
  const uintptr_t a0 =
      (d0 & ~static_cast<uintptr_t>(15)) + static_cast<uintptr_t>(tile) * kTileBytes;
  // the source of an aligned destination address sits d bytes into its
  // 16-byte block, the same d for the whole piece
  const int d = static_cast<int>((s_lo - d0) & 15u);
  const int lane = threadIdx.x & 31;
  uint4 v[kVecs];
  if (d == 0) {
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      const uintptr_t a = a0 + (static_cast<uintptr_t>(k) * kThreads + threadIdx.x) * 16;
      if (a >= d0 && a + 16 <= end &&
          ZCHECK(s_lo + (a - d0) + 16 <= s_hi, kSiteGather, static_cast<int64_t>(a - d0)))
        v[k] = __ldcs(reinterpret_cast<const uint4*>(src + (a - d0)));
    }
  } else {
    uint4 blk[kVecs], nxt[kVecs];
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      const uintptr_t a = a0 + (static_cast<uintptr_t>(k) * kThreads + threadIdx.x) * 16;
      const intptr_t rel = static_cast<intptr_t>(a - d0);  // negative before the piece
      const uintptr_t b = s_lo + static_cast<uintptr_t>(rel) - static_cast<uintptr_t>(d);
      const bool holds = rel + 16 - d > 0 && b < s_hi;
      // a block read must hold a byte of the source (the rest of its 16 bytes
      // lie in the same allocation granule)
      blk[k] = holds && ZCHECK(b + 16 > s_lo && b < s_hi, kSiteGather, rel)
                   ? __ldcs(reinterpret_cast<const uint4*>(b))
                   : make_uint4(0, 0, 0, 0);
      const bool full = a >= d0 && a + 16 <= end;
      nxt[k] = (lane == 31 && full && ZCHECK(b + 16 < s_hi, kSiteGather, rel))
                   ? __ldcs(reinterpret_cast<const uint4*>(b + 16))
                   : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      uint4 y;
      y.x = __shfl_down_sync(0xffffffffu, blk[k].x, 1);
      y.y = __shfl_down_sync(0xffffffffu, blk[k].y, 1);
      y.z = __shfl_down_sync(0xffffffffu, blk[k].z, 1);
      y.w = __shfl_down_sync(0xffffffffu, blk[k].w, 1);
      if (lane == 31) y = nxt[k];
      v[k] = bytes_at(blk[k], y, d);
    }
  }
#pragma unroll
  for (int k = 0; k < kVecs; ++k) {
    const uintptr_t a = a0 + (static_cast<uintptr_t>(k) * kThreads + threadIdx.x) * 16;
    if (a >= d0 && a + 16 <= end) {
      if (stream_stores) __stcs(reinterpret_cast<uint4*>(a), v[k]);
      else *reinterpret_cast<uint4*>(a) = v[k];
    } else if (a + 16 > d0 && a < end) {  // a partial vector at one end of the piece
      const uintptr_t lo = a > d0 ? a : d0;
      const uintptr_t hi = a + 16 < end ? a + 16 : end;
      for (uintptr_t b = lo; b < hi; b += 2)
        *reinterpret_cast<uint16_t*>(b) = *reinterpret_cast<const uint16_t*>(src + (b - d0));
    }
  }
}

__global__ void __launch_bounds__(kThreads) copy_kernel(const __grid_constant__ Args a) {
  pdl_begin();
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    // the piece holding tile t: the last one whose first tile is <= t
    int lo = 0, hi = a.n_pieces - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.piece[mid].tile0 <= t) lo = mid;
      else hi = mid - 1;
    }
    copy_tile(a.piece[lo].src, a.piece[lo].bytes, reinterpret_cast<uintptr_t>(a.piece[lo].dst),
              t - a.piece[lo].tile0, a.stream_stores != 0);
  }
}

// One CTA per tile: the hardware hands tiles to SMs as CTAs finish, which
// balanced the SMs best. Measured on 220 MB units, in fractions of copy
// bandwidth: one persistent wave 84 %, 8 CTAs per SM 90 %, 16 per SM 93.6 %,
// 32 per SM 94.5 %, one per tile 94.8 %. The stride loop only matters past
// the grid limit.
int flush(Args& a, cudaStream_t stream) {
  if (a.n_pieces == 0) return ZERO_OK;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(a.n_tiles, kMaxGrid));
  const cudaError_t e = launch_pdl(copy_kernel, dim3(grid), dim3(kThreads), 0, stream, a);
  a.n_pieces = 0;
  a.n_tiles = 0;  // stream_stores is kept for the next batch
  return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}

// gather: shards -> unit buffers; otherwise unit buffers -> shards
int copy_units(const zero_unit_plan* plan, int32_t unit_lo, int32_t unit_hi,
               const void* const* shards, void* const* unit_buffers, bool gather,
               void* stream) {
  if (!plan || !shards || !unit_buffers) return ZERO_EINVAL;
  if (unit_lo < 0 || unit_hi > plan->info.n_units || unit_lo >= unit_hi) return ZERO_EINVAL;
  const int32_t N = plan->info.n_ranks;
  for (int32_t r = 0; r < N; ++r) {
    if (!shards[r]) return ZERO_EINVAL;
    if (!zero_detail::aligned16(shards[r])) return ZERO_EALIGN;
  }
  for (int32_t u = unit_lo; u < unit_hi; ++u) {
    if (!unit_buffers[u - unit_lo]) return ZERO_EINVAL;
    if (!zero_detail::aligned16(unit_buffers[u - unit_lo])) return ZERO_EALIGN;
  }
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
    return ZERO_ECUDA;
  Args* a = new (std::nothrow) Args;
  if (!a) return ZERO_ENOMEM;
  std::memset(a, 0, sizeof(Args));
  // A window that fits in half of L2 is written normally, so that the layer
  // about to use it finds it there; a larger one streams past L2.
  int64_t window_bytes = 0;
  for (int32_t u = unit_lo; u < unit_hi; ++u) window_bytes += 2 * plan->units[u].psi_pad;
  a->stream_stores = window_bytes > static_cast<int64_t>(l2) / 2 ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = ZERO_OK;
  for (int32_t u = unit_lo; u < unit_hi && rc == ZERO_OK; ++u) {
    const zero_unit& U = plan->units[u];
    if (U.shard_elems == 0) continue;
    const int64_t bytes = 2 * U.shard_elems;
    uint8_t* unit_base = static_cast<uint8_t*>(unit_buffers[u - unit_lo]);
    for (int32_t r = 0; r < N && rc == ZERO_OK; ++r) {
      uint8_t* slice = const_cast<uint8_t*>(static_cast<const uint8_t*>(shards[r])) +
                       2 * U.shard_offset;
      uint8_t* part = unit_base + 2 * static_cast<int64_t>(r) * U.shard_elems;
      Piece& p = a->piece[a->n_pieces];
      p.src = gather ? slice : part;
      p.dst = gather ? part : slice;
      p.bytes = bytes;
      p.tile0 = a->n_tiles;
      const uintptr_t d0 = reinterpret_cast<uintptr_t>(p.dst);
      const int64_t span = static_cast<int64_t>(d0 + static_cast<uintptr_t>(bytes) -
                                                (d0 & ~static_cast<uintptr_t>(15)));
      a->n_tiles += (span + kTileBytes - 1) / kTileBytes;
      if (++a->n_pieces == kMaxPieces) rc = flush(*a, st);
    }
  }
  if (rc == ZERO_OK) rc = flush(*a, st);
  delete a;
  return rc;
}

}  // namespace zg

#ifdef ZERO_CHECKED
// this unit's counters, for zero_checked_status
extern "C" int zg_collect_checks(unsigned long long* count, unsigned long long* first) {
  return collect_checks(count, first);
}
#endif

extern "C" {

ZERO_API int zero_gather_units(const zero_unit_plan* plan, int32_t unit_lo, int32_t unit_hi,
                               const void* const* shards, void* const* unit_buffers,
                               void* stream) {
  return zg::copy_units(plan, unit_lo, unit_hi, shards, unit_buffers, true, stream);
}

ZERO_API int zero_shard_units(const zero_unit_plan* plan, int32_t unit_lo, int32_t unit_hi,
                              const void* const* unit_buffers, void* const* shards,
                              void* stream) {
  // the shard buffers are the destinations here; the pointer checks are the same
  return zg::copy_units(plan, unit_lo, unit_hi, const_cast<const void* const*>(shards),
                        const_cast<void* const*>(unit_buffers), false, stream);
}

}  // extern "C"
