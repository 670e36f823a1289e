/*
 * zero_kernels.cu -- sm_103a kernels of the sharded mixed-precision AdamW step
 * and the launch layer behind the C ABI (zero.h).
 *
 * Kernels
 *   bulk_kernel<MODE, dtype, ...>  the three streaming passes, each a
 *                             persistent cp.async.bulk + mbarrier pipeline
 *                             (one producer warp, sixteen consumer warps):
 *     kFused  reduce-scatter + unscale + non-finite vote + AdamW + cast in one
 *             pass; reads the current optimizer set, writes the other one
 *             (2N + 26 bytes per element);
 *     kReduce reduce-scatter + unscale + vote, writes fp32 g and the per-tile
 *             squared-norm records (2N + 4 bytes per element);
 *     kUpdate AdamW + cast from fp32 g after the overflow and clip decisions
 *             are known (30 bytes per element): into the other state set when
 *             the caller gives two (measured about 4 % faster on GB300 than
 *             writing each array back where it was read), else in place.
 *   step_kernel<MODE, dtype>  a plain tile-scheduled kernel for the two light
 *                             modes:
 *     kNorm   per-tile squared-norm records from fp32 g (4 bytes per element);
 *     kCast   16-bit working copy from an fp32 master set (6 bytes per element),
 *             optionally only when the step's overflow word is set, and then
 *             the step's bookkeeping in the last CTA.
 *   norm_owner_kernel,        fixed-partition float-float merge of each
 *   norm_final_kernel,        owner's tile records; owner records merged in
 *   norm_import_kernel        ascending owner order; fp64 norm and clip
 *                             coefficient (or the owner records exported for
 *                             a cross-process exchange, and their import).
 *   scaler_finish_kernel      loss-scale / skip / step-count bookkeeping (one
 *                             thread).
 *   short_fused_kernel        a whole fused step of at most 2^20 elements at
 *                             N <= 16: one wave of 256-thread CTAs without
 *                             the copy pipeline, each thread four elements,
 *                             the bookkeeping in the last CTA.
 *   ring_hop_kernel           one rank's part of one hop of the reduce-scatter
 *                             when the ranks are separate processes.
 *
 * Work decomposition: the owned elements are cut into segments (one bucket of
 * one rank) and each segment into tiles of ZERO_TILE_ELEMS elements. A
 * persistent grid walks the tiles round-robin. In the bulk passes an owner
 * whose slice starts off the windows' 8-element grid gets a shard-indexed
 * body whose replica chunks are copied from the 16-byte block below their
 * first element (see tile_geom); the few elements of a tile outside its
 * body take per-element paths.
 *
 * Arithmetic: every fp32 operation of the step is an explicit round-to-
 * nearest-even intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn) and
 * the file is built with --fmad=false, so results are the IEEE results of the
 * stated operation sequence; no flush-to-zero. Sum order: for owner i the
 * replicas are added in ring order i+1, ..., N-1, 0, ..., i ("How far does
 * splitting the batch get you?", "Why does the all-reduce not get more
 * expensive with more ranks?": a chunk is summed hop by hop around the ring
 * and is complete at rank i).
 */
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "checked.cuh"
#include "f64emu.h"
#include "pdl.cuh"
#include "zero_internal.h"

namespace zk {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = ZERO_TILE_ELEMS;
constexpr int kVec = 8;                       // 16-bit elements per 16-byte vector
constexpr int kMaxSegs = 128;                 // segments per launch (kernel parameter space)

static_assert(kTile % (kVec * kThreads) == 0, "tile must be a whole number of vector passes");

enum Mode : int { kFused = 0, kReduce = 1, kUpdate = 2, kNorm = 3, kCast = 4 };

// mode flags
constexpr int kFlagClip = 1;        // kUpdate: apply the clip coefficient from the scaler
constexpr int kFlagIfPending = 2;   // kCast: only when the overflow word is set
constexpr int kFlagUseScalerSet = 4;// kCast: master set = scaler->state_index
constexpr int kFlagPartials = 8;    // kReduce: write norm partials
constexpr int kFlagFinish = 16;     // kCast, kFused: also do the step's bookkeeping (once, last CTA)

struct Seg {
  int64_t lo, hi;          // flat element range
  int64_t tile_local0;     // first tile of this segment in this launch's numbering
  int64_t tile_global0;    // first tile in the plan's numbering (norm partial index)
  int32_t rank, bucket;
};

// Bulk pipeline stage plan for one element range (2048 or 4096 elements):
// stage i carries the replica chunks of ring positions [r_lo[i], r_hi[i])
// and, when states[i] is set, the state block (kFused: master, m, v;
// kUpdate: g, master, m, v) after them.
// 64 ranks with fp32 accumulators need 13 replica stages plus one state stage
constexpr int kMaxStagePlan = 16;
struct StagePlan {
  int32_t n;
  int16_t r_lo[kMaxStagePlan], r_hi[kMaxStagePlan];
  int32_t states[kMaxStagePlan];
  int32_t bytes_per_elem[kMaxStagePlan];
};

struct Args {
  const uint16_t* rep[ZERO_MAX_RANKS];      // replica windows (the last micro-batch's gradients)
  const float* acc[ZERO_MAX_RANKS];         // fp32 accumulators of the earlier micro-batches
  float* master[2][ZERO_MAX_RANKS];
  float* mom[2][ZERO_MAX_RANKS];
  float* var[2][ZERO_MAX_RANKS];
  float* ghat[ZERO_MAX_RANKS];
  uint16_t* flat;                           // parameter window
  zero_scaler* scaler;
  uint32_t* flags;
  float4* partials;  // norm records: one (hi, lo, bhi, blo) per tile
  int64_t wbase, shard, n_tiles;
  int32_t n_ranks, n_segs, n_sets, mode_flags;
  // step constants rounded once from the fp64 hyperparameters
  float b1, omb1, b2, omb2, lr, decay, eps;
  int32_t bk_dynamic, bk_growth, bk_flip;  // bookkeeping (kFlagFinish)
  int32_t n_micro;                          // micro-batches in this step (>= 1)
  int32_t has_acc;                          // 1: replica value = acc + 16-bit micro-batch value
  int32_t pad1;
  int64_t bucket_elems;                     // the plan's bucket size (0 = one bucket)
  double beta1, beta2;
  int64_t wend;       // window indices of this launch lie in [0, wend) (checked builds)
  int64_t n_records;  // norm records the workspace holds (checked builds)
  StagePlan plan;  // bulk pipeline: stages of one element range
  Seg segs[kMaxSegs];
};

// CUDA 12.1+ accepts up to 32,764 bytes of kernel parameters on sm_70 and newer
static_assert(sizeof(Args) <= 32000, "kernel arguments exceed the parameter space");

// per-CTA step scalars that depend on device-resident state
struct StepScalars {
  float inv;       // fp32(1 / (S_l * N))
  float bc1, bc2;  // fp32(1 - beta^(t+1))
  float clip;      // clip coefficient (1 when it does not apply)
  int src;         // optimizer set read
  int dst;         // optimizer set written
  int skip;        // 1: nothing to do in this launch
};

// Checked builds: see checked.cuh.
// one planted violation, to test the reporting path
#ifdef ZERO_CHECKED
__global__ void check_selftest_kernel() { (void)ZCHECK(threadIdx.x > 0, kSiteSelftest, 42); }
#endif

// ------------------------------------------------------------ primitives --

// Exact 16-bit -> fp32 widening: bf16 is the top half of an fp32; fp16 goes
// through the hardware conversion (measured faster than an integer/fp32-ALU
// rebuild of the bits).
template <bool kBf16>
__device__ __forceinline__ float widen(uint32_t h16) {
  if constexpr (kBf16) {
    return __uint_as_float(h16 << 16);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h16)));
  }
}

template <bool kBf16>
__device__ __forceinline__ uint16_t narrow(float x) {
  if constexpr (kBf16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  } else {
    return __half_as_ushort(__float2half_rn(x));
  }
}

template <bool kBf16>
__device__ __forceinline__ uint4 narrow8(const float (&x)[8]) {
  uint32_t u[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    u[k] = static_cast<uint32_t>(narrow<kBf16>(x[2 * k])) |
           (static_cast<uint32_t>(narrow<kBf16>(x[2 * k + 1])) << 16);
  return make_uint4(u[0], u[1], u[2], u[3]);
}

__device__ __forceinline__ bool nonfinite(float x) {
  return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

__device__ __forceinline__ void load8f(const float* p, float (&x)[8]) {
  float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// One AdamW update ("Training models too big for one GPU: ZeRO & FSDP",
// "Adam, and why it's expensive"; decoupled weight decay):
//   m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; mh = m/bc1; vh = v/bc2;
//   theta = theta (1 - lr wd) - lr mh / (sqrt(vh) + eps)
__device__ __forceinline__ void adamw(float& th, float& m, float& v, float g, const Args& a,
                                      const StepScalars& s) {
  float m_new = __fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.omb1, g));
  float gg = __fmul_rn(g, g);
  float v_new = __fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.omb2, gg));
  float mh = __fdiv_rn(m_new, s.bc1);
  float vh = __fdiv_rn(v_new, s.bc2);
  float den = __fadd_rn(__fsqrt_rn(vh), a.eps);
  float u = __fdiv_rn(mh, den);
  th = __fsub_rn(__fmul_rn(th, a.decay), __fmul_rn(a.lr, u));
  m = m_new;
  v = v_new;
}

// Squared-gradient accumulation with a float-float (hi, lo) pair: the square
// is split exactly into p + e (e = fma(g, g, -p)), p is added with an exact
// two-sum and all error terms collect in lo (relative accuracy ~2^-44 over a
// tile). Everything here is fp32: GB300's fp64 path is far too slow for
// per-element work. Magnitudes |g| >= 2^56 are scaled by 2^-96 and summed in
// a second pair (bhi, blo) that stands for 2^192 times its value, so no
// per-tile sum can overflow; a NaN or infinite g lands in the second pair
// and leaves it non-finite. Squares below 2^-126 are fp32 subnormals
// (absolute error < 2^-149 each).
__device__ __forceinline__ void ff_add_sq(float& hi, float& lo, float g) {
  float p = __fmul_rn(g, g);
  float e = __fmaf_rn(g, g, -p);
  float s = __fadd_rn(hi, p);
  float bb = __fsub_rn(s, hi);
  float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(p, bb));
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(err, e));
}

__device__ __forceinline__ void ff_merge(float& hi, float& lo, float h2, float l2) {
  float s = __fadd_rn(hi, h2);
  float bb = __fsub_rn(s, hi);
  float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(h2, bb));
  hi = s;
  lo = __fadd_rn(__fadd_rn(lo, l2), err);
}

constexpr float kNormMainLimit = 0x1p56f;
constexpr float kNormBigScale = 0x1p-96f;
// a running sum of squares below this holds no square of a |g| >= 2^56
constexpr float kNormSumLimit = 0x1p112f;

// Packed form of ff_add_sq for two independent accumulators at once, with
// sm_100+'s paired fp32 instructions (PTX add/sub/mul/fma .rn.f32x2: each
// lane is the ordinary IEEE fp32 operation, so lane k computes exactly what
// ff_add_sq computes).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t x, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_neg(uint64_t a) { return a ^ 0x8000000080000000ull; }

__device__ __forceinline__ void ff2_add_sq(uint64_t& hi, uint64_t& lo, uint64_t g) {
  const uint64_t p = f2_mul(g, g);
  const uint64_t e = f2_fma(g, g, f2_neg(p));
  const uint64_t s = f2_add(hi, p);
  const uint64_t bb = f2_sub(s, hi);
  const uint64_t err = f2_add(f2_sub(hi, f2_sub(s, bb)), f2_sub(p, bb));
  hi = s;
  lo = f2_add(lo, f2_add(err, e));
}

struct NormAcc {
  float hi = 0.f, lo = 0.f;    // sum of g^2 for |g| < 2^56
  float bhi = 0.f, blo = 0.f;  // sum of (g * 2^-96)^2 for the rest
  __device__ __forceinline__ void add(float g) {
    if (fabsf(g) < kNormMainLimit) {
      ff_add_sq(hi, lo, g);
    } else {
      ff_add_sq(bhi, blo, __fmul_rn(g, kNormBigScale));
    }
  }
  // true if any added g was NaN or infinite
  __device__ __forceinline__ bool nonfinite_seen() const {
    return !(fabsf(bhi) <= 3.4028234663852886e38f) || !(fabsf(blo) <= 3.4028234663852886e38f);
  }
  __device__ __forceinline__ void merge(float h2, float l2, float bh2, float bl2) {
    ff_merge(hi, lo, h2, l2);
    if (bh2 != 0.f || bl2 != 0.f || bhi != 0.f) ff_merge(bhi, blo, bh2, bl2);
  }
};

// Per-warp tile sums published to shared memory, double-buffered by tile
// parity so that one barrier per tile suffices.
constexpr int kMaxWarps = 16;
struct NormSlots {
  float hi[2][kMaxWarps], lo[2][kMaxWarps], bhi[2][kMaxWarps], blo[2][kMaxWarps];
};

// Fixed shuffle tree inside the warp, then lane 0 publishes the warp's sums.
__device__ __forceinline__ void tile_norm_publish(NormAcc acc, NormSlots& sl, int par, int warp,
                                                  int lane) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float h2 = __shfl_down_sync(0xFFFFFFFFu, acc.hi, off);
    float l2 = __shfl_down_sync(0xFFFFFFFFu, acc.lo, off);
    float bh2 = __shfl_down_sync(0xFFFFFFFFu, acc.bhi, off);
    float bl2 = __shfl_down_sync(0xFFFFFFFFu, acc.blo, off);
    if (lane < off) acc.merge(h2, l2, bh2, bl2);
  }
  if (lane == 0) {
    sl.hi[par][warp] = acc.hi;
    sl.lo[par][warp] = acc.lo;
    sl.bhi[par][warp] = acc.bhi;
    sl.blo[par][warp] = acc.blo;
  }
}

// After the barrier, run by all 32 lanes of one warp: lane l < n_warps
// takes warp l's sums, a fixed shuffle tree merges them (float-float, no
// fp64), lane 0 returns the tile's record (hi, lo, bhi, blo).
__device__ __forceinline__ float4 tile_norm_record(const NormSlots& sl, int par, int n_warps,
                                                   int lane) {
  NormAcc t;
  if (lane < n_warps) {
    t.hi = sl.hi[par][lane];
    t.lo = sl.lo[par][lane];
    t.bhi = sl.bhi[par][lane];
    t.blo = sl.blo[par][lane];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float h2 = __shfl_down_sync(0xFFFFFFFFu, t.hi, off);
    float l2 = __shfl_down_sync(0xFFFFFFFFu, t.lo, off);
    float bh2 = __shfl_down_sync(0xFFFFFFFFu, t.bhi, off);
    float bl2 = __shfl_down_sync(0xFFFFFFFFu, t.blo, off);
    if (lane < off) t.merge(h2, l2, bh2, bl2);
  }
  return make_float4(t.hi, t.lo, t.bhi, t.blo);
}

// Tile record from per-thread sums in shared memory (the bulk reduce pass):
// lane l merges the in-range sums of threads l, l + 32, ..., in that order,
// takes warp l's sums of big squares (lanes < n_warps), then the fixed
// shuffle tree merges the 32 lanes.
__device__ __forceinline__ float4 tile_norm_record_lanes(const float2* sums, const NormSlots& sl,
                                                         int par, int n_warps, int lane) {
  NormAcc t;
  for (int i = 0; i < n_warps; ++i) {
    const float2 x = sums[lane + 32 * i];
    ff_merge(t.hi, t.lo, x.x, x.y);
  }
  if (lane < n_warps) {
    t.bhi = sl.bhi[par][lane];
    t.blo = sl.blo[par][lane];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float h2 = __shfl_down_sync(0xFFFFFFFFu, t.hi, off);
    float l2 = __shfl_down_sync(0xFFFFFFFFu, t.lo, off);
    float bh2 = __shfl_down_sync(0xFFFFFFFFu, t.bhi, off);
    float bl2 = __shfl_down_sync(0xFFFFFFFFu, t.blo, off);
    if (lane < off) t.merge(h2, l2, bh2, bl2);
  }
  return make_float4(t.hi, t.lo, t.bhi, t.blo);
}

__device__ __forceinline__ void raise_flag(const Args& a, int32_t bucket) {
  atomicOr(&a.scaler->pending, 1u);
  if (a.flags) atomicOr(&a.flags[bucket], 1u);
}

__device__ __forceinline__ void set_error(zero_scaler* s, int code) {
  atomicCAS(&s->error, 0, code);
}

__device__ __forceinline__ int find_seg(const Args& a, int64_t g) {
  int lo = 0, hi = a.n_segs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a.segs[mid].tile_local0 <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Loss scale, skip and step-count bookkeeping at the end of a step
// ("Training models too big for one GPU: ZeRO & FSDP", "Mixed-precision
// training": pick the scale dynamically and skip a step on overflow).
// RN(x * y) in fp64, in integer arithmetic where f64emu covers it (the
// narrow fp64 pipe otherwise): the same bits either way.
__device__ __forceinline__ double dmul_exact(double x, double y) {
  uint64_t r;
  if (f64emu::mul(static_cast<uint64_t>(__double_as_longlong(x)),
                  static_cast<uint64_t>(__double_as_longlong(y)), &r))
    return __longlong_as_double(static_cast<long long>(r));
  return __dmul_rn(x, y);
}

// Adam's bias correction of step t + 1 from the stored power pw = beta^t:
// p = RN(pw beta) (the next stored power) and bc = RN32(RN(1 - p)).
__device__ __forceinline__ void bias_correction(double pw, double beta, double* p, float* bc) {
  const double q = dmul_exact(pw, beta);
  uint64_t d;
  uint32_t f;
  if (f64emu::one_minus(static_cast<uint64_t>(__double_as_longlong(q)), &d) &&
      f64emu::to_f32(d, &f)) {
    *bc = __uint_as_float(f);
  } else {
    *bc = __double2float_rn(__dsub_rn(1.0, q));
  }
  *p = q;
}

// fp32(1 / (S_l N k)) with the product and quotient in fp64. When S_l is a
// power of two and so is N k, the quotient is a power of two, exact in fp64
// and in fp32, formed from the exponents alone.
__device__ __forceinline__ float inverse_scale(float sl, int32_t n_ranks, int32_t n_micro) {
  const uint32_t sb = __float_as_uint(sl);
  const uint64_t nk = static_cast<uint64_t>(n_ranks) * static_cast<uint64_t>(n_micro);
  const int es = static_cast<int>((sb >> 23) & 0xFFu);
  if ((sb & 0x807FFFFFu) == 0 && es != 0 && es != 255 && nk != 0 && (nk & (nk - 1)) == 0) {
    const int e = es - 127 + (63 - __clzll(static_cast<long long>(nk)));
    if (e >= -126 && e <= 126) return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  }
  const double denom = __dmul_rn(__dmul_rn(static_cast<double>(sl), static_cast<double>(n_ranks)),
                                 static_cast<double>(n_micro));
  return __double2float_rn(__ddiv_rn(1.0, denom));
}

// The scaler fields the bookkeeping reads, taken before it writes any.
struct ScalerSnap {
  double p1, p2;  // beta1_pow * beta1, beta2_pow * beta2: the powers after a good step
  float scale;
  int32_t good_steps, t, n_skipped, state_index;
  uint32_t pending;
};

// The bookkeeping's stores, from a snapshot and the step's overflow vote.
__device__ __forceinline__ void bookkeeping_store(zero_scaler* sc, const ScalerSnap& q, bool ov,
                                                  int dynamic, int growth_interval,
                                                  int flip_sets) {
  sc->pending = 0;
  sc->overflow = ov ? 1u : 0u;
  if (ov) {
    if (dynamic) {
      const float half = __fmul_rn(q.scale, 0.5f);
      sc->scale = half < 1.0f ? 1.0f : half;
    }
    sc->good_steps = 0;
    sc->n_skipped = q.n_skipped + 1;
    return;
  }
  sc->t = q.t + 1;
  sc->beta1_pow = q.p1;
  sc->beta2_pow = q.p2;
  int good = q.good_steps + 1;
  if (dynamic && good >= growth_interval) {
    sc->scale = __fmul_rn(q.scale, 2.0f);
    good = 0;
  }
  sc->good_steps = good;
  if (flip_sets) sc->state_index = q.state_index ^ 1;
}

__device__ void step_bookkeeping(zero_scaler* sc, double beta1, double beta2, int dynamic,
                                 int growth_interval, int flip_sets) {
  ScalerSnap q;
  q.pending = sc->pending;
  q.scale = sc->scale;
  q.good_steps = sc->good_steps;
  q.t = sc->t;
  q.n_skipped = sc->n_skipped;
  q.state_index = sc->state_index;
  q.p1 = dmul_exact(sc->beta1_pow, beta1);
  q.p2 = dmul_exact(sc->beta2_pow, beta2);
  bookkeeping_store(sc, q, q.pending != 0, dynamic, growth_interval, flip_sets);
}

// -------------------------------------------------------------- prologue --

template <int MODE>
__device__ void compute_step_scalars(const Args& a, StepScalars* out) {
  zero_scaler* sc = a.scaler;
  StepScalars s;
  s.skip = 0;
  s.clip = 1.0f;
  s.inv = 1.0f;
  s.bc1 = s.bc2 = 1.0f;
  s.src = 0;
  s.dst = 0;
  if (MODE == kFused || MODE == kReduce) {
    // average over the N ranks and the k micro-batches of each, after the loss scale
    s.inv = inverse_scale(sc->scale, a.n_ranks, a.n_micro);
  }
  if (MODE == kFused || MODE == kUpdate) {
    double p1, p2;  // the next powers: only the bookkeeping stores them
    bias_correction(sc->beta1_pow, a.beta1, &p1, &s.bc1);
    bias_correction(sc->beta2_pow, a.beta2, &p2, &s.bc2);
    (void)p1;
    (void)p2;
    const int idx = sc->state_index;
    if (idx < 0 || idx >= a.n_sets || (MODE == kFused && a.n_sets != 2)) {
      set_error(sc, ZERO_DEVERR_STATE_INDEX);
      s.skip = 1;
    }
    s.src = idx;
    // the fused pass, and the update pass when the caller gives two sets,
    // write the other set (ping-pong); the finish then flips the index
    s.dst = (MODE == kFused || (MODE == kUpdate && a.n_sets == 2)) ? (idx ^ 1) : idx;
  }
  if (MODE == kUpdate) {
    if (sc->pending) s.skip = 1;  // the step is skipped: write nothing
    if (!s.skip && (a.mode_flags & kFlagClip)) {
      if (sc->norm_step != sc->t + 1) {
        set_error(sc, ZERO_DEVERR_NO_NORM);
        s.skip = 1;
      } else if (sc->clip_apply) {
        s.clip = sc->clip_coef;
      }
    }
  }
  if (MODE == kCast) {
    // without these flags the scaler is not read (it may be NULL)
    if (a.mode_flags & kFlagIfPending) s.skip = sc->pending ? 0 : 1;
    if (a.mode_flags & kFlagUseScalerSet) {
      const int idx = sc->state_index;
      if (idx < 0 || idx >= a.n_sets) {
        set_error(sc, ZERO_DEVERR_STATE_INDEX);
        s.skip = 1;
      }
      s.src = idx;
    }
  }
  *out = s;
}

// ------------------------------------------------------------- the body --

// Per-element work of step_kernel on a vector of 8 elements starting at flat
// index j: kNorm adds the squares of 8 reduced gradients to the tile's
// record, kCast writes 8 parameters from the master set.
template <int MODE, bool kBf16>
__device__ __forceinline__ void do_vector(const Args& a, const StepScalars& s, int64_t j,
                                          int32_t rank, NormAcc& nacc) {
  static_assert(MODE == kNorm || MODE == kCast, "step_kernel modes only");
  const int64_t w = j - a.wbase;                    // window index
  const int64_t k = j - static_cast<int64_t>(rank) * a.shard;  // shard index
  if (!ZCHECK(w >= 0 && w + 8 <= a.wend && k >= 0 && k + 8 <= a.shard, kSiteVector, j)) return;
  float x[8];
  if constexpr (MODE == kNorm) {
    load8f(a.ghat[rank] + k, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) nacc.add(x[e]);
  } else {
    load8f(a.master[s.src][rank] + k, x);
    __stcs(reinterpret_cast<uint4*>(a.flat + w), narrow8<kBf16>(x));
  }
}

// Scalar version for one element (segment heads/tails, misaligned segments).
template <int MODE, bool kBf16>
__device__ __forceinline__ void do_scalar(const Args& a, const StepScalars& s, int64_t j,
                                          int32_t rank, int first_rep, NormAcc& nacc,
                                          bool& bad) {
  const int64_t w = j - a.wbase;
  const int64_t k = j - static_cast<int64_t>(rank) * a.shard;
  if (!ZCHECK(w >= 0 && w < a.wend && k >= 0 && k < a.shard, kSiteScalar, j)) return;
  float g = 0.f, th = 0.f, m = 0.f, v = 0.f;
  if constexpr (MODE == kFused || MODE == kUpdate) {
    th = a.master[s.src][rank][k];
    m = a.mom[s.src][rank][k];
    v = a.var[s.src][rank][k];
  }
  if constexpr (MODE == kFused || MODE == kReduce) {
    const int N = a.n_ranks;
    float acc = 0.f;
    for (int p = 0; p < N; ++p) {
      int rr = first_rep + p;
      if (rr >= N) rr -= N;
      float x = widen<kBf16>(a.rep[rr][w]);
      if (a.has_acc) x = __fadd_rn(a.acc[rr][w], x);  // accumulated replica value
      acc = p == 0 ? x : __fadd_rn(acc, x);
    }
    g = __fmul_rn(acc, s.inv);
    bad |= nonfinite(g);
  }
  if constexpr (MODE == kUpdate || MODE == kNorm) g = a.ghat[rank][k];
  if constexpr (MODE == kReduce) {
    a.ghat[rank][k] = g;
    if (a.mode_flags & kFlagPartials) nacc.add(g);
  }
  if constexpr (MODE == kNorm) nacc.add(g);
  if constexpr (MODE == kFused || MODE == kUpdate) {
    if (MODE == kUpdate && s.clip != 1.0f) g = __fmul_rn(g, s.clip);
    adamw(th, m, v, g, a, s);
    a.master[s.dst][rank][k] = th;
    a.mom[s.dst][rank][k] = m;
    a.var[s.dst][rank][k] = v;
    a.flat[w] = narrow<kBf16>(th);
  }
  if constexpr (MODE == kCast) {
    th = a.master[s.src][rank][k];
    a.flat[w] = narrow<kBf16>(th);
  }
}

// One edge element of a tile by a whole warp (kFused / kReduce): lane p
// loads the replica values at ring positions p and p + 32, so all N loads
// are in flight together, and every lane adds them in ring order through
// shuffles (the same operations in the same order as do_scalar); lane 0
// then finishes the element. Used when a tile has only a few elements
// outside its aligned body: the per-thread path would chain N dependent
// global loads on one thread and hold up the whole tile.
template <int MODE, bool kBf16>
__device__ __forceinline__ void do_scalar_warp(const Args& a, const StepScalars& s, int64_t j,
                                               int32_t rank, int first_rep, NormAcc& nacc,
                                               bool& bad, int lane) {
  static_assert(MODE == kFused || MODE == kReduce, "replica modes only");
  const int64_t w = j - a.wbase;
  const int64_t k = j - static_cast<int64_t>(rank) * a.shard;
  if (!ZCHECK(w >= 0 && w < a.wend && k >= 0 && k < a.shard, kSiteScalar, j)) return;
  const int N = a.n_ranks;
  float x0 = 0.f, x1 = 0.f;
  if (lane < N) {
    int rr = first_rep + lane;
    if (rr >= N) rr -= N;
    x0 = widen<kBf16>(a.rep[rr][w]);
    if (a.has_acc) x0 = __fadd_rn(a.acc[rr][w], x0);
  }
  if (lane + 32 < N) {
    int rr = first_rep + lane + 32;
    if (rr >= N) rr -= N;
    x1 = widen<kBf16>(a.rep[rr][w]);
    if (a.has_acc) x1 = __fadd_rn(a.acc[rr][w], x1);
  }
  float acc = 0.f;
  for (int p = 0; p < N; ++p) {
    const float x = __shfl_sync(0xFFFFFFFFu, p < 32 ? x0 : x1, p & 31);
    acc = p == 0 ? x : __fadd_rn(acc, x);
  }
  if (lane != 0) return;
  const float g = __fmul_rn(acc, s.inv);
  bad |= nonfinite(g);
  if constexpr (MODE == kReduce) {
    a.ghat[rank][k] = g;
    if (a.mode_flags & kFlagPartials) nacc.add(g);
  } else {
    float th = a.master[s.src][rank][k];
    float m = a.mom[s.src][rank][k];
    float v = a.var[s.src][rank][k];
    adamw(th, m, v, g, a, s);
    a.master[s.dst][rank][k] = th;
    a.mom[s.dst][rank][k] = m;
    a.var[s.dst][rank][k] = v;
    a.flat[w] = narrow<kBf16>(th);
  }
}

// The light modes (kNorm, kCast) as a plain tile-scheduled kernel: 16-byte
// vectors of 8 elements where an owner's slice sits on the windows'
// 8-element grid and its shard on the 4-element grid, single elements
// elsewhere (coalesced over the CTA's threads).
template <int MODE, bool kBf16>
__global__ void __launch_bounds__(kThreads, 2) step_kernel(const __grid_constant__ Args a) {
  static_assert(MODE == kNorm || MODE == kCast, "the streaming modes run in bulk_kernel");
  __shared__ StepScalars sh_s;
  __shared__ NormSlots sh_norm;
  pdl_begin();
  if (threadIdx.x == 0) compute_step_scalars<MODE>(a, &sh_s);
  __syncthreads();
  const StepScalars s = sh_s;
  if (s.skip) {
    // no overflow: nothing to re-cast; the step's bookkeeping, once
    if (MODE == kCast && (a.mode_flags & kFlagFinish) && blockIdx.x == 0 && threadIdx.x == 0)
      step_bookkeeping(a.scaler, a.beta1, a.beta2, a.bk_dynamic, a.bk_growth, a.bk_flip);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint32_t tile_no = 0;  // tiles done by this CTA

  for (int64_t g = blockIdx.x; g < a.n_tiles; g += gridDim.x, ++tile_no) {
    const Seg& sg = a.segs[find_seg(a, g)];
    const int64_t lo = sg.lo + (g - sg.tile_local0) * kTile;
    const int64_t hi = min(lo + kTile, sg.hi);
    const int32_t rank = sg.rank;
    NormAcc nacc;
    bool unused = false;

    // vector body [va, vb): 8-element aligned in the windows and 4-element
    // aligned in the shards; otherwise every element takes the single path
    const int64_t rank0 = static_cast<int64_t>(rank) * a.shard;
    const bool vec_ok = (((rank0 - a.wbase) & 3) == 0);
    int64_t va = hi, vb = hi;
    if (vec_ok) {
      va = lo + ((a.wbase - lo) & 7);   // first j >= lo with (j - wbase) % 8 == 0
      if (va > hi) va = hi;
      vb = va + ((hi - va) & ~static_cast<int64_t>(7));
    }
    const int nvec = static_cast<int>((vb - va) >> 3);
    for (int q = threadIdx.x; q < nvec; q += kThreads)
      do_vector<MODE, kBf16>(a, s, va + static_cast<int64_t>(q) * kVec, rank, nacc);
    // head [lo, va) and tail [vb, hi)
    const int nhead = static_cast<int>(va - lo);
    const int ntail = static_cast<int>(hi - vb);
    for (int q = threadIdx.x; q < nhead + ntail; q += kThreads) {
      const int64_t j = q < nhead ? lo + q : vb + (q - nhead);
      do_scalar<MODE, kBf16>(a, s, j, rank, 0, nacc, unused);
    }

    if constexpr (MODE == kNorm) {
      // publish, one barrier, and the tile's record formed by warp
      // (tile_no mod 8), so that the merge rotates over the warps
      const int par = tile_no & 1;
      tile_norm_publish(nacc, sh_norm, par, warp, lane);
      __syncthreads();
      if (warp == static_cast<int>(tile_no % kWarps)) {
        const float4 rec = tile_norm_record(sh_norm, par, kWarps, lane);
        const int64_t r = sg.tile_global0 + (g - sg.tile_local0);
        if (lane == 0 && ZCHECK(r >= 0 && r < a.n_records, kSiteRecord, r)) a.partials[r] = rec;
      }
    }
  }
  if constexpr (MODE == kCast) {
    if (a.mode_flags & kFlagFinish) {
      // overflow path: the last CTA to finish its re-cast does the bookkeeping
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(&a.scaler->finish_count, 1u);
        if (done == gridDim.x - 1) {
          __threadfence();
          step_bookkeeping(a.scaler, a.beta1, a.beta2, a.bk_dynamic, a.bk_growth, a.bk_flip);
          a.scaler->finish_count = 0;
        }
      }
    }
  }
}

// -------------------------------------------------- bulk-copy pipeline --
//
// kFused, kReduce and kUpdate stream their inputs through shared memory.
// Work is cut into element ranges of E = 512 * EPT elements (EPT = 8, one
// 4096-element tile, when a range's whole input fits one 64 KB stage; else
// EPT = 4). The inputs of one range are chunks: one per replica (ring order,
// 2E bytes) and the state block (master, m, v; for kUpdate also g; 4E bytes
// each). The host packs the chunks of a range into at most 64 KB stages
// (StagePlan): N = 8 fused is one 56 KB stage, N = 64 fused is four stages
// of 16 replicas and one state stage. One producer warp posts each stage's
// byte count on the slot's "full" mbarrier and its 32 lanes issue the
// stage's cp.async.bulk copies in parallel; sixteen consumer warps wait on
// "full", accumulate the replicas of the stage in registers (thread t owns
// elements [EPT*t, EPT*t+EPT) of the range, held across the range's
// stages), finish the step when the state block arrives, write results to
// global memory with streaming stores and release the slot on its "empty"
// mbarrier. With S slots, S - 1 stages (~100-170 KB per SM) are in flight
// while one is computed, independent of the register budget.
// An owner whose slice starts off the windows' 8-element grid gets a
// shard-indexed body: its chunks are copied from the 16-byte block below
// their first element (16 bytes longer) and the values picked out in shared
// memory (tile_geom). The few elements of a tile outside its body (at a
// bucket boundary or an owner's last tile) are done by the consumers with
// plain loads, one warp per element (do_scalar_warp) or one thread each.
// Every mbarrier wait is bounded by kWaitLimitNs of %globaltimer; on expiry
// the thread records ZERO_DEVERR_TIMEOUT, the CTA stops issuing, the
// producer waits (again bounded) for the copies it issued, and all return.

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kBulkThreads = kConsumers + 32;
constexpr int kMaxStages = 6;
constexpr int kStageBudget = 64 * 1024;         // bytes per stage, upper bound
constexpr int kSmemCap = 216 * 1024;            // dynamic shared memory per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static_assert(kTile % (kConsumers * 8) == 0, "tile must hold whole ranges");
static_assert(kConsumerWarps <= kMaxWarps, "norm slots");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// true when the phase of the given parity has completed; false after the limit
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// global -> shared bulk copy completing on `bar`; addresses 16-byte aligned,
// bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

struct TileGeom {
  int64_t lo, hi, va, vb, partial;
  int32_t rank, bucket, first_rep;
  int32_t shift;  // window elements from the 16-byte block below va to va (shard-indexed bodies)
};

// a0 += low half of w, a1 += high half of w, each 16-bit value widened
// exactly to fp32 and the sum rounded once to nearest even: sm_100+'s
// mixed-precision add (PTX add.rn.f32.f16 / add.rn.f32.bf16) does the
// widening inside the add, one instruction per element and replica.
template <bool kBf16>
__device__ __forceinline__ void add_halves(float& a0, float& a1, uint32_t w) {
  if constexpr (kBf16) {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
        " add.rn.f32.bf16 %0, l, %0;\n add.rn.f32.bf16 %1, h, %1;\n}"
        : "+f"(a0), "+f"(a1)
        : "r"(w));
  } else {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
        " add.rn.f32.f16 %0, l, %0;\n add.rn.f32.f16 %1, h, %1;\n}"
        : "+f"(a0), "+f"(a1)
        : "r"(w));
  }
}

// EPT consecutive 16-bit values (one 8- or 16-byte shared-memory load).
template <int EPT>
struct HalfVec;
template <>
struct HalfVec<4> {
  uint2 v;
  __device__ __forceinline__ void load(const unsigned char* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ uint32_t word(int i) const { return i == 0 ? v.x : v.y; }
};
template <>
struct HalfVec<8> {
  uint4 v;
  __device__ __forceinline__ void load(const unsigned char* p) { v = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ uint32_t word(int i) const {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  }
};

// d0 = a0 + low half of w, d1 = a1 + high half of w (same mixed-precision add)
template <bool kBf16>
__device__ __forceinline__ void add_halves_to(float& d0, float& d1, uint32_t w, float a0,
                                              float a1) {
  if constexpr (kBf16) {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
        " add.rn.f32.bf16 %0, l, %3;\n add.rn.f32.bf16 %1, h, %4;\n}"
        : "=f"(d0), "=f"(d1)
        : "r"(w), "f"(a0), "f"(a1));
  } else {
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
        " add.rn.f32.f16 %0, l, %3;\n add.rn.f32.f16 %1, h, %4;\n}"
        : "=f"(d0), "=f"(d1)
        : "r"(w), "f"(a0), "f"(a1));
  }
}

// With fp32 accumulators of earlier micro-batches: replica value
// A = acc + widen(micro) (one rounding), then the ring sum sum += A.
// micro chunks are mstride bytes apart, accumulator chunks astride.
template <bool kBf16, int EPT>
__device__ __forceinline__ void acc_stage_accum(const unsigned char* mp, const unsigned char* ap,
                                                int mstride, int astride, int n,
                                                float (&sum)[EPT]) {
#pragma unroll 2
  for (int p = 0; p < n; ++p) {
    HalfVec<EPT> w;
    w.load(mp + static_cast<size_t>(p) * mstride);
    float av[EPT];
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i) {
      const float4 q = reinterpret_cast<const float4*>(ap + static_cast<size_t>(p) * astride)[i];
      av[4 * i] = q.x;
      av[4 * i + 1] = q.y;
      av[4 * i + 2] = q.z;
      av[4 * i + 3] = q.w;
    }
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) {
      float v0, v1;
      add_halves_to<kBf16>(v0, v1, w.word(i), av[2 * i], av[2 * i + 1]);
      sum[2 * i] = __fadd_rn(sum[2 * i], v0);
      sum[2 * i + 1] = __fadd_rn(sum[2 * i + 1], v1);
    }
  }
}

// acc[e] += replica chunks 0..R-1 of this thread's EPT elements, in ring
// order; all R shared-memory loads are issued before the adds. `stride` is
// the chunk size in bytes.
template <bool kBf16, int R, int EPT>
__device__ __forceinline__ void acc_reps(const unsigned char* rp, int stride, float (&acc)[EPT]) {
  HalfVec<EPT> w[R];
#pragma unroll
  for (int p = 0; p < R; ++p) w[p].load(rp + static_cast<size_t>(p) * stride);
#pragma unroll
  for (int p = 0; p < R; ++p) {
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) add_halves<kBf16>(acc[2 * i], acc[2 * i + 1], w[p].word(i));
  }
}

template <bool kBf16, int EPT>
__device__ __forceinline__ void acc_stage(const unsigned char* rp, int stride, int n,
                                          float (&acc)[EPT]) {
  switch (n) {
    case 1: acc_reps<kBf16, 1, EPT>(rp, stride, acc); break;
    case 2: acc_reps<kBf16, 2, EPT>(rp, stride, acc); break;
    case 3: acc_reps<kBf16, 3, EPT>(rp, stride, acc); break;
    case 4: acc_reps<kBf16, 4, EPT>(rp, stride, acc); break;
    case 5: acc_reps<kBf16, 5, EPT>(rp, stride, acc); break;
    case 6: acc_reps<kBf16, 6, EPT>(rp, stride, acc); break;
    case 7: acc_reps<kBf16, 7, EPT>(rp, stride, acc); break;
    case 8: acc_reps<kBf16, 8, EPT>(rp, stride, acc); break;
    case 9: acc_reps<kBf16, 9, EPT>(rp, stride, acc); break;
    case 10: acc_reps<kBf16, 10, EPT>(rp, stride, acc); break;
    case 11: acc_reps<kBf16, 11, EPT>(rp, stride, acc); break;
    case 12: acc_reps<kBf16, 12, EPT>(rp, stride, acc); break;
    case 13: acc_reps<kBf16, 13, EPT>(rp, stride, acc); break;
    case 14: acc_reps<kBf16, 14, EPT>(rp, stride, acc); break;
    case 15: acc_reps<kBf16, 15, EPT>(rp, stride, acc); break;
    case 16: acc_reps<kBf16, 16, EPT>(rp, stride, acc); break;
    default:  // the stage plan never puts more than 16 replicas in a stage
      for (int p = 0; p < n; ++p)
        acc_reps<kBf16, 1, EPT>(rp + static_cast<size_t>(p) * stride, stride, acc);
  }
}

template <int EPT>
__device__ __forceinline__ void lds_fv(const unsigned char* p, float (&x)[EPT]) {
#pragma unroll
  for (int i = 0; i < EPT / 4; ++i) {
    const float4 a = reinterpret_cast<const float4*>(p)[i];
    x[4 * i] = a.x;
    x[4 * i + 1] = a.y;
    x[4 * i + 2] = a.z;
    x[4 * i + 3] = a.w;
  }
}

template <int EPT>
__device__ __forceinline__ void stg_fv(float* p, const float (&x)[EPT]) {
#pragma unroll
  for (int i = 0; i < EPT / 4; ++i)
    __stcs(reinterpret_cast<float4*>(p) + i,
           make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]));
}

template <bool kBf16, int EPT>
__device__ __forceinline__ void stg_hv(uint16_t* p, const float (&x)[EPT]) {
  uint32_t u[EPT / 2];
#pragma unroll
  for (int i = 0; i < EPT / 2; ++i)
    u[i] = static_cast<uint32_t>(narrow<kBf16>(x[2 * i])) |
           (static_cast<uint32_t>(narrow<kBf16>(x[2 * i + 1])) << 16);
  if constexpr (EPT == 4) {
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(u[0], u[1]));
  } else {
    __stcs(reinterpret_cast<uint4*>(p), make_uint4(u[0], u[1], u[2], u[3]));
  }
}

// Shifted replica values. A thread's EPT values start `shift` elements
// (0 < shift < 8) past its position p in a replica chunk. For EPT = 4 (p
// 8-byte aligned) they lie in the 16 bytes from the 8-byte block that holds
// the first of them: two aligned 8-byte loads, then a word select and, for
// an odd shift, a funnel shift. For EPT = 8 (p 16-byte aligned) they lie in
// the 32 bytes from p: two 16-byte loads, a two-step word select and the
// funnel shift. The chunk holds 16 bytes past its last thread's position.
template <int EPT>
struct ShiftedVec;
template <>
struct ShiftedVec<4> {
  uint2 a, c;
  __device__ __forceinline__ void load(const unsigned char* p, int shift) {
    const unsigned char* b = p + ((shift >> 2) << 3);
    a = *reinterpret_cast<const uint2*>(b);
    c = *reinterpret_cast<const uint2*>(b + 8);
  }
  // the EPT / 2 words of values, low element in the low half
  __device__ __forceinline__ void words(int shift, uint32_t (&x)[2]) const {
    const int s = shift & 3;  // elements past the first loaded block
    const uint32_t w0 = (s & 2) ? a.y : a.x;
    const uint32_t w1 = (s & 2) ? c.x : a.y;
    const uint32_t w2 = (s & 2) ? c.y : c.x;
    x[0] = (s & 1) ? __funnelshift_r(w0, w1, 16) : w0;
    x[1] = (s & 1) ? __funnelshift_r(w1, w2, 16) : w1;
  }
};
template <>
struct ShiftedVec<8> {
  uint4 a, b;
  __device__ __forceinline__ void load(const unsigned char* p, int) {
    a = *reinterpret_cast<const uint4*>(p);
    b = *reinterpret_cast<const uint4*>(p + 16);
  }
  __device__ __forceinline__ void words(int shift, uint32_t (&x)[4]) const {
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const int q = shift >> 1;
    uint32_t t[6], u[5];
#pragma unroll
    for (int j = 0; j < 6; ++j) t[j] = (q & 2) ? wd[j + 2] : wd[j];
#pragma unroll
    for (int j = 0; j < 5; ++j) u[j] = (q & 1) ? t[j + 1] : t[j];  // u[j] = wd[q + j]
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = (shift & 1) ? __funnelshift_r(u[j], u[j + 1], 16) : u[j];
  }
};

// acc[e] += replica chunks 0..R-1 of a shifted body, loads first.
template <bool kBf16, int R, int EPT>
__device__ __forceinline__ void acc_reps_shifted(const unsigned char* rp, int stride, int shift,
                                                 float (&acc)[EPT]) {
  ShiftedVec<EPT> w[R];
#pragma unroll
  for (int p = 0; p < R; ++p) w[p].load(rp + static_cast<size_t>(p) * stride, shift);
#pragma unroll
  for (int p = 0; p < R; ++p) {
    uint32_t x[EPT / 2];
    w[p].words(shift, x);
#pragma unroll
    for (int i = 0; i < EPT / 2; ++i) add_halves<kBf16>(acc[2 * i], acc[2 * i + 1], x[i]);
  }
}

// acc[e] += replica chunks 0..n-1 of this thread's EPT elements, in ring
// order, for a shifted body: groups of G chunks (32 loaded words), each
// group loaded before it is added. The same additions in the same order as
// acc_stage.
template <bool kBf16, int EPT>
__device__ __forceinline__ void acc_stage_shifted(const unsigned char* rp, int stride, int n,
                                                  int shift, float (&acc)[EPT]) {
  constexpr int G = EPT == 4 ? 8 : 4;
  int p = 0;
  for (; p + G <= n; p += G)
    acc_reps_shifted<kBf16, G, EPT>(rp + static_cast<size_t>(p) * stride, stride, shift, acc);
  rp += static_cast<size_t>(p) * stride;
  switch (n - p) {
    case 1: acc_reps_shifted<kBf16, 1, EPT>(rp, stride, shift, acc); break;
    case 2: acc_reps_shifted<kBf16, 2, EPT>(rp, stride, shift, acc); break;
    case 3: acc_reps_shifted<kBf16, 3, EPT>(rp, stride, shift, acc); break;
    case 4: if constexpr (G > 4) acc_reps_shifted<kBf16, 4, EPT>(rp, stride, shift, acc); break;
    case 5: if constexpr (G > 5) acc_reps_shifted<kBf16, 5, EPT>(rp, stride, shift, acc); break;
    case 6: if constexpr (G > 6) acc_reps_shifted<kBf16, 6, EPT>(rp, stride, shift, acc); break;
    case 7: if constexpr (G > 7) acc_reps_shifted<kBf16, 7, EPT>(rp, stride, shift, acc); break;
    default: break;
  }
}

// acc_stage_accum for a shifted body (4 elements per thread): the micro
// values start `shift` elements past mp in each micro chunk, the
// accumulator values (shift & 3) floats past ap (16-byte aligned; 32 bytes
// readable) in each accumulator chunk. The same operations in the same
// order as acc_stage_accum.
template <bool kBf16>
__device__ __forceinline__ void acc_stage_accum_shifted(const unsigned char* mp,
                                                        const unsigned char* ap, int mstride,
                                                        int astride, int n, int shift,
                                                        float (&sum)[4]) {
  const int sa = shift & 3;
#pragma unroll 2
  for (int p = 0; p < n; ++p) {
    ShiftedVec<4> w;
    w.load(mp + static_cast<size_t>(p) * mstride, shift);
    uint32_t x[2];
    w.words(shift, x);
    const float4* q = reinterpret_cast<const float4*>(ap + static_cast<size_t>(p) * astride);
    const float4 f0 = q[0], f1 = q[1];
    const float fd[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    float t[6], av[4];
#pragma unroll
    for (int j = 0; j < 6; ++j) t[j] = (sa & 2) ? fd[j + 2] : fd[j];
#pragma unroll
    for (int j = 0; j < 4; ++j) av[j] = (sa & 1) ? t[j + 1] : t[j];  // av[j] = fd[sa + j]
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float v0, v1;
      add_halves_to<kBf16>(v0, v1, x[i], av[2 * i], av[2 * i + 1]);
      sum[2 * i] = __fadd_rn(sum[2 * i], v0);
      sum[2 * i + 1] = __fadd_rn(sum[2 * i + 1], v1);
    }
  }
}

// 16-bit parameter stores of a shifted body: one 8-byte store when p is
// 8-byte aligned, two 4-byte stores when it is 4-byte aligned, four 2-byte
// stores otherwise.
template <bool kBf16>
__device__ __forceinline__ void stg_hv_unaligned(uint16_t* p, const float (&x)[4]) {
  const unsigned int h0 = narrow<kBf16>(x[0]), h1 = narrow<kBf16>(x[1]);
  const unsigned int h2 = narrow<kBf16>(x[2]), h3 = narrow<kBf16>(x[3]);
  if ((reinterpret_cast<uintptr_t>(p) & 7) == 0) {
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(h0 | (h1 << 16), h2 | (h3 << 16)));
  } else if ((reinterpret_cast<uintptr_t>(p) & 3) == 0) {
    unsigned int* q = reinterpret_cast<unsigned int*>(p);
    __stcs(q, h0 | (h1 << 16));
    __stcs(q + 1, h2 | (h3 << 16));
  } else {
    unsigned short* q = reinterpret_cast<unsigned short*>(p);
    __stcs(q, static_cast<unsigned short>(h0));
    __stcs(q + 1, static_cast<unsigned short>(h1));
    __stcs(q + 2, static_cast<unsigned short>(h2));
    __stcs(q + 3, static_cast<unsigned short>(h3));
  }
}

// Tile g of this launch: element range, owner, and the aligned body
// [va, vb). When the owner's shard starts on the windows' 8-element grid
// the body starts where the window index is a multiple of 8 (16-byte
// replica chunks, 16-byte state chunks). Otherwise it starts where the
// shard index is a multiple of 4 (16-byte state chunks), `shift` elements
// past a 16-byte block of the windows: replica and accumulator chunks are
// copied from that block and parameter stores are unaligned. Either way a
// whole tile has no elements outside its body; a tile that starts at a
// bucket boundary or ends an owner's slice has a few. A kernel built
// without off-grid support (`off` false; the host launches it only when
// every owner is on the grid) would take such tiles element by element.
// (A forward scan from the previous tile's segment measured slower than this
// binary search.)
__device__ __forceinline__ TileGeom tile_geom(const Args& a, int64_t g, bool off) {
  const Seg& sg = a.segs[find_seg(a, g)];
  TileGeom t;
  t.lo = sg.lo + (g - sg.tile_local0) * kTile;
  t.hi = min(t.lo + kTile, sg.hi);
  t.rank = sg.rank;
  t.bucket = sg.bucket;
  t.partial = sg.tile_global0 + (g - sg.tile_local0);
  t.first_rep = sg.rank + 1 == a.n_ranks ? 0 : sg.rank + 1;
  const int64_t rank0 = static_cast<int64_t>(sg.rank) * a.shard;
  t.shift = 0;
  if (((rank0 - a.wbase) & 7) == 0) {
    t.va = min(t.lo + ((a.wbase - t.lo) & 7), t.hi);
  } else if (off) {
    t.va = min(t.lo + ((rank0 - t.lo) & 3), t.hi);
    t.shift = static_cast<int32_t>((t.va - a.wbase) & 7);
  } else {
    t.va = t.hi;
  }
  t.vb = t.va + ((t.hi - t.va) & ~static_cast<int64_t>(7));
  return t;
}

// The step's finish folded into a single-launch fused pass (kFlagFinish):
// run by the 512 consumer threads after their last tile. Every CTA counts
// itself done (after its stores, made visible); the last one to finish does
// the bookkeeping. When the step overflowed it first re-casts the whole
// launch's parameters from the kept state set, alone: slow (one SM), but an
// overflow is rare and the host folds only windows of at most
// kFoldMaxElems elements. No CTA waits for another.
template <bool kBf16>
__device__ void fused_finish(const Args& a, const StepScalars& s) {
  __shared__ int sh_last;
  consumer_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(&a.scaler->finish_count, 1u);
    sh_last = done == gridDim.x - 1;
    if (sh_last) __threadfence();
  }
  consumer_sync();
  if (!sh_last) return;
  if (*reinterpret_cast<volatile uint32_t*>(&a.scaler->pending)) {
    // the re-cast of every tile of the launch, as step_kernel<kCast> does it:
    // 16-byte vectors where the owner sits on the grid, single elements at
    // the edges
    NormAcc unused_acc;
    bool unused = false;
    for (int64_t g = 0; g < a.n_tiles; ++g) {
      const Seg& sg = a.segs[find_seg(a, g)];
      const int64_t lo = sg.lo + (g - sg.tile_local0) * kTile;
      const int64_t hi = min(lo + kTile, sg.hi);
      const int64_t rank0 = static_cast<int64_t>(sg.rank) * a.shard;
      int64_t va = hi, vb = hi;
      if (((rank0 - a.wbase) & 3) == 0) {
        va = min(lo + ((a.wbase - lo) & 7), hi);
        vb = va + ((hi - va) & ~static_cast<int64_t>(7));
      }
      const int nvec = static_cast<int>((vb - va) >> 3);
      for (int q = threadIdx.x; q < nvec; q += kConsumers)
        do_vector<kCast, kBf16>(a, s, va + static_cast<int64_t>(q) * kVec, sg.rank, unused_acc);
      const int nhead = static_cast<int>(va - lo), ntail = static_cast<int>(hi - vb);
      for (int q = threadIdx.x; q < nhead + ntail; q += kConsumers)
        do_scalar<kCast, kBf16>(a, s, q < nhead ? lo + q : vb + (q - nhead), sg.rank, 0,
                                unused_acc, unused);
    }
    consumer_sync();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    step_bookkeeping(a.scaler, a.beta1, a.beta2, a.bk_dynamic, a.bk_growth, a.bk_flip);
    a.scaler->finish_count = 0;
  }
}

template <int MODE, bool kBf16, int EPT, bool kAcc, bool kOff>
__global__ void __launch_bounds__(kBulkThreads, 1) bulk_kernel(const __grid_constant__ Args a,
                                                               int n_slots,
                                                               uint32_t slot_bytes) {
  constexpr int E = kConsumers * EPT;  // elements per range
  // 8 elements per thread only in the reduce pass: the fused and update
  // passes store their 16-bit parameters 4 elements at a time
  static_assert(MODE == kReduce || EPT == 4, "8 elements per thread: reduce pass only");
  // shifted bodies (owner shard off the windows' 8-element grid): each
  // replica chunk holds up to 7 extra elements and each accumulator chunk up
  // to 3, so chunks are 16 bytes longer. The update pass bulk-copies only
  // shard-indexed arrays (g, master, m, v); only its parameter stores see
  // the window's phase.
  constexpr bool kShift = kOff && (MODE == kFused || MODE == kReduce);
  constexpr int kPad = kShift ? 16 : 0;  // extra bytes per chunk of a shifted tile
  __shared__ StepScalars sh_s;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ NormSlots sh_norm;
  // reduce pass: every consumer thread's in-range tile sums (hi, lo), by
  // tile parity (8 KB)
  __shared__ float2 sh_sums[MODE == kReduce ? 2 : 1][MODE == kReduce ? kConsumers : 1];
  __shared__ int sh_abort;
  extern __shared__ __align__(128) unsigned char stage_mem[];

  pdl_begin();
  if (threadIdx.x == 0) {
    compute_step_scalars<MODE>(a, &sh_s);
    for (int i = 0; i < n_slots; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    sh_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const StepScalars s = sh_s;
  if (s.skip) {
    // a folded finish still runs once (the state index was invalid: the
    // error is recorded, the bookkeeping follows as it would in the finish)
    if constexpr (MODE == kFused) {
      if ((a.mode_flags & kFlagFinish) && threadIdx.x == 0) {
        const uint32_t done = atomicAdd(&a.scaler->finish_count, 1u);
        if (done == gridDim.x - 1) {
          step_bookkeeping(a.scaler, a.beta1, a.beta2, a.bk_dynamic, a.bk_growth, a.bk_flip);
          a.scaler->finish_count = 0;
        }
      }
    }
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.n_ranks;
  const int n_plan = a.plan.n;
  volatile int* abort_flag = &sh_abort;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // lane 0 owns the barriers; the 32 lanes issue the stage's copies in
    // parallel (chunk c by lane c mod 32)
    const uint64_t pol = evict_first_policy();
    uint32_t it = 0;
    int slot = 0;
    uint32_t phase = 0;  // == (it / n_slots) & 1
    bool stop = false;
    for (int64_t g = blockIdx.x; g < a.n_tiles && !stop; g += gridDim.x) {
      const TileGeom t = tile_geom(a, g, kOff);
      const int64_t rank0 = static_cast<int64_t>(t.rank) * a.shard;
      for (int64_t j0 = t.va; j0 < t.vb && !stop; j0 += E) {
        const uint32_t len = static_cast<uint32_t>(min(static_cast<int64_t>(E), t.vb - j0));
        const int64_t w = j0 - a.wbase;
        const int64_t kk = j0 - rank0;
        // replica copies start at the 16-byte block holding element w
        const int64_t rw = w - t.shift;
        const uint32_t rlen = t.shift ? ((len + t.shift + 7) & ~7u) : len;
        // accumulator copies start at the 16-byte block holding element w
        const int32_t ashift = t.shift & 3;
        const int64_t aw = w - ashift;
        const uint32_t alen = (len + ashift + 3) & ~3u;
        // stage layout of this tile: replica chunks, accumulator chunks, states
        const int rstride = 2 * E + (t.shift ? kPad : 0);
        const int astride = 4 * E + (t.shift ? kPad : 0);
        const int rblock = kAcc ? rstride + astride : rstride;
        for (int st = 0; st < n_plan; ++st, ++it) {
          int go = 1;
          if (lane == 0) {
            if (*abort_flag) {
              go = 0;
            } else if (!mbar_wait(&empty_bar[slot], phase ^ 1u)) {
              set_error(a.scaler, ZERO_DEVERR_TIMEOUT);
              *abort_flag = 1;
              go = 0;
            } else {
              const uint32_t nr = static_cast<uint32_t>(a.plan.r_hi[st] - a.plan.r_lo[st]);
              const uint32_t ns = a.plan.states[st] ? (MODE == kUpdate ? 4u : 3u) : 0u;
              mbar_expect_tx(&full_bar[slot],
                             nr * (2 * rlen + (kAcc ? 4 * alen : 0)) + ns * 4 * len);
            }
          }
          if (!__shfl_sync(0xFFFFFFFFu, go, 0)) {
            stop = true;
            break;
          }
          unsigned char* buf = stage_mem + static_cast<size_t>(slot) * slot_bytes;
          const int r_lo = a.plan.r_lo[st], r_hi = a.plan.r_hi[st];
          const int n_rep = r_hi - r_lo;
          const int n_state = a.plan.states[st] ? (MODE == kUpdate ? 4 : 3) : 0;
          const int n_rep_chunks = kAcc ? 2 * n_rep : n_rep;
          for (int c = lane; c < n_rep_chunks + n_state; c += 32) {
            if (c < n_rep) {
              int rr = t.first_rep + r_lo + c;
              if (rr >= N) rr -= N;
              // a shifted copy may read the rest of the 16-byte block that
              // holds the window's last element
              if (ZCHECK(rw >= 0 && rw + rlen <= ((a.wend + 7) & ~static_cast<int64_t>(7)),
                         kSiteRepCopy, w) &&
                  ZCHECK(c * rstride + 2 * rlen <= slot_bytes, kSiteStageBytes, c))
                bulk_g2s(buf + static_cast<size_t>(c) * rstride, a.rep[rr] + rw, rlen * 2,
                         &full_bar[slot], pol);
            } else if (kAcc && c < n_rep_chunks) {
              int rr = t.first_rep + r_lo + (c - n_rep);
              if (rr >= N) rr -= N;
              if (ZCHECK(aw >= 0 && aw + alen <= ((a.wend + 3) & ~static_cast<int64_t>(3)),
                         kSiteAccCopy, w) &&
                  ZCHECK(n_rep * rstride + (c - n_rep) * astride + 4 * alen <= slot_bytes,
                         kSiteStageBytes, c))
                bulk_g2s(buf + static_cast<size_t>(n_rep) * rstride +
                             static_cast<size_t>(c - n_rep) * astride,
                         a.acc[rr] + aw, alen * 4, &full_bar[slot], pol);
            } else {
              const int q = c - n_rep_chunks;
              const float* src;
              if (MODE == kUpdate) {
                src = q == 0 ? a.ghat[t.rank]
                             : (q == 1 ? a.master[s.src][t.rank]
                                       : (q == 2 ? a.mom[s.src][t.rank] : a.var[s.src][t.rank]));
              } else {
                src = q == 0 ? a.master[s.src][t.rank]
                             : (q == 1 ? a.mom[s.src][t.rank] : a.var[s.src][t.rank]);
              }
              if (ZCHECK(kk >= 0 && kk + len <= a.shard, kSiteStateCopy, kk) &&
                  ZCHECK(n_rep * rblock + (q + 1) * (4 * E) <= static_cast<int>(slot_bytes),
                         kSiteStageBytes, c))
                bulk_g2s(buf + static_cast<size_t>(n_rep) * rblock +
                             static_cast<size_t>(q) * (4 * E),
                         src + kk, len * 4, &full_bar[slot], pol);
            }
          }
          __syncwarp();
          if (++slot == n_slots) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    // make sure no copy is still landing when the CTA exits (bounded)
    if (lane == 0) {
      const uint32_t issued = it;
      for (uint32_t back = 0; back < static_cast<uint32_t>(n_slots) && back < issued; ++back) {
        const uint32_t i = issued - 1 - back;
        if (!mbar_wait(&full_bar[i % n_slots], (i / n_slots) & 1u))
          set_error(a.scaler, ZERO_DEVERR_TIMEOUT);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;
  const int t_off = tid * EPT;
  int slot = 0;
  uint32_t phase = 0;
  uint32_t tile_no = 0;
  bool dead = false;
  const bool partials = MODE == kReduce && (a.mode_flags & kFlagPartials);
  for (int64_t g = blockIdx.x; g < a.n_tiles; g += gridDim.x, ++tile_no) {
    const TileGeom t = tile_geom(a, g, kOff);
    NormAcc nacc;
    uint64_t phi = 0, plo = 0;  // packed in-range accumulators (even | odd elements)
    bool bad = false;
    const int64_t rank0 = static_cast<int64_t>(t.rank) * a.shard;
    const int rstride = 2 * E + (t.shift ? kPad : 0);  // stage layout, as the producer's
    const int astride = 4 * E + (t.shift ? kPad : 0);
    const int rblock = kAcc ? rstride + astride : rstride;
    for (int64_t j0 = t.va; j0 < t.vb; j0 += E) {
      const int len = static_cast<int>(min(static_cast<int64_t>(E), t.vb - j0));
      const bool mine = t_off < len;
      const int64_t j = j0 + t_off;
      const int64_t w = j - a.wbase;
      const int64_t k = j - rank0;
      // ring sum in fp32, starting from -0 (x + -0 == x for every x, so this
      // equals starting from the first replica's value)
      float acc[EPT], gv[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[e] = -0.0f;
      for (int st = 0; st < n_plan; ++st) {
        const int cur = slot;
        const uint32_t ph = phase;
        if (++slot == n_slots) {
          slot = 0;
          phase ^= 1u;
        }
        // keep `dead` uniform across the warp so the warp-level syncs below
        // always see all 32 lanes
        if (!dead) dead = __any_sync(0xFFFFFFFFu, *abort_flag != 0);
        if (!dead) {
          const bool landed = mbar_wait(&full_bar[cur], ph);
          if (!__all_sync(0xFFFFFFFFu, landed)) {
            if (lane == 0) {
              set_error(a.scaler, ZERO_DEVERR_TIMEOUT);
              *abort_flag = 1;
            }
            dead = true;
          }
        }
        if (dead) continue;
        const unsigned char* buf = stage_mem + static_cast<size_t>(cur) * slot_bytes;
        const int r_lo = a.plan.r_lo[st], r_hi = a.plan.r_hi[st];
        if constexpr (MODE == kFused || MODE == kReduce) {
          const bool completes = r_hi == N && r_lo < r_hi;  // stage ends the range's sum
          if (mine) {
            if constexpr (kAcc) {
              const unsigned char* mp = buf + t_off * 2;
              const unsigned char* ap =
                  buf + static_cast<size_t>(r_hi - r_lo) * rstride + t_off * 4;
              if (kShift && t.shift)
                acc_stage_accum_shifted<kBf16>(mp, ap, rstride, astride, r_hi - r_lo,
                                               t.shift, acc);
              else
                acc_stage_accum<kBf16, EPT>(mp, ap, rstride, astride, r_hi - r_lo, acc);
            } else if (kShift && t.shift) {
              acc_stage_shifted<kBf16, EPT>(buf + t_off * 2, rstride, r_hi - r_lo, t.shift,
                                            acc);
            } else {
              acc_stage<kBf16, EPT>(buf + t_off * 2, rstride, r_hi - r_lo, acc);
            }
            if (completes) {
              const uint64_t inv2 = f2_pack(s.inv, s.inv);
#pragma unroll
              for (int i = 0; i < EPT / 2; ++i)
                f2_unpack(f2_mul(f2_pack(acc[2 * i], acc[2 * i + 1]), inv2), gv[2 * i],
                          gv[2 * i + 1]);
              if (!partials) {
#pragma unroll
                for (int e = 0; e < EPT; ++e) bad |= nonfinite(gv[e]);
              }
              if constexpr (MODE == kReduce) {
                if (ZCHECK(k >= 0 && k + EPT <= a.shard, kSiteStore, k))
                  stg_fv<EPT>(a.ghat[t.rank] + k, gv);
              }
            }
          }
          if (partials && completes) {
            // squares of this thread's elements on the straight-line
            // paired-fp32 path, whatever their size: a square of 2^112 or
            // more (|g| >= 2^56) or a non-finite one shows in the
            // accumulators at the end of the tile, which then redoes this
            // thread's body with the per-element split
            float q[EPT];
#pragma unroll
            for (int e = 0; e < EPT; ++e) q[e] = mine ? gv[e] : 0.0f;
#pragma unroll
            for (int i = 0; i < EPT / 2; ++i) ff2_add_sq(phi, plo, f2_pack(q[2 * i], q[2 * i + 1]));
          }
        }
        if (mine) {
          if constexpr (MODE == kFused || MODE == kUpdate) {
            if (a.plan.states[st]) {
              const unsigned char* sb = buf + static_cast<size_t>(r_hi - r_lo) * rblock;
              if constexpr (MODE == kUpdate) {
                lds_fv<EPT>(sb + t_off * 4, gv);
                sb += 4 * E;
                if (s.clip != 1.0f) {
#pragma unroll
                  for (int e = 0; e < EPT; ++e) gv[e] = __fmul_rn(gv[e], s.clip);
                }
              }
              float th[EPT], m[EPT], v[EPT];
              lds_fv<EPT>(sb + t_off * 4, th);
              lds_fv<EPT>(sb + 4 * E + t_off * 4, m);
              lds_fv<EPT>(sb + 8 * E + t_off * 4, v);
#pragma unroll
              for (int e = 0; e < EPT; ++e) adamw(th[e], m[e], v[e], gv[e], a, s);
              if (ZCHECK(k >= 0 && k + EPT <= a.shard && w >= 0 && w + EPT <= a.wend,
                         kSiteStore, k)) {
                stg_fv<EPT>(a.master[s.dst][t.rank] + k, th);
                stg_fv<EPT>(a.mom[s.dst][t.rank] + k, m);
                stg_fv<EPT>(a.var[s.dst][t.rank] + k, v);
                if (kOff && t.shift)
                  stg_hv_unaligned<kBf16>(a.flat + w, th);
                else
                  stg_hv<kBf16, EPT>(a.flat + w, th);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[cur]);
      }
    }
    // head [lo, va) and tail [vb, hi) outside the body, with plain loads,
    // after the body so that the producer streams the next tile meanwhile:
    // in the fused and reduce passes up to 32 such elements one warp each
    // (at most 7 on each side of a body), otherwise one thread per element
    // (coalesced)
    const int nhead = static_cast<int>(t.va - t.lo);
    const int ntail = static_cast<int>(t.hi - t.vb);
    bool by_warp = false;
    if constexpr (MODE == kFused || MODE == kReduce) by_warp = nhead + ntail <= 2 * kConsumerWarps;
    if (by_warp) {
      if constexpr (MODE == kFused || MODE == kReduce) {
        for (int q = warp; q < nhead + ntail; q += kConsumerWarps) {
          const int64_t j = q < nhead ? t.lo + q : t.vb + (q - nhead);
          do_scalar_warp<MODE, kBf16>(a, s, j, t.rank, t.first_rep, nacc, bad, lane);
        }
      }
    } else {
      for (int q = tid; q < nhead + ntail; q += kConsumers) {
        const int64_t j = q < nhead ? t.lo + q : t.vb + (q - nhead);
        do_scalar<MODE, kBf16>(a, s, j, t.rank, t.first_rep, nacc, bad);
      }
    }
    if constexpr (MODE == kFused || MODE == kReduce) {
      if (partials) {
        float h0, h1, l0, l1;
        f2_unpack(phi, h0, h1);
        f2_unpack(plo, l0, l1);
        if (h0 < kNormSumLimit && h1 < kNormSumLimit) {  // false for NaN as well
          nacc.merge(h0, l0, 0.f, 0.f);
          nacc.merge(h1, l1, 0.f, 0.f);
        } else if constexpr (MODE == kReduce) {
          // rare: redo this thread's body elements with the split into
          // in-range and scaled big squares, from the reduced gradient this
          // thread stored above (its own stores, so its loads see them)
          for (int64_t j0 = t.va; j0 < t.vb && !dead; j0 += E) {
            const int len = static_cast<int>(min(static_cast<int64_t>(E), t.vb - j0));
            const int64_t k = j0 + t_off - rank0;
            if (t_off < len && ZCHECK(k >= 0 && k + EPT <= a.shard, kSiteLoad, k)) {
              const float* gp = a.ghat[t.rank] + k;
#pragma unroll
              for (int e = 0; e < EPT; ++e) nacc.add(gp[e]);
            }
          }
        }
        bad |= nacc.nonfinite_seen();
      }
      if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) raise_flag(a, t.bucket);
    }
    if constexpr (MODE == kReduce) {
      if (a.mode_flags & kFlagPartials) {
        // Each thread leaves its in-range sums in shared memory; only the
        // rare sums of big (or non-finite) squares are merged per warp, and
        // only in a warp that has any. One barrier, then the tile's record
        // warp merges everything in a fixed order.
        const int par = tile_no & 1;
        sh_sums[par][tid] = make_float2(nacc.hi, nacc.lo);
        float bh = nacc.bhi, bl = nacc.blo;
        if (__any_sync(0xFFFFFFFFu, bh != 0.f || bl != 0.f)) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const float h2 = __shfl_down_sync(0xFFFFFFFFu, bh, off);
            const float l2 = __shfl_down_sync(0xFFFFFFFFu, bl, off);
            if (lane < off) ff_merge(bh, bl, h2, l2);
          }
        }
        if (lane == 0) {
          sh_norm.bhi[par][warp] = bh;
          sh_norm.blo[par][warp] = bl;
        }
        consumer_sync();
        if (warp == static_cast<int>(tile_no % kConsumerWarps)) {
          const float4 rec =
              tile_norm_record_lanes(sh_sums[par], sh_norm, par, kConsumerWarps, lane);
          if (lane == 0 &&
              ZCHECK(t.partial >= 0 && t.partial < a.n_records, kSiteRecord, t.partial))
            a.partials[t.partial] = rec;
        }
      }
    }
  }
  if constexpr (MODE == kFused) {
    if (a.mode_flags & kFlagFinish) fused_finish<kBf16>(a, s);
  }
}

// ------------------------------------------------------------ short steps --
//
// A fused step over few elements is bound by start-up and by how evenly its
// work spreads over the SMs, not by DRAM: 34 MB of a 1M-parameter step at
// N = 4 arrive in about 5 us. short_fused_kernel takes such a step in one
// wave of small CTAs. Every CTA works inside one owner's slice, so the
// owner and every pointer derived from it are the same for all its
// threads. Each thread owns 4 consecutive shard elements (16-byte aligned
// in the shard), issues its replica loads before the step scalars are
// known, then its state loads, and finishes the elements with the
// operations of the pipelined pass in the same order (ring sum from the
// first replica in ring order, unscale, vote, AdamW, cast), so the results
// are the same bits. The last CTA to finish does the step's bookkeeping,
// after re-casting the parameters from the kept state set when the step
// overflowed. No CTA waits for another.
// 256 threads, 8 CTAs per SM: half as many CTAs count at the end as with 128 (at least 128:
// threads 0, 32, 64 and 96 form the step scalars)
constexpr int kShortThreads = 256;
constexpr int kShortChunk = 4;  // replicas whose loads are in flight together
constexpr uint32_t kShortVoteUnit = 1u << 16;  // finish_count: CTAs below, votes above

// The fused pass's step scalars, computed by four threads of different warps
// at once (every warp of the CTA waits for the last of them), plus the
// scaler fields the bookkeeping needs. Same values as
// compute_step_scalars<kFused>.
__device__ __forceinline__ void short_step_scalars(const Args& a, StepScalars* sh,
                                                   ScalerSnap* snap) {
  zero_scaler* sc = a.scaler;
  const int t = threadIdx.x;
  if (t == 0) {
    const float sl = sc->scale;
    sh->inv = inverse_scale(sl, a.n_ranks, a.n_micro);
    sh->clip = 1.0f;
    snap->scale = sl;
  } else if (t == 32) {
    bias_correction(sc->beta1_pow, a.beta1, &snap->p1, &sh->bc1);
  } else if (t == 64) {
    bias_correction(sc->beta2_pow, a.beta2, &snap->p2, &sh->bc2);
  } else if (t == 96) {
    snap->pending = sc->pending;
    snap->good_steps = sc->good_steps;
    snap->t = sc->t;
    snap->n_skipped = sc->n_skipped;
    const int idx = sc->state_index;
    snap->state_index = idx;
    int skip = 0;
    if (idx < 0 || idx >= a.n_sets || a.n_sets != 2) {
      set_error(sc, ZERO_DEVERR_STATE_INDEX);
      skip = 1;
    }
    sh->src = idx;
    sh->dst = idx ^ 1;
    sh->skip = skip;
  }
}

// 4 consecutive 16-bit values at element offset w of p (a 16-byte aligned
// window): one 8-byte load when w is a multiple of 4, two 4-byte loads when
// it is even, four 2-byte loads otherwise. `shift` is w mod 4, the same for
// every thread of a CTA.
__device__ __forceinline__ void ld4_h(const unsigned short* p, int64_t w, int shift,
                                      uint32_t (&h)[4]) {
  if (shift == 0) {
    const uint2 x = __ldcs(reinterpret_cast<const uint2*>(p + w));
    h[0] = x.x & 0xFFFFu; h[1] = x.x >> 16; h[2] = x.y & 0xFFFFu; h[3] = x.y >> 16;
  } else if (shift == 2) {
    const uint32_t x = __ldcs(reinterpret_cast<const unsigned int*>(p + w));
    const uint32_t y = __ldcs(reinterpret_cast<const unsigned int*>(p + w) + 1);
    h[0] = x & 0xFFFFu; h[1] = x >> 16; h[2] = y & 0xFFFFu; h[3] = y >> 16;
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __ldcs(p + w + e);
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kShortThreads, 2048 / kShortThreads) short_fused_kernel(
    const __grid_constant__ Args a, int32_t own_lo, uint32_t ctas_per_owner,
    uint32_t quads_per_owner) {
  __shared__ StepScalars sh_s;
  __shared__ ScalerSnap sh_snap;
  __shared__ int sh_last;
  pdl_begin();
  short_step_scalars(a, &sh_s, &sh_snap);
  // the CTA's owner (uniform); 32-bit quad indices: the host takes this
  // kernel for at most kShortMaxElems elements
  const uint32_t o = blockIdx.x / ctas_per_owner;
  const int32_t rank = own_lo + static_cast<int32_t>(o);
  const uint32_t qi = (blockIdx.x - o * ctas_per_owner) * kShortThreads + threadIdx.x;
  const int64_t k0 = static_cast<int64_t>(qi) * 4;
  int n = qi < quads_per_owner ? static_cast<int>(min(static_cast<int64_t>(4), a.shard - k0)) : 0;
  const int64_t wr = static_cast<int64_t>(rank) * a.shard - a.wbase;  // owner's window offset
  const int64_t w0 = wr + k0;
  const int64_t j0 = w0 + a.wbase;
  const int shift = static_cast<int>(wr & 3);
  const int N = a.n_ranks;
  const int first_rep = rank + 1 == N ? 0 : rank + 1;
  if (n > 0 && !ZCHECK(w0 >= 0 && w0 + n <= a.wend && k0 + n <= a.shard, kSiteVector, j0))
    n = 0;
  float acc[4] = {-0.0f, -0.0f, -0.0f, -0.0f};
  for (int base = 0; base < N; base += kShortChunk) {
    uint32_t h[kShortChunk][4];
#pragma unroll
    for (int c = 0; c < kShortChunk; ++c) {
      const int p = base + c;
      if (p < N) {
        int rr = first_rep + p;
        if (rr >= N) rr -= N;
        const unsigned short* src = reinterpret_cast<const unsigned short*>(a.rep[rr]);
        if (n == 4) {
          ld4_h(src, w0, shift, h[c]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) h[c][e] = e < n ? __ldcs(src + w0 + e) : 0u;
        }
      }
    }
#pragma unroll
    for (int c = 0; c < kShortChunk; ++c) {
      if (base + c < N) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(acc[e], widen<kBf16>(h[c][e]));
      }
    }
  }
  // the state set read is the scaler's index: each thread reads it itself,
  // so its state loads go out before the step scalars are in shared memory
  // (an index outside the sets reads set 0 here, and the scalars then skip
  // the step); both sets' pointers are uniform, the choice a select
  const int src = a.scaler->state_index == 1 && a.n_sets == 2 ? 1 : 0;
  float th[4], m[4], v[4];
  if (n > 0) {
    const float* pm = (src ? a.master[1][rank] : a.master[0][rank]) + k0;
    const float* pv1 = (src ? a.mom[1][rank] : a.mom[0][rank]) + k0;
    const float* pv2 = (src ? a.var[1][rank] : a.var[0][rank]) + k0;
    if (n == 4) {
      const float4 x = __ldcs(reinterpret_cast<const float4*>(pm));
      const float4 y = __ldcs(reinterpret_cast<const float4*>(pv1));
      const float4 z = __ldcs(reinterpret_cast<const float4*>(pv2));
      th[0] = x.x; th[1] = x.y; th[2] = x.z; th[3] = x.w;
      m[0] = y.x; m[1] = y.y; m[2] = y.z; m[3] = y.w;
      v[0] = z.x; v[1] = z.y; v[2] = z.z; v[3] = z.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        th[e] = e < n ? pm[e] : 0.0f;
        m[e] = e < n ? pv1[e] : 0.0f;
        v[e] = e < n ? pv2[e] : 0.0f;
      }
    }
  }
  __syncthreads();
  const StepScalars s = sh_s;
  bool raised = false;
  if (!s.skip && n > 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e < n) {
        const float g = __fmul_rn(acc[e], s.inv);
        if (nonfinite(g)) {
          if (!raised) atomicOr(&a.scaler->pending, 1u);
          raised = true;
          if (a.flags)
            atomicOr(&a.flags[a.bucket_elems ? (j0 + e) / a.bucket_elems : 0], 1u);
        }
        adamw(th[e], m[e], v[e], g, a, s);
      }
    }
    float* qm = (s.dst ? a.master[1][rank] : a.master[0][rank]) + k0;
    float* qv1 = (s.dst ? a.mom[1][rank] : a.mom[0][rank]) + k0;
    float* qv2 = (s.dst ? a.var[1][rank] : a.var[0][rank]) + k0;
    if (n == 4) {
      __stcs(reinterpret_cast<float4*>(qm), make_float4(th[0], th[1], th[2], th[3]));
      __stcs(reinterpret_cast<float4*>(qv1), make_float4(m[0], m[1], m[2], m[3]));
      __stcs(reinterpret_cast<float4*>(qv2), make_float4(v[0], v[1], v[2], v[3]));
      stg_hv_unaligned<kBf16>(a.flat + w0, th);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e < n) {
          qm[e] = th[e];
          qv1[e] = m[e];
          qv2[e] = v[e];
          a.flat[w0 + e] = narrow<kBf16>(th[e]);
        }
      }
    }
  }
  // The step's bookkeeping, once, by the last CTA to finish. The CTA count
  // and the number of CTAs that saw a non-finite gradient share one word
  // (low and high 16 bits; at most 2^18 / kShortThreads + 4 CTAs), so the
  // last CTA learns the step's vote from its own atomic: together with the
  // pending word read at the start (a vote of an earlier launch) it is the
  // pending word at the end. The scaler's other fields were read at the
  // start too (nothing else writes them during the step), so the
  // bookkeeping is stores only. The fence before the count orders this
  // CTA's parameter stores before an overflowed step's re-cast.
  const int cta_raised = __syncthreads_or(raised ? 1 : 0);
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old =
        atomicAdd(&a.scaler->finish_count, cta_raised ? kShortVoteUnit + 1u : 1u);
    const bool last = (old & (kShortVoteUnit - 1u)) == gridDim.x - 1;
    const bool ov = (old >> 16) != 0 || cta_raised || sh_snap.pending != 0;
    sh_last = last ? (ov ? 2 : 1) : 0;
  }
  __syncthreads();
  if (!sh_last) return;
  const bool ov = sh_last == 2;
  if (!s.skip && ov) {
    __threadfence();  // the other CTAs' parameter stores come before the re-cast's
    // re-cast every owner's parameters from the kept set, four quads in
    // flight per thread
    const uint32_t qpo = quads_per_owner;
    const uint32_t n_quads = (gridDim.x / ctas_per_owner) * qpo;
    for (uint32_t q0 = threadIdx.x; q0 < n_quads; q0 += 4 * kShortThreads) {
      float4 x[4];
      int64_t kk[4], ww[4];
      int nn[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t qq = q0 + u * kShortThreads;
        nn[u] = 0;
        if (qq < n_quads) {
          const uint32_t o = qq / qpo;
          const int32_t r = own_lo + static_cast<int32_t>(o);
          kk[u] = static_cast<int64_t>(qq - o * qpo) * 4;
          nn[u] = static_cast<int>(min(static_cast<int64_t>(4), a.shard - kk[u]));
          ww[u] = static_cast<int64_t>(r) * a.shard + kk[u] - a.wbase;
          const float* pm = a.master[s.src][r] + kk[u];
          if (nn[u] == 4) {
            x[u] = __ldcs(reinterpret_cast<const float4*>(pm));
          } else {
            x[u] = make_float4(pm[0], nn[u] > 1 ? pm[1] : 0.f, nn[u] > 2 ? pm[2] : 0.f, 0.f);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (nn[u] == 0 || !ZCHECK(ww[u] >= 0 && ww[u] + nn[u] <= a.wend, kSiteStore, ww[u]))
          continue;
        if (nn[u] == 4) {
          const float t4[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
          stg_hv_unaligned<kBf16>(a.flat + ww[u], t4);
        } else {
          a.flat[ww[u]] = narrow<kBf16>(x[u].x);
          if (nn[u] > 1) a.flat[ww[u] + 1] = narrow<kBf16>(x[u].y);
          if (nn[u] > 2) a.flat[ww[u] + 2] = narrow<kBf16>(x[u].z);
        }
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    bookkeeping_store(a.scaler, sh_snap, ov, a.bk_dynamic, a.bk_growth, a.bk_flip);
    a.scaler->finish_count = 0;
  }
}

// Norm finish. The global squared norm is defined so that it does not depend
// on how the owners are split over calls or processes:
//   owner record R_i: owner i's tile records merged in float-float over a
//     fixed partition of its own tiles (kOwnerBlocks contiguous shares;
//     inside a share thread k takes every kFinishThreads-th record, then a
//     fixed CTA tree; the kOwnerBlocks share records then a fixed 16-lane
//     shuffle tree);
//   total = R_lo + ... + R_{hi-1}: float-float merges in ascending owner
//     order (a zero record merges as the identity, so owners outside a
//     window change nothing);
//   norm^2 = hi + lo + 2^192 (bhi + blo) in fp64, the norm and the clip
//     coefficient c = max_norm / (norm + 1e-6) in fp64 (applied, rounded to
//     fp32, only when c < 1).
// R_i depends only on owner i's gradients, so processes that own disjoint
// windows can export their records (norm_final_kernel, export mode), add the
// exports up and import the sum (norm_import_kernel): each then holds what
// one call over all owners computes, bit for bit.
constexpr int kOwnerBlocks = zero_detail::kNormOwnerBlocks;
constexpr int kFinishThreads = 256;
static_assert(kOwnerBlocks * ZERO_MAX_RANKS <= 1024, "one final CTA holds every share record");

// first tile (plan numbering) of each owner of a window, plus the end
struct OwnerTiles {
  int64_t t[ZERO_MAX_RANKS + 1];
};

// Merge the kFinishThreads per-thread accumulators of a CTA; result in
// thread 0.
__device__ NormAcc cta_merge(NormAcc t, float4* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float h2 = __shfl_down_sync(0xFFFFFFFFu, t.hi, off);
    float l2 = __shfl_down_sync(0xFFFFFFFFu, t.lo, off);
    float bh2 = __shfl_down_sync(0xFFFFFFFFu, t.bhi, off);
    float bl2 = __shfl_down_sync(0xFFFFFFFFu, t.blo, off);
    if (lane < off) t.merge(h2, l2, bh2, bl2);
  }
  if (lane == 0) sh[warp] = make_float4(t.hi, t.lo, t.bhi, t.blo);
  __syncthreads();
  NormAcc r;
  if (warp == 0) {
    if (lane < kFinishThreads / 32) {
      const float4 q = sh[lane];
      r.hi = q.x;
      r.lo = q.y;
      r.bhi = q.z;
      r.blo = q.w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float h2 = __shfl_down_sync(0xFFFFFFFFu, r.hi, off);
      float l2 = __shfl_down_sync(0xFFFFFFFFu, r.lo, off);
      float bh2 = __shfl_down_sync(0xFFFFFFFFu, r.bhi, off);
      float bl2 = __shfl_down_sync(0xFFFFFFFFu, r.blo, off);
      if (lane < off) r.merge(h2, l2, bh2, bl2);
    }
  }
  return r;
}

// CTA (b, i): share b of the tiles of owner rank_lo + i. Tile t's record is
// records[t - rec_base]; the share's record goes to
// blocks[owner * kOwnerBlocks + b].
__global__ void __launch_bounds__(kFinishThreads) norm_owner_kernel(
    const float4* __restrict__ records, int64_t rec_base, int64_t n_records,
    const __grid_constant__ OwnerTiles ot, int32_t rank_lo, float4* __restrict__ blocks) {
  __shared__ float4 sh[kFinishThreads / 32];
  pdl_begin();
  const int i = blockIdx.y;
  const int64_t t0 = ot.t[i], t1 = ot.t[i + 1];
  const int64_t chunk = (t1 - t0 + kOwnerBlocks - 1) / kOwnerBlocks;
  const int64_t b0 = t0 + blockIdx.x * chunk;
  const int64_t b1 = min(b0 + chunk, t1);
  NormAcc t;
  for (int64_t k = b0 + threadIdx.x; k < b1; k += kFinishThreads) {
    const int64_t r = k - rec_base;
    if (!ZCHECK(r >= 0 && r < n_records, kSiteRecord, r)) continue;
    const float4 q = records[r];
    t.merge(q.x, q.y, q.z, q.w);
  }
  const NormAcc m = cta_merge(t, sh);
  if (threadIdx.x == 0)
    blocks[(rank_lo + i) * kOwnerBlocks + blockIdx.x] = make_float4(m.hi, m.lo, m.bhi, m.blo);
}

// norm^2, the norm and the clip coefficient from a total record.
__device__ void finish_norm(const NormAcc& r, double max_norm, zero_scaler* sc) {
  double nsq = __dadd_rn(static_cast<double>(r.hi), static_cast<double>(r.lo));
  if (r.bhi != 0.f || r.blo != 0.f)
    nsq = __dadd_rn(nsq, __dmul_rn(__dadd_rn(static_cast<double>(r.bhi),
                                             static_cast<double>(r.blo)),
                                   0x1p192));
  const double nrm = __dsqrt_rn(nsq);
  const double c = __ddiv_rn(max_norm, __dadd_rn(nrm, 1e-6));
  sc->norm_sq = nsq;
  sc->norm = nrm;
  sc->clip_apply = c < 1.0 ? 1 : 0;
  sc->clip_coef = c < 1.0 ? __double2float_rn(c) : 1.0f;
  sc->norm_step = sc->t + 1;
}

constexpr int kFinalThreads = kOwnerBlocks * ZERO_MAX_RANKS;

// One CTA. Owner records R_o of [rank_lo, rank_hi) from the share records
// (16 lanes per owner). Apply mode: total in ascending owner order, then
// the scaler's norm fields. Export mode: the records of the window and
// zeros elsewhere, and the scaler's overflow word, into *ex.
__global__ void __launch_bounds__(kFinalThreads) norm_final_kernel(
    const float4* __restrict__ blocks, int32_t rank_lo, int32_t rank_hi, int32_t export_mode,
    double max_norm, zero_scaler* sc, zero_exchange* ex) {
  __shared__ float4 sh_owner[ZERO_MAX_RANKS];
  pdl_begin();
  const int tid = threadIdx.x;
  const int o = rank_lo + tid / kOwnerBlocks;
  const int part = tid % kOwnerBlocks;
  NormAcc t;
  if (o < rank_hi) {
    const float4 q = blocks[o * kOwnerBlocks + part];
    t.hi = q.x;
    t.lo = q.y;
    t.bhi = q.z;
    t.blo = q.w;
  }
#pragma unroll
  for (int off = kOwnerBlocks / 2; off > 0; off >>= 1) {
    float h2 = __shfl_down_sync(0xFFFFFFFFu, t.hi, off, kOwnerBlocks);
    float l2 = __shfl_down_sync(0xFFFFFFFFu, t.lo, off, kOwnerBlocks);
    float bh2 = __shfl_down_sync(0xFFFFFFFFu, t.bhi, off, kOwnerBlocks);
    float bl2 = __shfl_down_sync(0xFFFFFFFFu, t.blo, off, kOwnerBlocks);
    if (part < off) t.merge(h2, l2, bh2, bl2);
  }
  if (part == 0 && o < rank_hi) sh_owner[o] = make_float4(t.hi, t.lo, t.bhi, t.blo);
  __syncthreads();
  if (export_mode) {
    for (int k = tid; k < ZERO_MAX_RANKS; k += kFinalThreads) {
      const float4 q = (k >= rank_lo && k < rank_hi) ? sh_owner[k] : make_float4(0.f, 0.f, 0.f, 0.f);
      ex->owner[k].hi = q.x;
      ex->owner[k].lo = q.y;
      ex->owner[k].big_hi = q.z;
      ex->owner[k].big_lo = q.w;
    }
    if (tid == 0) {
      ex->overflow = sc->pending ? 1u : 0u;
      ex->reserved[0] = ex->reserved[1] = ex->reserved[2] = 0u;
    }
    return;
  }
  if (tid == 0) {
    NormAcc total;
    for (int k = rank_lo; k < rank_hi; ++k) {
      const float4 q = sh_owner[k];
      total.merge(q.x, q.y, q.z, q.w);
    }
    finish_norm(total, max_norm, sc);
  }
}

// Import of an exchange: the step's overflow word, and with clipping the
// norm fields from the records of all n_ranks owners in ascending order.
__global__ void norm_import_kernel(const zero_exchange* ex, int32_t n_ranks, int32_t clip,
                                   double max_norm, zero_scaler* sc) {
  pdl_begin();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  if (ex->overflow) sc->pending |= 1u;
  if (!clip) return;
  NormAcc total;
  for (int k = 0; k < n_ranks; ++k) {
    const zero_norm_record q = ex->owner[k];
    total.merge(q.hi, q.lo, q.big_hi, q.big_lo);
  }
  finish_norm(total, max_norm, sc);
}

// First tile (plan numbering) of owner o; the plan's tile count for o = N.
int64_t owner_tile0(const zero_plan* p, int32_t o) {
  const int32_t s = p->rank_seg0[o];
  return s < p->info.n_segments ? p->seg_tile0[s] : p->info.n_tiles;
}

// The owner records of [rank_lo, rank_hi) from the tile records, into
// blocks (kOwnerBlocks share records per owner, indexed by absolute owner);
// then the final kernel in apply or export mode. Tile t's record is
// records[t - rec_base], n_records of them.
int launch_norm_finish(const zero_plan* p, int32_t rank_lo, int32_t rank_hi,
                       const float4* records, int64_t rec_base, int64_t n_records, float4* blocks,
                       int export_mode, double max_norm, zero_scaler* sc, zero_exchange* ex,
                       cudaStream_t st) {
  if (rank_hi > rank_lo) {
    OwnerTiles ot{};
    for (int32_t o = rank_lo; o <= rank_hi; ++o) ot.t[o - rank_lo] = owner_tile0(p, o);
    if (launch_pdl(norm_owner_kernel, dim3(kOwnerBlocks, rank_hi - rank_lo),
                   dim3(kFinishThreads), 0, st, records, rec_base, n_records, ot, rank_lo,
                   blocks) != cudaSuccess)
      return ZERO_ECUDA;
  }
  if (launch_pdl(norm_final_kernel, dim3(1), dim3(kFinalThreads), 0, st,
                 static_cast<const float4*>(blocks), rank_lo, rank_hi, export_mode, max_norm,
                 sc, ex) != cudaSuccess)
    return ZERO_ECUDA;
  return ZERO_OK;
}

// Bookkeeping alone (two-pass path, and plans without elements).
__global__ void scaler_finish_kernel(zero_scaler* sc, double beta1, double beta2, int dynamic,
                                     int growth_interval, int flip_sets) {
  pdl_begin();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  step_bookkeeping(sc, beta1, beta2, dynamic, growth_interval, flip_sets);
}

// Self-test of the bounded wait: nothing ever arrives on the barrier.
__global__ void wait_timeout_probe_kernel(zero_scaler* sc, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, limit_ns)) set_error(sc, ZERO_DEVERR_TIMEOUT);
}

// ----------------------------------------------------------- launch layer --

// Launch configuration, queried once per device and kept: the SM count, the
// resident CTAs per SM of a kernel at a given block and dynamic shared
// memory size, and the kernel's dynamic shared memory limit (raised only
// when a launch needs more than the last setting). These runtime calls cost
// microseconds each, which a short step or a small bucket would otherwise
// pay on every call.
constexpr int kCfgDevices = 64;
std::mutex g_cfg_mu;
int g_cfg_sms[kCfgDevices] = {};
std::map<std::tuple<const void*, int, int, size_t>, int> g_cfg_resident;
std::map<std::pair<const void*, int>, size_t> g_cfg_smem_limit;

// SM count of the current device (0 on error).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kCfgDevices) return 0;
  std::lock_guard<std::mutex> lock(g_cfg_mu);
  if (!g_cfg_sms[dev]) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_cfg_sms[dev] = sms;
  }
  return g_cfg_sms[dev];
}

// Resident CTAs per SM of `fn` on the current device (at least 1), or -1 on
// error. big_smem: first make sure the kernel's dynamic shared memory limit
// admits `smem` bytes.
int resident_ctas(const void* fn, int threads, size_t smem, bool big_smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(g_cfg_mu);
  if (big_smem) {
    size_t& limit = g_cfg_smem_limit[{fn, dev}];
    if (limit < smem) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return -1;
      limit = smem;
    }
  }
  const auto key = std::make_tuple(fn, dev, threads, smem);
  auto it = g_cfg_resident.find(key);
  if (it == g_cfg_resident.end()) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess)
      return -1;
    it = g_cfg_resident.emplace(key, std::max(per_sm, 1)).first;
  }
  return it->second;
}

template <int MODE, bool kBf16>
int grid_size() {
  const int sms = device_sms();
  const int per_sm =
      resident_ctas(reinterpret_cast<const void*>(step_kernel<MODE, kBf16>), kThreads, 0, false);
  if (sms <= 0 || per_sm <= 0) return -1;
  return sms * per_sm;
}

// Greedy packing of one element range's chunks (range of E elements) into
// stages of at most kStageBudget bytes: replica chunks (2 bytes per element
// each, 6 with the fp32 accumulator beside it) in ring order, then the indivisible state block (kFused 12, kUpdate
// 16 bytes per element) in the last stage if it fits, else in a stage of
// its own. rep_extra bytes follow every replica chunk (the 16-byte block a
// shifted body's chunk copies ahead of its first element); the slot holds
// the largest stage.
inline StagePlan make_stage_plan(int mode, int n_ranks, int E, int rep_bytes, int rep_extra,
                                 uint32_t* slot_bytes) {
  StagePlan pl{};
  const int budget = kStageBudget / E;  // bytes per element
  const int n_rep = mode == kUpdate ? 0 : n_ranks;
  const int state_bpe = mode == kFused ? 12 : (mode == kUpdate ? 16 : 0);
  int lo = 0, cur = 0;
  int64_t max_bytes = 0;
  bool overflow = false;
  auto close = [&](int hi, int with_states) {
    const int bpe = rep_bytes * (hi - lo) + (with_states ? state_bpe : 0);
    if (pl.n >= kMaxStagePlan) {  // reported through n = 0 below
      overflow = true;
      return;
    }
    pl.r_lo[pl.n] = static_cast<int16_t>(lo);
    pl.r_hi[pl.n] = static_cast<int16_t>(hi);
    pl.states[pl.n] = with_states;
    pl.bytes_per_elem[pl.n] = bpe;
    max_bytes = std::max(max_bytes, static_cast<int64_t>(bpe) * E +
                                        static_cast<int64_t>(rep_extra) * (hi - lo));
    ++pl.n;
    lo = hi;
    cur = 0;
  };
  for (int p = 0; p < n_rep; ++p) {
    if (cur + rep_bytes > budget) close(p, 0);
    cur += rep_bytes;
  }
  if (state_bpe > 0) {
    if (cur > 0 && cur + state_bpe <= budget) {
      close(n_rep, 1);
    } else {
      if (cur > 0) close(n_rep, 0);
      close(n_rep, 1);
    }
  } else if (cur > 0) {
    close(n_rep, 0);
  }
  if (overflow) pl.n = 0;
  *slot_bytes = static_cast<uint32_t>((max_bytes + 127) & ~static_cast<int64_t>(127));
  return pl;
}

template <int MODE, bool kBf16, int EPT, bool kAcc, bool kOff>
int launch_bulk_ept(Args& a, int64_t tiles, cudaStream_t stream) {
  constexpr int E = kConsumers * EPT;
  uint32_t slot_bytes = 0;
  constexpr int kRepExtra = kOff && (MODE == kFused || MODE == kReduce) ? (kAcc ? 32 : 16) : 0;
  a.plan = make_stage_plan(MODE, a.n_ranks, E, kAcc ? 6 : 2, kRepExtra, &slot_bytes);
  if (a.plan.n < 1 || a.plan.n > kMaxStagePlan || slot_bytes == 0) return ZERO_ERANGE;
  const int slots = std::min(kMaxStages, kSmemCap / static_cast<int>(slot_bytes));
  if (slots < 2) return ZERO_ERANGE;
  const size_t smem = static_cast<size_t>(slots) * slot_bytes;
  auto kern = bulk_kernel<MODE, kBf16, EPT, kAcc, kOff>;
  const int sms = device_sms();
  const int per_sm = resident_ctas(reinterpret_cast<const void*>(kern), kBulkThreads, smem, true);
  if (sms <= 0 || per_sm <= 0) return ZERO_ECUDA;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(std::min<int64_t>(tiles, cap));
  return launch_pdl(kern, dim3(grid), dim3(kBulkThreads), smem, stream, a, slots, slot_bytes) ==
                 cudaSuccess
             ? ZERO_OK
             : ZERO_ECUDA;
}

// The reduce pass moves few bytes per element at small N, so its fixed
// per-range costs are amortised over 4096-element ranges (8 elements per
// consumer thread, one tile) whenever a range's replicas fit one stage
// (N <= 8); the update and fused passes measured faster with 2048-element
// ranges and more, smaller slots.
template <int MODE, bool kBf16, bool kOff>
int launch_bulk_off(Args& a, int64_t tiles, cudaStream_t stream) {
  if constexpr (MODE == kFused || MODE == kReduce) {
    if (a.has_acc) return launch_bulk_ept<MODE, kBf16, 4, true, kOff>(a, tiles, stream);
  }
  if constexpr (MODE == kReduce) {
    if (2 * a.n_ranks * kConsumers * 8 <= kStageBudget)
      return launch_bulk_ept<MODE, kBf16, 8, false, kOff>(a, tiles, stream);
  }
  return launch_bulk_ept<MODE, kBf16, 4, false, kOff>(a, tiles, stream);
}

// The reduce and update passes are built twice: with support for owners
// off the windows' 8-element grid (shifted bodies) and without it. The
// leaner build runs whenever every owner of the launch is on the grid:
// carrying the shifted paths measured 2-3 % slower in aligned reduce and
// update passes on one box (no different on another). The fused pass
// measured the other way round: 167.2 against 162.6 Gparams/s on the GPT-2
// list at N = 8 with the shifted paths built in (same box, same data), so
// it always runs that build.
template <int MODE, bool kBf16>
int launch_bulk(Args& a, int64_t tiles, cudaStream_t stream) {
  if constexpr (MODE == kFused) {
    return launch_bulk_off<MODE, kBf16, true>(a, tiles, stream);
  } else {
    bool off = false;
    for (int i = 0; i < a.n_segs; ++i)
      off = off || ((static_cast<int64_t>(a.segs[i].rank) * a.shard - a.wbase) & 7) != 0;
    return off ? launch_bulk_off<MODE, kBf16, true>(a, tiles, stream)
               : launch_bulk_off<MODE, kBf16, false>(a, tiles, stream);
  }
}

template <int MODE, bool kBf16>
int launch_mode(const zero_plan* p, Args& a, int32_t seg_begin, int32_t seg_end,
                cudaStream_t stream) {
  constexpr bool kBulk = MODE == kFused || MODE == kReduce || MODE == kUpdate;
  const bool finish = MODE == kCast && (a.mode_flags & kFlagFinish);
  int grid_cap = 1;
  if constexpr (!kBulk) grid_cap = grid_size<MODE, kBf16>();
  if (grid_cap <= 0) return ZERO_ECUDA;
  if (finish) {
    // one CTA per SM: the no-overflow case exits at once, the rare re-cast
    // still has every SM
    const int sms = device_sms();
    if (sms <= 0) return ZERO_ECUDA;
    grid_cap = std::min(grid_cap, sms);
  }
  const int flags = a.mode_flags;
  for (int32_t s0 = seg_begin; s0 < seg_end; s0 += kMaxSegs) {
    const int32_t s1 = std::min(seg_end, s0 + kMaxSegs);
    // the bookkeeping rides on the last launch only
    a.mode_flags = (finish && s1 < seg_end) ? (flags & ~kFlagFinish) : flags;
    int64_t tiles = 0;
    for (int32_t s = s0; s < s1; ++s) {
      Seg& d = a.segs[s - s0];
      d.lo = p->segs[s].lo;
      d.hi = p->segs[s].hi;
      d.rank = p->segs[s].rank;
      d.bucket = p->segs[s].bucket;
      d.tile_local0 = tiles;
      d.tile_global0 = p->seg_tile0[s];
      tiles += p->seg_tiles[s];
    }
    a.n_segs = s1 - s0;
    a.n_tiles = tiles;
    // extents for the checked build: the window indices this launch may
    // touch and the records the workspace holds
    a.wend = p->segs[s1 - 1].hi - a.wbase;
    a.n_records = p->info.n_tiles;
    if (tiles == 0) continue;
    if constexpr (kBulk) {
      const int rc = launch_bulk<MODE, kBf16>(a, tiles, stream);
      if (rc) return rc;
    } else {
      const int grid = static_cast<int>(std::min<int64_t>(tiles, grid_cap));
      if (launch_pdl(step_kernel<MODE, kBf16>, dim3(grid), dim3(kThreads), 0, stream, a) !=
          cudaSuccess)
        return ZERO_ECUDA;
    }
  }
  return ZERO_OK;
}

template <int MODE>
int launch(const zero_plan* p, Args& a, int32_t seg_begin, int32_t seg_end, cudaStream_t st) {
  if (p->info.grad_dtype == ZERO_BF16) return launch_mode<MODE, true>(p, a, seg_begin, seg_end, st);
  return launch_mode<MODE, false>(p, a, seg_begin, seg_end, st);
}

void fill_constants(Args& a, const zero_hparams* hp) {
  a.b1 = static_cast<float>(hp->beta1);
  a.omb1 = static_cast<float>(1.0 - hp->beta1);
  a.b2 = static_cast<float>(hp->beta2);
  a.omb2 = static_cast<float>(1.0 - hp->beta2);
  a.lr = static_cast<float>(hp->lr);
  const double lr_wd = hp->lr * hp->weight_decay;
  a.decay = static_cast<float>(1.0 - lr_wd);
  a.eps = static_cast<float>(hp->eps);
  a.beta1 = hp->beta1;
  a.beta2 = hp->beta2;
}

bool ranks_ok(const zero_plan* p, int32_t lo, int32_t hi) {
  return p && lo >= 0 && hi <= p->info.n_ranks && lo < hi;
}

int check_ptr_array(const void* const* arr, int32_t lo, int32_t hi, int32_t stride, int32_t sets) {
  if (!arr) return ZERO_EINVAL;
  for (int32_t s = 0; s < sets; ++s)
    for (int32_t i = lo; i < hi; ++i) {
      const void* q = arr[s * stride + i];
      if (!q) return ZERO_EINVAL;
      if (!zero_detail::aligned16(q)) return ZERO_EALIGN;
    }
  return ZERO_OK;
}

int set_replicas(Args& a, const zero_plan* p, const void* const* replicas) {
  const int32_t N = p->info.n_ranks;
  int rc = check_ptr_array(replicas, 0, N, N, 1);
  if (rc) return rc;
  for (int32_t r = 0; r < N; ++r) a.rep[r] = static_cast<const uint16_t*>(replicas[r]);
  return ZERO_OK;
}

// Earlier micro-batches' fp32 accumulators (all N replicas) when n_micro > 1.
int set_accumulators(Args& a, const zero_plan* p, const float* const* accum, int32_t n_micro) {
  if (n_micro < 1) return ZERO_EINVAL;
  a.n_micro = n_micro;
  a.has_acc = n_micro > 1 ? 1 : 0;
  if (!a.has_acc) return ZERO_OK;
  const int32_t N = p->info.n_ranks;
  int rc = check_ptr_array(reinterpret_cast<const void* const*>(accum), 0, N, N, 1);
  if (rc) return rc;
  for (int32_t r = 0; r < N; ++r) a.acc[r] = accum[r];
  return ZERO_OK;
}

int window_ok(const zero_plan* p, int32_t rank_lo, int64_t wbase) {
  return wbase >= 0 && wbase <= static_cast<int64_t>(rank_lo) * p->info.shard_elems;
}

Args* new_args(const zero_plan* p) {
  Args* a = new (std::nothrow) Args;
  if (!a) return nullptr;
  std::memset(a, 0, sizeof(Args));
  a->n_ranks = p->info.n_ranks;
  a->shard = p->info.shard_elems;
  a->n_micro = 1;
  return a;
}

int seg_range(const zero_plan* p, int32_t bucket, int32_t rank_lo, int32_t rank_hi,
              std::vector<std::pair<int32_t, int32_t>>& runs) {
  const int32_t s0 = p->rank_seg0[rank_lo], s1 = p->rank_seg0[rank_hi];
  if (bucket < 0) {
    runs.emplace_back(s0, s1);
    return ZERO_OK;
  }
  // segments of one bucket inside [s0, s1) are contiguous
  int32_t b0 = -1, b1 = -1;
  for (int32_t s = s0; s < s1; ++s) {
    if (p->segs[s].bucket == bucket) {
      if (b0 < 0) b0 = s;
      b1 = s + 1;
    }
  }
  if (b0 >= 0) runs.emplace_back(b0, b1);
  return ZERO_OK;
}

// A fused step folds its finish into the pass (one launch, the last CTA does
// the bookkeeping) when the pass is one launch over at most kFoldMaxElems
// elements: short steps then pay one launch instead of two, and the rare
// overflow's re-cast by one CTA stays under about 25 MB of traffic.
constexpr int64_t kFoldMaxElems = int64_t(1) << 22;

// Fused steps over at most kShortMaxElems elements of at most kShortMaxRanks
// replicas, without micro-batch accumulators, run short_fused_kernel (one
// wave of 256-thread CTAs) instead of the pipelined pass. Measured on GB300,
// cold, CUDA events, short kernel against pipelined pass: 1M parameters at
// N = 4 16.4 against 20.9 us, N = 8 18.5 against 20.9, N = 16 22.7 against
// 24.7; the pipelined pass was faster at N = 64 (48 against 55 us for 1M)
// and from 2M elements on (2M at N = 8 a tie, 4M at N = 4 37 against 40),
// and with accumulators, so those keep it.
constexpr int64_t kShortMaxElems = int64_t(1) << 20;
constexpr int32_t kShortMaxRanks = 16;

int launch_short(const zero_plan* p, Args& a, int32_t rank_lo, int32_t rank_hi,
                 cudaStream_t st) {
  const int64_t S = p->info.shard_elems;
  const uint32_t qpo = static_cast<uint32_t>((S + 3) / 4);
  const uint32_t cpo = (qpo + kShortThreads - 1) / kShortThreads;  // CTAs per owner
  a.wend = static_cast<int64_t>(rank_hi) * S - a.wbase;
  a.bucket_elems = p->info.bucket_elems;
  const dim3 grid(cpo * static_cast<uint32_t>(rank_hi - rank_lo));
  if (grid.x >= kShortVoteUnit) return ZERO_ERANGE;  // the CTA count shares a word with the vote
  const cudaError_t e =
      p->info.grad_dtype == ZERO_BF16
          ? launch_pdl(short_fused_kernel<true>, grid, dim3(kShortThreads), 0, st, a, rank_lo,
                       cpo, qpo)
          : launch_pdl(short_fused_kernel<false>, grid, dim3(kShortThreads), 0, st, a, rank_lo,
                       cpo, qpo);
  return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}

bool fold_finish(const zero_plan* p, int32_t rank_lo, int32_t rank_hi) {
  const int32_t s0 = p->rank_seg0[rank_lo], s1 = p->rank_seg0[rank_hi];
  if (s1 <= s0 || s1 - s0 > kMaxSegs) return false;
  const int64_t elems = static_cast<int64_t>(rank_hi - rank_lo) * p->info.shard_elems;
  return elems > 0 && elems <= kFoldMaxElems;
}

}  // namespace zk

using namespace zk;

extern "C" {

ZERO_API int zero_reduce_scatter(const zero_plan* plan, int32_t bucket, int32_t rank_lo,
                                 int32_t rank_hi, const void* const* replicas,
                                 int64_t window_base, float* const* grad_shards,
                                 zero_scaler* d_scaler, uint32_t* d_bucket_flags,
                                 void* d_workspace, void* stream) {
  return zero_reduce_scatter_accum(plan, bucket, rank_lo, rank_hi, replicas, nullptr, 1,
                                   window_base, grad_shards, d_scaler, d_bucket_flags,
                                   d_workspace, stream);
}

ZERO_API int zero_reduce_scatter_accum(const zero_plan* plan, int32_t bucket, int32_t rank_lo,
                                       int32_t rank_hi, const void* const* replicas,
                                       const float* const* accum, int32_t n_micro,
                                       int64_t window_base, float* const* grad_shards,
                                       zero_scaler* d_scaler, uint32_t* d_bucket_flags,
                                       void* d_workspace, void* stream) {
  if (!ranks_ok(plan, rank_lo, rank_hi) || !d_scaler) return ZERO_EINVAL;
  if (bucket < -1 || bucket >= plan->info.n_buckets) return ZERO_EINVAL;
  if (!window_ok(plan, rank_lo, window_base)) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler) || !zero_detail::aligned16(d_bucket_flags) ||
      !zero_detail::aligned16(d_workspace))
    return ZERO_EALIGN;
  int rc = check_ptr_array(reinterpret_cast<const void* const*>(grad_shards), rank_lo, rank_hi,
                           0, 1);
  if (rc) return rc;
  Args* a = new_args(plan);
  if (!a) return ZERO_ENOMEM;
  rc = set_replicas(*a, plan, replicas);
  if (!rc) rc = set_accumulators(*a, plan, accum, n_micro);
  if (!rc) {
    for (int32_t i = rank_lo; i < rank_hi; ++i) a->ghat[i] = grad_shards[i];
    a->wbase = window_base;
    a->scaler = d_scaler;
    a->flags = d_bucket_flags;
    a->partials = static_cast<float4*>(d_workspace);
    a->mode_flags = d_workspace ? kFlagPartials : 0;
    std::vector<std::pair<int32_t, int32_t>> runs;
    seg_range(plan, bucket, rank_lo, rank_hi, runs);
    for (auto& r : runs) {
      rc = launch<kReduce>(plan, *a, r.first, r.second, static_cast<cudaStream_t>(stream));
      if (rc) break;
    }
  }
  delete a;
  return rc;
}

namespace {

// Tile records of the owners [rank_lo, rank_hi) recomputed from the reduced
// gradients (kNorm pass), into the workspace's tile records.
int recompute_records(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                      const float* const* grad_shards, zero_scaler* d_scaler, void* d_workspace,
                      cudaStream_t st) {
  int rc = check_ptr_array(reinterpret_cast<const void* const*>(grad_shards), rank_lo, rank_hi,
                           0, 1);
  if (rc) return rc;
  Args* a = new_args(plan);
  if (!a) return ZERO_ENOMEM;
  for (int32_t i = rank_lo; i < rank_hi; ++i) a->ghat[i] = const_cast<float*>(grad_shards[i]);
  a->scaler = d_scaler;
  a->partials = static_cast<float4*>(d_workspace);
  rc = launch<kNorm>(plan, *a, plan->rank_seg0[rank_lo], plan->rank_seg0[rank_hi], st);
  delete a;
  return rc;
}

}  // namespace

ZERO_API int zero_grad_norm(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                            const float* const* grad_shards, const zero_hparams* hp,
                            zero_scaler* d_scaler, void* d_workspace, void* stream) {
  if (!ranks_ok(plan, rank_lo, rank_hi) || !hp || !d_scaler || !d_workspace) return ZERO_EINVAL;
  if (!(hp->max_grad_norm > 0.0)) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler) || !zero_detail::aligned16(d_workspace))
    return ZERO_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (grad_shards) {
    const int rc = recompute_records(plan, rank_lo, rank_hi, grad_shards, d_scaler, d_workspace,
                                     st);
    if (rc) return rc;
  }
  float4* records = static_cast<float4*>(d_workspace);
  return launch_norm_finish(plan, rank_lo, rank_hi, records, 0, plan->info.n_tiles,
                            records + plan->info.n_tiles, 0, hp->max_grad_norm, d_scaler,
                            nullptr, st);
}

ZERO_API int zero_grad_norm_local(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                                  const float* const* grad_shards, const zero_hparams* hp,
                                  zero_scaler* d_scaler, void* d_workspace,
                                  zero_exchange* d_exchange, void* stream) {
  if (!ranks_ok(plan, rank_lo, rank_hi) || !hp || !d_scaler || !d_exchange) return ZERO_EINVAL;
  const bool clip = hp->max_grad_norm > 0.0;
  if (clip && !d_workspace) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler) || !zero_detail::aligned16(d_workspace) ||
      !zero_detail::aligned16(d_exchange))
    return ZERO_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (clip && grad_shards) {
    const int rc = recompute_records(plan, rank_lo, rank_hi, grad_shards, d_scaler, d_workspace,
                                     st);
    if (rc) return rc;
  }
  float4* records = static_cast<float4*>(d_workspace);
  // without clipping only the overflow word is exported (no owners)
  return launch_norm_finish(plan, clip ? rank_lo : 0, clip ? rank_hi : 0, records, 0,
                            plan->info.n_tiles, clip ? records + plan->info.n_tiles : nullptr, 1,
                            hp->max_grad_norm, d_scaler, d_exchange, st);
}

ZERO_API int zero_grad_norm_apply(const zero_plan* plan, const zero_exchange* d_exchange,
                                  const zero_hparams* hp, zero_scaler* d_scaler, void* stream) {
  if (!plan || !hp || !d_scaler || !d_exchange) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler) || !zero_detail::aligned16(d_exchange))
    return ZERO_EALIGN;
  const int clip = hp->max_grad_norm > 0.0 ? 1 : 0;
  return launch_pdl(norm_import_kernel, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream),
                    d_exchange, plan->info.n_ranks, clip, hp->max_grad_norm, d_scaler) ==
                 cudaSuccess
             ? ZERO_OK
             : ZERO_ECUDA;
}

namespace {

// Argument checks and kernel arguments shared by the step entry points.
int prepare_step(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi, float* const* master,
                 float* const* exp_avg, float* const* exp_avg_sq, int32_t n_sets,
                 const float* const* grad_shards, const void* const* replicas,
                 int64_t window_base, void* flat_params, const zero_hparams* hp,
                 zero_scaler* d_scaler, uint32_t* d_bucket_flags, bool need_moments,
                 bool need_replicas, Args** out) {
  *out = nullptr;
  if (!ranks_ok(plan, rank_lo, rank_hi) || !hp || !d_scaler || !flat_params) return ZERO_EINVAL;
  if (n_sets < 1 || n_sets > 2) return ZERO_EINVAL;
  if (hp->growth_interval < 1) return ZERO_EINVAL;
  if (!window_ok(plan, rank_lo, window_base)) return ZERO_EINVAL;
  const bool fused = grad_shards == nullptr;
  const bool clip = hp->max_grad_norm > 0.0;
  if (fused && (clip || n_sets != 2)) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler) || !zero_detail::aligned16(d_bucket_flags) ||
      !zero_detail::aligned16(flat_params))
    return ZERO_EALIGN;
  const int32_t N = plan->info.n_ranks;
  int rc;
  if ((rc = check_ptr_array(reinterpret_cast<const void* const*>(master), rank_lo, rank_hi, N,
                            n_sets)))
    return rc;
  if (need_moments) {
    if ((rc = check_ptr_array(reinterpret_cast<const void* const*>(exp_avg), rank_lo, rank_hi, N,
                              n_sets)))
      return rc;
    if ((rc = check_ptr_array(reinterpret_cast<const void* const*>(exp_avg_sq), rank_lo,
                              rank_hi, N, n_sets)))
      return rc;
    if (!fused && (rc = check_ptr_array(reinterpret_cast<const void* const*>(grad_shards),
                                        rank_lo, rank_hi, 0, 1)))
      return rc;
  }
  Args* a = new_args(plan);
  if (!a) return ZERO_ENOMEM;
  if (fused && need_replicas && (rc = set_replicas(*a, plan, replicas))) {
    delete a;
    return rc;
  }
  for (int32_t s = 0; s < n_sets; ++s)
    for (int32_t i = rank_lo; i < rank_hi; ++i) {
      a->master[s][i] = master[s * N + i];
      if (need_moments) {
        a->mom[s][i] = exp_avg[s * N + i];
        a->var[s][i] = exp_avg_sq[s * N + i];
      }
    }
  if (!fused && need_moments)
    for (int32_t i = rank_lo; i < rank_hi; ++i) a->ghat[i] = const_cast<float*>(grad_shards[i]);
  a->n_sets = n_sets;
  a->flat = static_cast<uint16_t*>(flat_params);
  a->wbase = window_base;
  a->scaler = d_scaler;
  a->flags = d_bucket_flags;
  a->mode_flags = (!fused && clip) ? kFlagClip : 0;
  fill_constants(*a, hp);
  *out = a;
  return ZERO_OK;
}

}  // namespace

ZERO_API int zero_step_update(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                              float* const* master, float* const* exp_avg,
                              float* const* exp_avg_sq, int32_t n_sets,
                              const float* const* grad_shards, const void* const* replicas,
                              int64_t window_base, void* flat_params, const zero_hparams* hp,
                              zero_scaler* d_scaler, uint32_t* d_bucket_flags, void* stream) {
  return zero_step_update_accum(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets,
                                grad_shards, replicas, nullptr, 1, window_base, flat_params, hp,
                                d_scaler, d_bucket_flags, stream);
}

ZERO_API int zero_step_update_accum(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                                    float* const* master, float* const* exp_avg,
                                    float* const* exp_avg_sq, int32_t n_sets,
                                    const float* const* grad_shards, const void* const* replicas,
                                    const float* const* accum, int32_t n_micro,
                                    int64_t window_base, void* flat_params,
                                    const zero_hparams* hp, zero_scaler* d_scaler,
                                    uint32_t* d_bucket_flags, void* stream) {
  Args* a = nullptr;
  int rc = prepare_step(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets, grad_shards,
                        replicas, window_base, flat_params, hp, d_scaler, d_bucket_flags, true,
                        true, &a);
  if (rc) return rc;
  if (grad_shards == nullptr && (rc = set_accumulators(*a, plan, accum, n_micro))) {
    delete a;
    return rc;
  }
  const int32_t s0 = plan->rank_seg0[rank_lo], s1 = plan->rank_seg0[rank_hi];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = grad_shards == nullptr ? launch<kFused>(plan, *a, s0, s1, st)
                              : launch<kUpdate>(plan, *a, s0, s1, st);
  delete a;
  return rc;
}

ZERO_API int zero_step_finish(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                              float* const* master, int32_t n_sets,
                              const float* const* grad_shards, int64_t window_base,
                              void* flat_params, const zero_hparams* hp, zero_scaler* d_scaler,
                              void* stream) {
  Args* a = nullptr;
  int rc = prepare_step(plan, rank_lo, rank_hi, master, nullptr, nullptr, n_sets, grad_shards,
                        nullptr, window_base, flat_params, hp, d_scaler, nullptr, false, false,
                        &a);
  if (rc) return rc;
  const bool fused = grad_shards == nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int32_t s0 = plan->rank_seg0[rank_lo], s1 = plan->rank_seg0[rank_hi];
  if (fused && s0 < s1) {
    // one launch: re-cast the parameters from the kept master set if the
    // step overflowed, and the bookkeeping
    a->mode_flags = kFlagIfPending | kFlagUseScalerSet | kFlagFinish;
    a->bk_dynamic = hp->dynamic_scale;
    a->bk_growth = hp->growth_interval;
    a->bk_flip = 1;
    rc = launch<kCast>(plan, *a, s0, s1, st);
    delete a;
    return rc;
  }
  delete a;
  if (launch_pdl(scaler_finish_kernel, dim3(1), dim3(32), 0, st, d_scaler, hp->beta1, hp->beta2,
                 hp->dynamic_scale, hp->growth_interval, (fused || n_sets == 2) ? 1 : 0) !=
      cudaSuccess)
    return ZERO_ECUDA;
  return ZERO_OK;
}

ZERO_API int zero_selftest_wait_timeout(zero_scaler* d_scaler, int64_t limit_ns, void* stream) {
  if (!d_scaler || limit_ns < 1000 || limit_ns > 10000000000ll) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler)) return ZERO_EALIGN;
  return launch_plain(wait_timeout_probe_kernel, dim3(1), dim3(32), 0,
                      static_cast<cudaStream_t>(stream), d_scaler,
                      static_cast<uint64_t>(limit_ns)) == cudaSuccess
             ? ZERO_OK
             : ZERO_ECUDA;
}

#ifdef ZERO_CHECKED
int zg_collect_checks(unsigned long long* count, unsigned long long* first);  // gather.cu (C linkage)
#endif

ZERO_API int zero_checked_status(int64_t* violations, int64_t* first, void* stream) {
  if (!violations || !first) return ZERO_EINVAL;
  *violations = 0;
  *first = 0;
#ifdef ZERO_CHECKED
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ZERO_ECUDA;
  unsigned long long count = 0, code = 0;
  if (collect_checks(&count, &code) != 0 || zg_collect_checks(&count, &code) != 0)
    return ZERO_ECUDA;
  *violations = static_cast<int64_t>(count);
  *first = static_cast<int64_t>(code);
  return ZERO_OK;
#else
  (void)stream;
  return ZERO_ESTATE;
#endif
}

ZERO_API int zero_selftest_check(void* stream) {
#ifdef ZERO_CHECKED
  return launch_plain(zk::check_selftest_kernel, dim3(1), dim3(1), 0,
                      static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ZERO_OK
             : ZERO_ECUDA;
#else
  (void)stream;
  return ZERO_ESTATE;
#endif
}

ZERO_API int zero_step(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                       float* const* master, float* const* exp_avg, float* const* exp_avg_sq,
                       int32_t n_sets, const float* const* grad_shards,
                       const void* const* replicas, int64_t window_base, void* flat_params,
                       const zero_hparams* hp, zero_scaler* d_scaler,
                       uint32_t* d_bucket_flags, void* stream) {
  return zero_step_accum(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets,
                         grad_shards, replicas, nullptr, 1, window_base, flat_params, hp,
                         d_scaler, d_bucket_flags, stream);
}

ZERO_API int zero_step_accum(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                             float* const* master, float* const* exp_avg,
                             float* const* exp_avg_sq, int32_t n_sets,
                             const float* const* grad_shards, const void* const* replicas,
                             const float* const* accum, int32_t n_micro, int64_t window_base,
                             void* flat_params, const zero_hparams* hp, zero_scaler* d_scaler,
                             uint32_t* d_bucket_flags, void* stream) {
  if (grad_shards == nullptr && ranks_ok(plan, rank_lo, rank_hi) &&
      fold_finish(plan, rank_lo, rank_hi)) {
    Args* a = nullptr;
    int rc = prepare_step(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets, nullptr,
                          replicas, window_base, flat_params, hp, d_scaler, d_bucket_flags, true,
                          true, &a);
    if (rc) return rc;
    if ((rc = set_accumulators(*a, plan, accum, n_micro))) {
      delete a;
      return rc;
    }
    a->mode_flags |= kFlagFinish;
    a->bk_dynamic = hp->dynamic_scale;
    a->bk_growth = hp->growth_interval;
    a->bk_flip = 1;
    const int64_t elems = static_cast<int64_t>(rank_hi - rank_lo) * plan->info.shard_elems;
    const bool short_step = elems <= kShortMaxElems && plan->info.n_ranks <= kShortMaxRanks &&
                            !a->has_acc;
    rc = short_step
             ? launch_short(plan, *a, rank_lo, rank_hi, static_cast<cudaStream_t>(stream))
             : launch<kFused>(plan, *a, plan->rank_seg0[rank_lo], plan->rank_seg0[rank_hi],
                              static_cast<cudaStream_t>(stream));
    delete a;
    return rc;
  }
  int rc = zero_step_update_accum(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets,
                                  grad_shards, replicas, accum, n_micro, window_base,
                                  flat_params, hp, d_scaler, d_bucket_flags, stream);
  if (rc) return rc;
  return zero_step_finish(plan, rank_lo, rank_hi, master, n_sets, grad_shards, window_base,
                          flat_params, hp, d_scaler, stream);
}

ZERO_API int zero_cast_params(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                              const float* const* master, void* flat_params,
                              int64_t window_base, void* stream) {
  if (!ranks_ok(plan, rank_lo, rank_hi) || !flat_params) return ZERO_EINVAL;
  if (!window_ok(plan, rank_lo, window_base)) return ZERO_EINVAL;
  if (!zero_detail::aligned16(flat_params)) return ZERO_EALIGN;
  int rc = check_ptr_array(reinterpret_cast<const void* const*>(master), rank_lo, rank_hi, 0, 1);
  if (rc) return rc;
  Args* a = new_args(plan);
  if (!a) return ZERO_ENOMEM;
  for (int32_t i = rank_lo; i < rank_hi; ++i) a->master[0][i] = const_cast<float*>(master[i]);
  a->n_sets = 1;
  a->flat = static_cast<uint16_t*>(flat_params);
  a->wbase = window_base;
  a->mode_flags = 0;
  // kCast without kFlagIfPending/kFlagUseScalerSet never touches the scaler
  zero_scaler* dummy = nullptr;
  a->scaler = dummy;
  const int32_t s0 = plan->rank_seg0[rank_lo], s1 = plan->rank_seg0[rank_hi];
  rc = launch<kCast>(plan, *a, s0, s1, static_cast<cudaStream_t>(stream));
  delete a;
  return rc;
}

}  // extern "C"

// ------------------------------------------- micro-batch accumulation --
//
// "How far does splitting the batch get you?", "What does gradient
// accumulation actually buy?": run k micro-batches, accumulate each rank's
// gradients locally in fp32, reduce once. accumulate_kernel adds one
// micro-batch's 16-bit gradients of every replica into the fp32
// accumulators (first micro-batch: the widened values themselves); the last
// micro-batch is added inside the reduce pass (bulk_kernel<.., kAcc>), so
// the accumulators are never written for it.

struct AccArgs {
  const uint16_t* micro[ZERO_MAX_RANKS];
  float* acc[ZERO_MAX_RANKS];
  int64_t off, len;  // window elements [off, off + len) of every replica
  int32_t n_ranks, first;
  int32_t vec;       // 1: off is on the 4-element grid (8- and 16-byte vectors)
  int32_t pad;
};

// Quads (4 elements) in flight per thread: eight 8-byte loads (and, after
// the first micro-batch, eight 16-byte accumulator loads) are issued before
// the first store, which the write-heavy first pass needs to keep HBM busy.
constexpr int kAccQuads = 8;
constexpr int kAccThreads = 256;

template <bool kBf16>
__device__ __forceinline__ float4 widen4(const uint2& w) {
  return make_float4(widen<kBf16>(w.x & 0xFFFFu), widen<kBf16>(w.x >> 16),
                     widen<kBf16>(w.y & 0xFFFFu), widen<kBf16>(w.y >> 16));
}

// grid: x strides over one replica's window, y = replica
template <bool kBf16>
__global__ void __launch_bounds__(kAccThreads)
    accumulate_kernel(const __grid_constant__ AccArgs a) {
  pdl_begin();
  const int r = blockIdx.y;
  const uint16_t* src = a.micro[r] + a.off;
  float* dst = a.acc[r] + a.off;
  const int64_t nq = a.vec ? (a.len >> 2) : 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint2* src4 = reinterpret_cast<const uint2*>(src);
  float4* dst4 = reinterpret_cast<float4*>(dst);
  for (int64_t q0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q0 < nq;
       q0 += stride * kAccQuads) {
    uint2 w[kAccQuads];
    float4 y[kAccQuads];
#pragma unroll
    for (int u = 0; u < kAccQuads; ++u) {
      const int64_t q = q0 + u * stride;
      if (q < nq && ZCHECK(a.off + 4 * q + 4 <= a.off + a.len, kSiteAccumulate, q))
        w[u] = __ldcs(src4 + q);
    }
    if (!a.first) {
#pragma unroll
      for (int u = 0; u < kAccQuads; ++u) {
        const int64_t q = q0 + u * stride;
        if (q < nq) y[u] = __ldcs(dst4 + q);
      }
    }
#pragma unroll
    for (int u = 0; u < kAccQuads; ++u) {
      const int64_t q = q0 + u * stride;
      if (q < nq) {
        float4 x = widen4<kBf16>(w[u]);
        if (!a.first) {
          x.x = __fadd_rn(y[u].x, x.x);
          x.y = __fadd_rn(y[u].y, x.y);
          x.z = __fadd_rn(y[u].z, x.z);
          x.w = __fadd_rn(y[u].w, x.w);
        }
        __stcs(dst4 + q, x);
      }
    }
  }
  // ragged tail of the window (or all of it when off is off the grid)
  for (int64_t j = (nq << 2) + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       j < a.len; j += stride) {
    const float x = widen<kBf16>(src[j]);
    dst[j] = a.first ? x : __fadd_rn(dst[j], x);
  }
}

extern "C" ZERO_API int zero_accumulate(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                                        const void* const* micro, float* const* accum,
                                        int64_t window_base, int32_t first, void* stream) {
  if (!ranks_ok(plan, rank_lo, rank_hi)) return ZERO_EINVAL;
  if (!window_ok(plan, rank_lo, window_base)) return ZERO_EINVAL;
  const int32_t N = plan->info.n_ranks;
  int rc = check_ptr_array(micro, 0, N, N, 1);
  if (rc) return rc;
  if ((rc = check_ptr_array(reinterpret_cast<const void* const*>(accum), 0, N, N, 1))) return rc;
  AccArgs* a = new (std::nothrow) AccArgs;
  if (!a) return ZERO_ENOMEM;
  std::memset(a, 0, sizeof(AccArgs));
  for (int32_t r = 0; r < N; ++r) {
    a->micro[r] = static_cast<const uint16_t*>(micro[r]);
    a->acc[r] = accum[r];
  }
  const int64_t S = plan->info.shard_elems;
  a->off = static_cast<int64_t>(rank_lo) * S - window_base;
  a->len = static_cast<int64_t>(rank_hi - rank_lo) * S;
  a->n_ranks = N;
  a->first = first ? 1 : 0;
  // the vector body needs the window offset on the 4-element grid of both
  // arrays (8-byte source, 16-byte accumulator vectors); otherwise the whole
  // window takes the element-wise loop
  a->vec = (a->off & 3) == 0 ? 1 : 0;
  const int sms = device_sms();
  if (sms <= 0) {
    delete a;
    return ZERO_ECUDA;
  }
  rc = ZERO_OK;
  if (a->len > 0) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // about 8 CTAs per SM in all, split evenly over the replicas
    const dim3 grid(static_cast<unsigned>(std::max(1, sms * 8 / N)), static_cast<unsigned>(N));
    if (plan->info.grad_dtype == ZERO_BF16)
      rc = launch_pdl(accumulate_kernel<true>, grid, dim3(kAccThreads), 0, st, *a) == cudaSuccess
               ? ZERO_OK
               : ZERO_ECUDA;
    else
      rc = launch_pdl(accumulate_kernel<false>, grid, dim3(kAccThreads), 0, st, *a) ==
                   cudaSuccess
               ? ZERO_OK
               : ZERO_ECUDA;
  }
  delete a;
  return rc;
}

// ------------------------------------------------- ring reduce-scatter --
//
// "How far does splitting the batch get you?", "Why does the all-reduce not
// get more expensive with more ranks?": with the N ranks in N processes (one
// gradient replica each), chunk i -- owner i's slice -- walks the ring. Rank
// i+1 starts it with its own values, every rank on the way adds its own and
// passes the partial on, and after N - 1 hops rank i adds its own last and
// holds the full sum: the ring order i+1, ..., N-1, 0, ..., i of the one-GPU
// reduce. The partials stay fp32 between hops ("What does gradient
// accumulation actually buy?": an fp32 reduce-scatter). ring_hop_kernel is
// one rank's part of one hop: out = widen(own chunk) on the first hop,
// recv + widen(own chunk) on the middle ones, and on the last hop (the
// rank's own slice) the unscaled gradient (recv + widen(own)) * fp32(1/(S_l N))
// with the non-finite vote.

struct RingArgs {
  const uint16_t* own;   // this rank's gradient at the chunk's first element
  const float* recv;     // partial from the previous rank (NULL on the first hop)
  float* out;            // partial for the next rank, or the reduced gradient
  zero_scaler* scaler;
  uint32_t* flags;
  int64_t n;             // elements of the chunk (S)
  int64_t chunk0;        // flat index of the chunk's first element
  int64_t bucket_elems;  // 0 = one bucket
  int32_t n_ranks;
  int32_t final_hop;
};

constexpr int kRingThreads = 256;

template <bool kBf16>
__device__ __forceinline__ float ring_elem(const RingArgs& a, int64_t k, float inv, bool& bad) {
  float x = widen<kBf16>(__ldcs(reinterpret_cast<const unsigned short*>(a.own) + k));
  if (a.recv) x = __fadd_rn(__ldcs(a.recv + k), x);
  if (a.final_hop) {
    x = __fmul_rn(x, inv);
    if (nonfinite(x)) {
      bad = true;
      if (a.flags) atomicOr(&a.flags[a.bucket_elems ? (a.chunk0 + k) / a.bucket_elems : 0], 1u);
    }
  }
  return x;
}

// Grid-stride over quads of 4 elements: the partials move as 16-byte vectors
// (recv and out are 16-byte aligned), the 16-bit values as 2-byte loads (a
// chunk of an odd-sized shard starts at any element).
template <bool kBf16>
__global__ void __launch_bounds__(kRingThreads) ring_hop_kernel(const __grid_constant__ RingArgs a) {
  pdl_begin();
  float inv = 1.0f;
  if (a.final_hop) {
    const double denom =
        __dmul_rn(static_cast<double>(a.scaler->scale), static_cast<double>(a.n_ranks));
    inv = __double2float_rn(__ddiv_rn(1.0, denom));
  }
  bool bad = false;
  const int64_t nq = (a.n + 3) >> 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < nq;
       q += stride) {
    const int64_t k0 = q << 2;
    if (k0 + 4 <= a.n) {
      float y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = ring_elem<kBf16>(a, k0 + e, inv, bad);
      __stcs(reinterpret_cast<float4*>(a.out + k0), make_float4(y[0], y[1], y[2], y[3]));
    } else {
      for (int64_t k = k0; k < a.n; ++k) a.out[k] = ring_elem<kBf16>(a, k, inv, bad);
    }
  }
  if (a.final_hop && __any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0)
    atomicOr(&a.scaler->pending, 1u);
}

extern "C" ZERO_API int zero_ring_hop(const zero_plan* plan, int32_t rank, int32_t hop,
                                      const void* grad, const float* recv, float* out,
                                      zero_scaler* d_scaler, uint32_t* d_bucket_flags,
                                      void* stream) {
  if (!plan || !grad || !out || !d_scaler) return ZERO_EINVAL;
  const int32_t N = plan->info.n_ranks;
  if (rank < 0 || rank >= N || hop < 1 || hop > N) return ZERO_EINVAL;
  if ((hop == 1) != (recv == nullptr)) return ZERO_EINVAL;
  if (!zero_detail::aligned16(grad) || !zero_detail::aligned16(recv) ||
      !zero_detail::aligned16(out) || !zero_detail::aligned16(d_scaler) ||
      !zero_detail::aligned16(d_bucket_flags))
    return ZERO_EALIGN;
  const int64_t S = plan->info.shard_elems;
  const int32_t c = ((rank - hop) % N + N) % N;
  RingArgs a{};
  a.own = static_cast<const uint16_t*>(grad) + static_cast<int64_t>(c) * S;
  a.recv = recv;
  a.out = out;
  a.scaler = d_scaler;
  a.flags = d_bucket_flags;
  a.n = S;
  a.chunk0 = static_cast<int64_t>(c) * S;
  a.bucket_elems = plan->info.bucket_elems;
  a.n_ranks = N;
  a.final_hop = hop == N ? 1 : 0;
  if (S == 0) return ZERO_OK;
  const int sms = device_sms();
  if (sms <= 0) return ZERO_ECUDA;
  const int64_t want = (S + 4 * kRingThreads - 1) / (4 * kRingThreads);
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      plan->info.grad_dtype == ZERO_BF16
          ? launch_pdl(ring_hop_kernel<true>, dim3(grid), dim3(kRingThreads), 0, st, a)
          : launch_pdl(ring_hop_kernel<false>, dim3(grid), dim3(kRingThreads), 0, st, a);
  return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}

// ------------------------------------------------ no-allocation norm entry --
//
// zero_grad_norm_noalloc: the same norm and clip coefficient as
// zero_grad_norm, for callers that cannot hand the library a device
// workspace. Its tile partials live in a fixed device array in this file.

namespace zk {

constexpr int64_t kNoallocTiles = ZERO_NOALLOC_MAX_TILES;
constexpr int64_t kNoallocBlocks = static_cast<int64_t>(ZERO_MAX_RANKS) * kOwnerBlocks;

// One 16-byte norm record per tile, then the finish kernels' share records
// (kOwnerBlocks per owner), 8 MiB + 16 KiB. Every GPU that loads this
// library holds this array until the process exits. All calls share it, and
// each call overwrites the records of exactly the tiles and shares it later
// reads, so nothing has to be cleared between calls. Calls that overlap on
// the GPU (different streams, or different host threads without ordering)
// race on it.
static __device__ __align__(256) float4 g_noalloc_partials[kNoallocTiles + kNoallocBlocks];

// Device address of g_noalloc_partials per device ordinal, resolved once per
// device with that device current. In host code the array's name only stands
// for the symbol; it is never a device address. The address belongs to the
// device's context at the time of the first call: a process that destroys
// that context (cudaDeviceReset) must not call the entry point afterwards.
constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
float4* g_noalloc_ptr[kNoallocMaxDevices] = {};

int noalloc_scratch(float4** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ECUDA;
  if (dev < 0 || dev >= kNoallocMaxDevices) return ZERO_ERANGE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return ZERO_ECUDA;
    g_noalloc_ptr[dev] = static_cast<float4*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return ZERO_OK;
}

}  // namespace zk

extern "C" ZERO_API int zero_grad_norm_noalloc(const zero_plan* plan, int32_t rank_lo,
                                               int32_t rank_hi, const float* const* grad_shards,
                                               const zero_hparams* hp, zero_scaler* d_scaler,
                                               void* stream) {
  if (!ranks_ok(plan, rank_lo, rank_hi) || !hp || !d_scaler || !grad_shards) return ZERO_EINVAL;
  if (!(hp->max_grad_norm > 0.0)) return ZERO_EINVAL;
  if (!zero_detail::aligned16(d_scaler)) return ZERO_EALIGN;
  int rc = check_ptr_array(reinterpret_cast<const void* const*>(grad_shards), rank_lo, rank_hi,
                           0, 1);
  if (rc) return rc;
  const int32_t s0 = plan->rank_seg0[rank_lo], s1 = plan->rank_seg0[rank_hi];
  const int64_t t0 = owner_tile0(plan, rank_lo);
  const int64_t t1 = owner_tile0(plan, rank_hi);
  if (t1 - t0 > kNoallocTiles) return ZERO_ERANGE;
  float4* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;

  Args* a = new_args(plan);
  if (!a) return ZERO_ENOMEM;
  for (int32_t i = rank_lo; i < rank_hi; ++i) a->ghat[i] = const_cast<float*>(grad_shards[i]);
  a->scaler = d_scaler;
  a->partials = scratch;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid_cap = grid_size<kNorm, true>();
  if (grid_cap <= 0) rc = ZERO_ECUDA;
  // tiles are numbered from t0 so that the records start at the array's
  // base; segments go kMaxSegs to a launch
  for (int32_t b0 = s0; !rc && b0 < s1; b0 += kMaxSegs) {
    const int32_t b1 = std::min(s1, b0 + kMaxSegs);
    int64_t tiles = 0;
    for (int32_t s = b0; s < b1; ++s) {
      Seg& d = a->segs[s - b0];
      d.lo = plan->segs[s].lo;
      d.hi = plan->segs[s].hi;
      d.rank = plan->segs[s].rank;
      d.bucket = plan->segs[s].bucket;
      d.tile_local0 = tiles;
      d.tile_global0 = plan->seg_tile0[s] - t0;
      tiles += plan->seg_tiles[s];
    }
    a->n_segs = b1 - b0;
    a->n_tiles = tiles;
    // extents for the checked build: window indices of this launch (the
    // window is the whole flat buffer) and the records the array holds
    a->wend = plan->segs[b1 - 1].hi;
    a->n_records = kNoallocTiles;
    if (tiles == 0) continue;
    const int grid = static_cast<int>(std::min<int64_t>(tiles, grid_cap));
    // the kNorm body only reads fp32 gradients, so one instantiation serves
    // both 16-bit formats
    if (launch_pdl(step_kernel<kNorm, true>, dim3(grid), dim3(kThreads), 0, st, *a) !=
        cudaSuccess)
      rc = ZERO_ECUDA;
  }
  delete a;
  if (rc) return rc;
  return launch_norm_finish(plan, rank_lo, rank_hi, scratch, t0, kNoallocTiles,
                            scratch + kNoallocTiles, 0, hp->max_grad_norm, d_scaler, nullptr,
                            st);
}
