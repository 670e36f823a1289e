/*
 * synth.h -- seeded, counter-based synthetic input generator.
 *
 * This module produces the INPUTS of a sharded mixed-precision AdamW step:
 * per-rank gradient replicas and the initial fp32 master weights. It holds
 * none of the step's arithmetic (no reduction, no optimizer, no cast to a
 * half format): every function returns an fp32 value, and each consumer
 * (the CUDA harness kernels and the CPU checker) converts to bf16/fp16 with
 * its own code.
 *
 * Both consumers compile this one header, so the values are bit-identical on
 * the host and on the GPU:
 *   - integer hashing only, then a few fp32 multiplies/adds that are written
 *     with ZS_MUL / ZS_ADD so no compiler may fuse them into an FMA
 *     (host code must also be built with -ffp-contract=off);
 *   - no transcendental functions.
 *
 * Generator definition (a convention of this project, not of the pages):
 *   key(seed, tag, step, rank) = mix64(seed * G ^ (tag << 56 | step << 32 | rank))
 *   u64(seed, tag, step, rank, e) = mix64(key + (e + 1) * G)
 * i.e. element e reads output e+1 of a SplitMix64 sequence started at `key`,
 * where mix64 is the SplitMix64 output function and G = 0x9E3779B97F4A7C15
 * (Steele, Lea and Flood, "Fast Splittable Pseudorandom Number Generators",
 * OOPSLA 2014).
 *
 * Approximate normal: Irwin-Hall sum of the four 16-bit lanes of one u64,
 *   s = l0 + l1 + l2 + l3,  z = (float)(s - 131070) * C0,
 * C0 = fp32(sqrt(3) / 65536), so z has mean 0 and unit variance and is
 * bounded by |z| <= 131070 * C0 ~= 3.464.
 */
#ifndef ZSYNTH_H
#define ZSYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define ZS_FN static __host__ __device__ __forceinline__
#else
#define ZS_FN static inline
#endif

#if defined(__CUDA_ARCH__)
#define ZS_MUL(a, b) __fmul_rn((a), (b))
#define ZS_ADD(a, b) __fadd_rn((a), (b))
#else
#define ZS_MUL(a, b) ((float)(a) * (float)(b))
#define ZS_ADD(a, b) ((float)(a) + (float)(b))
#endif

#define ZS_GOLDEN 0x9E3779B97F4A7C15ull

/* tags: disjoint random streams */
#define ZS_TAG_GRAD    1u
#define ZS_TAG_OUTLIER 2u
#define ZS_TAG_BIAS    3u
#define ZS_TAG_MASTER  4u

/* fp32(sqrt(3)/65536), exact hex of the rounded value */
#define ZS_NORMAL_C0 0x1.bb67aep-16f

/* SplitMix64 output function (variant 13 of Stafford's mixers, as used by
 * SplitMix64). */
ZS_FN uint64_t zs_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

ZS_FN uint64_t zs_key(uint64_t seed, uint32_t tag, uint32_t step, uint32_t rank) {
  uint64_t word = ((uint64_t)(tag & 0xFFu) << 56) |
                  ((uint64_t)(step & 0xFFFFFFu) << 32) | (uint64_t)rank;
  return zs_mix64((seed * ZS_GOLDEN) ^ word);
}

ZS_FN uint64_t zs_u64(uint64_t key, uint64_t elem) {
  return zs_mix64(key + (elem + 1u) * ZS_GOLDEN);
}

/* Irwin-Hall(4) approximate standard normal from one 64-bit hash. */
ZS_FN float zs_normal(uint64_t h) {
  int32_t s = (int32_t)(h & 0xFFFFu) + (int32_t)((h >> 16) & 0xFFFFu) +
              (int32_t)((h >> 32) & 0xFFFFu) + (int32_t)(h >> 48);
  return ZS_MUL((float)(s - 131070), ZS_NORMAL_C0);
}

/* Gradient recipe for one rank's replica. */
typedef struct zs_grad_spec {
  uint64_t seed;
  float sigma;        /* standard deviation of the base normal */
  float bias_sigma;   /* >0: add one per-(step, rank) offset b ~ N(0, bias_sigma) */
  float loss_scale;   /* multiplies the value last (a power of two in practice) */
  int32_t outliers;   /* 1: with probability 1049/2^20 (~0.1%) multiply by 100 */
  int64_t psi;        /* elements >= psi are padding and are exactly 0 */
} zs_grad_spec;

/* fp32 value of gradient element `elem` of rank `rank` at step `step`
 * (before the cast to the gradient's 16-bit format). */
ZS_FN float zs_grad_value(const zs_grad_spec* g, uint32_t step, uint32_t rank,
                          int64_t elem) {
  if (elem >= g->psi) return 0.0f;
  float x = ZS_MUL(zs_normal(zs_u64(zs_key(g->seed, ZS_TAG_GRAD, step, rank),
                                    (uint64_t)elem)),
                   g->sigma);
  if (g->bias_sigma > 0.0f) {
    float b = ZS_MUL(zs_normal(zs_u64(zs_key(g->seed, ZS_TAG_BIAS, step, rank), 0u)),
                     g->bias_sigma);
    x = ZS_ADD(x, b);
  }
  if (g->outliers) {
    uint64_t o = zs_u64(zs_key(g->seed, ZS_TAG_OUTLIER, step, rank), (uint64_t)elem);
    if ((o & 0xFFFFFu) < 1049u) x = ZS_MUL(x, 100.0f);
  }
  return ZS_MUL(x, g->loss_scale);
}

/* The same values with the per-(step, rank) keys and bias formed once:
 * zs_grad_stream_value(zs_grad_stream_make(g, step, rank), e) equals
 * zs_grad_value(g, step, rank, e) for every e. */
typedef struct zs_grad_stream {
  uint64_t key_grad, key_outlier;
  float sigma, bias, loss_scale;
  int32_t has_bias, outliers;
  int64_t psi;
} zs_grad_stream;

ZS_FN zs_grad_stream zs_grad_stream_make(const zs_grad_spec* g, uint32_t step, uint32_t rank) {
  zs_grad_stream s;
  s.key_grad = zs_key(g->seed, ZS_TAG_GRAD, step, rank);
  s.key_outlier = zs_key(g->seed, ZS_TAG_OUTLIER, step, rank);
  s.sigma = g->sigma;
  s.has_bias = g->bias_sigma > 0.0f;
  s.bias = s.has_bias
               ? ZS_MUL(zs_normal(zs_u64(zs_key(g->seed, ZS_TAG_BIAS, step, rank), 0u)),
                        g->bias_sigma)
               : 0.0f;
  s.loss_scale = g->loss_scale;
  s.outliers = g->outliers;
  s.psi = g->psi;
  return s;
}

ZS_FN float zs_grad_stream_value(const zs_grad_stream* s, int64_t elem) {
  if (elem >= s->psi) return 0.0f;
  float x = ZS_MUL(zs_normal(zs_u64(s->key_grad, (uint64_t)elem)), s->sigma);
  if (s->has_bias) x = ZS_ADD(x, s->bias);
  if (s->outliers) {
    uint64_t o = zs_u64(s->key_outlier, (uint64_t)elem);
    if ((o & 0xFFFFFu) < 1049u) x = ZS_MUL(x, 100.0f);
  }
  return ZS_MUL(x, s->loss_scale);
}

/* Initial fp32 master weight of flat element `elem`: U(-0.05, 0.05) from a
 * 23-bit uniform integer u: ((u + 0.5) * 2^-23) * 0.1 - 0.05 (u + 0.5 and the
 * power-of-two scaling are exact). Padding elements (elem >= psi) start at 0. */
ZS_FN float zs_master_value(uint64_t seed, int64_t psi, int64_t elem) {
  if (elem >= psi) return 0.0f;
  uint64_t h = zs_u64(zs_key(seed, ZS_TAG_MASTER, 0u, 0u), (uint64_t)elem);
  float u = ZS_MUL(ZS_ADD((float)(uint32_t)(h >> 41), 0.5f), 0x1p-23f);
  return ZS_ADD(ZS_MUL(u, 0.1f), -0.05f);
}

#endif /* ZSYNTH_H */
