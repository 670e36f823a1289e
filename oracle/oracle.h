/*
 * oracle.h -- plain, slow CPU checker for the sharded mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library; the product path never does.
 * It shares no code with the CUDA library: its only shared dependency is the
 * seeded input generator (synth.h), which holds none of the step's arithmetic.
 *
 * Pages cited (title, then section):
 *   [ZF]  "Training models too big for one GPU: ZeRO & FSDP"
 *   [SR]  "Stop Replicating What You Can Shard: ZeRO and FSDP"
 *   [TM]  "The redundancy hiding in data parallelism" (transformer math: ZeRO)
 *   [Z3]  "ZeRO Stage 3 Math"
 *   [SB]  "How far does splitting the batch get you?" (interrogating
 *         parallelism, part 2: splitting the batch)
 *
 * Floating point: the pages fix fp32 for the master weights, Adam moments and
 * the gradient reduction, and bf16/fp16 for gradients and working weights, so
 * the checker computes in those precisions, one IEEE round-to-nearest-even
 * operation per C statement (built with -ffp-contract=off, no fast-math).
 * Quantities the pages leave to accounting (bills, norms) are fp64.
 *
 * Parity status per function is listed beside each declaration; every
 * function here is pinned by a CPU test (closed forms, printed worked
 * examples, invariants, exhaustive comparison, brute force).
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>
#include "synth.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- plan ---- */

typedef struct orc_segment {
  int64_t lo, hi;      /* flat element range [lo, hi) */
  int32_t rank;        /* owner: rank whose 1/N slice contains the range */
  int32_t bucket;      /* bucket containing the range */
} orc_segment;

typedef struct orc_plan {
  int64_t psi;         /* total parameters (sum of tensor sizes) */
  int64_t pad;         /* zeros appended so that psi_pad is a multiple of n_ranks */
  int64_t psi_pad;
  int64_t shard;       /* psi_pad / n_ranks: elements each rank owns */
  int64_t bucket_elems;/* bucket size in elements, 0 = one bucket */
  int32_t n_ranks;
  int32_t n_buckets;
  int32_t n_segments;
  int32_t reserved;
  /* per-device model-state bytes, K = 12 (mixed-precision Adam) */
  double bill_ddp, bill_z1, bill_z2, bill_z3;
  /* ring all-reduce of 2*psi bytes of 16-bit gradients */
  double ring_bytes_per_rank; /* 2(d-1)M/d */
  double ring_hops;           /* 2(d-1) */
  /* communication volume per step in elements */
  double comm_ddp, comm_z1, comm_z2, comm_z3;
} orc_plan;

/* Flatten a tensor list, pad to a multiple of N, shard, bucket.
 * [ZF] "FSDP: the same idea, one unit at a time" (parameters flattened and
 * sharded); [ZF] "ZeRO stages 1, 2 and 3" (GPU i updates its 1/N slice);
 * [SB] "How does the collective hide behind the backward pass?" (buckets).
 * offsets: n_tensors entries or NULL. segs: capacity seg_cap or NULL.
 * Returns 0; -1 on invalid arguments; -2 if seg_cap is too small
 * (out->n_segments then holds the count needed). */
int orc_plan_make(const int64_t* numels, int32_t n_tensors, int32_t n_ranks,
                  int64_t bucket_elems, orc_plan* out, int64_t* offsets,
                  orc_segment* segs, int32_t seg_cap);

/* Model-state bytes per device for psi parameters, K = 12.
 * [ZF] "The memory bill: 16 bytes per parameter", "ZeRO stages 1, 2 and 3";
 * [TM] "The per-stage memory formula and a worked example";
 * [Z3] "Stage 3: divide everything by N". out[0..3] = DDP, Z1, Z2, Z3. */
void orc_bills(double psi, int32_t n_ranks, double out[4]);

/* Bytes each rank sends in a ring all-reduce of m_bytes over d ranks:
 * 2(d-1)M/d. [SB] "Why does the all-reduce not get more expensive with more
 * ranks?"; [ZF] "Data parallelism and the all-reduce". */
double orc_ring_bytes(double m_bytes, int32_t d);

/* --------------------------------------------------------------- casts ---- */
/* IEEE 754 binary16 and bfloat16 (fp32 with the mantissa cut to 7 bits),
 * round to nearest, ties to even; overflow to infinity; subnormals kept.
 * [ZF] "How a computer stores real numbers" (format table) and
 * "Mixed-precision training" (the fp32 master is rounded to half). */
uint16_t orc_f32_to_f16(float x);
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float x);
float orc_bf16_to_f32(uint16_t h);
void orc_cast_array(const float* in, uint16_t* out, int64_t n, int32_t is_bf16);
void orc_widen_array(const uint16_t* in, float* out, int64_t n, int32_t is_bf16);

/* --------------------------------------------------- step building blocks ---- */

typedef struct orc_hparams {
  double lr, beta1, beta2, eps, weight_decay;
  double max_grad_norm;     /* <= 0: no clipping */
  int32_t dynamic_scale;    /* 1: halve on overflow, double after growth_interval good steps */
  int32_t growth_interval;
} orc_hparams;

typedef struct orc_scaler {
  float scale;              /* loss scale S */
  int32_t good_steps;       /* consecutive good steps since the last change */
  int32_t t;                /* applied optimizer steps */
  int32_t overflow;         /* 1 if the last step was skipped */
  double norm_sq, norm;     /* last global gradient norm (clip configs) */
  float clip_coef;          /* coefficient applied in the last step (1 = none) */
  int32_t reserved;
} orc_scaler;

typedef struct orc_adam_scalars {
  float b1, omb1, b2, omb2; /* beta1, 1-beta1, beta2, 1-beta2 rounded from fp64 */
  float bc1, bc2;           /* 1 - beta^t rounded from fp64, beta^t by t products */
  float lr, decay, eps;     /* decay = 1 - lr*weight_decay rounded from fp64 */
} orc_adam_scalars;

/* Sum of the N replicas' values of one element in ring order for owner i:
 * ranks i+1, i+2, ..., N-1, 0, ..., i, fp32 accumulation.
 * [SB] "Why does the all-reduce not get more expensive with more ranks?"
 * (a chunk walks the ring, summed hop by hop, and is complete at rank i after
 * d-1 hops); [SB] "What does gradient accumulation actually buy?" (fp32
 * reduce-scatter). vals[r] is rank r's value widened to fp32. */
float orc_ring_sum(const float* vals, int32_t n_ranks, int32_t owner);

/* fp32(1 / (S * N)): divide by the loss scale ([ZF] "Mixed-precision
 * training") and average over the N replicas ([ZF] "Data parallelism and the
 * all-reduce"). */
float orc_unscale_factor(float scale, int32_t n_ranks);

/* fp32(1 / (S * N * k)) for a step of k micro-batches per rank: the average
 * over every micro-batch of every rank ([SB] "What does gradient
 * accumulation actually buy?": run k micro-batches, accumulate, reduce
 * once). k = 1 is orc_unscale_factor. */
float orc_unscale_factor_k(float scale, int32_t n_ranks, int32_t n_micro);

/* FP32 gradient accumulation over micro-batches ([SB] "What does gradient
 * accumulation actually buy?": the accumulator has to be fp32):
 * acc[k] = first ? widen(micro[k]) : acc[k] + widen(micro[k]). */
void orc_accumulate(const uint16_t* micro, float* acc, int64_t n, int32_t is_bf16,
                    int32_t first);

/* Adam scalars for optimizer step t (t >= 1). [ZF] "Adam, and why it's
 * expensive" (bias corrections 1 - beta^t). */
orc_adam_scalars orc_adam_scalars_make(const orc_hparams* hp, int32_t t);

/* One AdamW update of one element ([ZF] "Adam, and why it's expensive":
 * moments, bias correction, eps outside the square root; decoupled weight
 * decay as named there): m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g);
 * mh = m/bc1; vh = v/bc2; u = mh/(sqrt(vh)+eps); theta = theta*decay;
 * theta = theta - lr*u. */
void orc_adamw_elem(float* theta, float* m, float* v, float g, const orc_adam_scalars* a);

/* Clip coefficient from the global sum of squares: c = max_norm/(sqrt(nsq)+1e-6),
 * applied (rounded to fp32) only when c < 1. Returns 1 if it applies. */
int32_t orc_clip_coef(double norm_sq, double max_norm, float* coef, double* norm);

/* Loss-scale bookkeeping after a step ([ZF] "Mixed-precision training": pick
 * S dynamically, skip a step on overflow). Overflow: no state change, t kept,
 * S halved (floor 1) when dynamic, good_steps reset. Otherwise t += 1,
 * good_steps += 1 and S doubles after growth_interval good steps when
 * dynamic. */
void orc_scaler_finish(orc_scaler* s, const orc_hparams* hp, int32_t overflow);

/* ------------------------------------------------------ whole-step drivers ---- */

/* One full step on explicit host arrays, for owners [rank_lo, rank_hi).
 * replicas[r][j - wbase] is rank r's 16-bit gradient of flat element j;
 * master/m/v/params/ghat are indexed by j - wbase as well.
 * Processes flat elements [rank_lo*S, rank_hi*S) in ascending order:
 *   reduce (ring order, fp32) -> unscale -> non-finite flag per bucket ->
 *   if any flag: skip (nothing written, scaler updated) ->
 *   optional clip (global L2 norm over the processed elements) ->
 *   AdamW on the fp32 master/m/v -> cast to the 16-bit working copy.
 * bucket_flags (n_buckets, may be NULL) are OR-ed. ghat (may be NULL)
 * receives the unscaled, unclipped reduced gradient.
 * Norm: squares summed in fp64 in ascending element order within fixed
 * chunks of 2^20 elements (counted from rank_lo*S), chunk sums added in
 * ascending order. Returns 0, or -1 on bad arguments. */
int orc_step_arrays(const orc_plan* p, int32_t rank_lo, int32_t rank_hi, int32_t is_bf16,
                    const uint16_t* const* replicas, int64_t wbase, float* master,
                    float* m, float* v, uint16_t* params, float* ghat,
                    uint32_t* bucket_flags, const orc_hparams* hp, orc_scaler* sc);

/* orc_step_arrays for a step of n_micro micro-batches: replicas[r][j - wbase]
 * is rank r's fp32 accumulated gradient (sum of its micro-batches, from
 * orc_accumulate); the unscale is orc_unscale_factor_k; is_bf16 selects the
 * working copy's format. */
int orc_step_arrays_f32(const orc_plan* p, int32_t rank_lo, int32_t rank_hi, int32_t is_bf16,
                        const float* const* replicas, int32_t n_micro, int64_t wbase,
                        float* master, float* m, float* v, uint16_t* params, float* ghat,
                        uint32_t* bucket_flags, const orc_hparams* hp, orc_scaler* sc);

/* Input recipe for the generator-driven driver: replica r's element j at
 * step s is cast16(zs_grad_value(spec with loss_scale = current S, s, r, j)),
 * except one optional injected 16-bit pattern. */
typedef struct orc_gen {
  zs_grad_spec spec;
  int32_t is_bf16;
  int32_t inject_step;      /* < 0: no injection */
  int32_t inject_rank;
  uint32_t inject_bits;     /* 16-bit pattern written at (inject_step, inject_rank, inject_elem) */
  int64_t inject_elem;
} orc_gen;

/* One full step at any size without storing replicas: regenerates every
 * replica value on the fly (n_threads workers over the fixed 2^20-element
 * chunks, results combined in chunk order, so the output does not depend on
 * n_threads). Applies the update only to the sampled flat elements
 * elems[0..n_elems) (ascending, inside [rank_lo*S, rank_hi*S)), whose states
 * master/m/v/params are given as arrays of length n_elems. Global results
 * (flags, overflow, norm) cover all processed elements. */
int orc_gen_step(const orc_plan* p, int32_t rank_lo, int32_t rank_hi, const orc_gen* g,
                 uint32_t step, int32_t n_threads, const int64_t* elems, int64_t n_elems,
                 float* master, float* m, float* v, uint16_t* params,
                 uint32_t* bucket_flags, const orc_hparams* hp, orc_scaler* sc);

/* Reduced, unscaled gradient at sampled elements, regenerated (no clip). */
int orc_gen_ghat(const orc_plan* p, const orc_gen* g, uint32_t step, float scale,
                 const int64_t* elems, int64_t n_elems, float* ghat);

/* -------------------------------------------------- stage-3 FSDP units ---- */

typedef struct orc_unit {
  int64_t psi;          /* parameters of the unit's tensors */
  int64_t pad;          /* zeros appended so that psi_pad is a multiple of N * align */
  int64_t psi_pad;
  int64_t shard;        /* psi_pad / N: elements of the unit each rank holds */
  int64_t shard_offset; /* where the unit's slice starts in every rank's shard buffer */
  int64_t flat_offset;  /* where the padded unit starts in the concatenation of all units */
  int32_t n_tensors;    /* tensors of the unit */
  int32_t first_slot;   /* its first entry in slot_tensor */
} orc_unit;

typedef struct orc_unit_plan {
  int64_t psi;          /* all parameters */
  int64_t psi_pad;      /* sum of the units' psi_pad */
  int64_t shard;        /* elements each rank holds: sum of the units' shard */
  int64_t max_unit_psi_pad;
  int32_t n_units, n_ranks, n_tensors, align_elems;
  /* per-rank bytes, K = 12 (16 bytes per held element) */
  double persistent_bytes;     /* 16 * shard */
  double peak_one_bytes;       /* persistent + one gathered unit (2 bytes per element) */
  double peak_two_bytes;       /* persistent + two adjacent gathered units (prefetch) */
  double peak_backward_bytes;  /* persistent + one unit's parameters and full gradient */
  double max_unit_fraction;    /* largest unit's psi / psi */
  /* wire per rank per step */
  double comm_elems;           /* 3 psi_pad: two all-gathers and one reduce-scatter */
  double comm_bytes;           /* 2 bytes per element of comm_elems */
  double ring_bytes;           /* ring collectives: 3 (N-1) shard elements of 2 bytes */
  int32_t n_gathers;           /* 2 per unit: forward and backward */
  int32_t reserved;
} orc_unit_plan;

/* Per-unit flatten, pad and shard of a tensor list for stage 3.
 * [ZF] "FSDP: the same idea, one unit at a time" (each unit's parameters are
 * flattened and sharded; peak = sharded states + one or two gathered units);
 * [Z3] "Just-in-time all-gather: how the weights reappear" (units of one
 * layer, gathered before the layer's forward and again before its backward)
 * and "Peak transient memory" (peak = persistent 16 psi / N + one layer's
 * full parameters + activations; activations need a model and are left out);
 * [SB] "What does each stage cost on the wire?" (stage 3 moves 3 psi).
 * unit_of_tensor[k] in [0, n_units) names tensor k's unit; a unit's tensors
 * keep their list order and every unit needs at least one. Unit u is padded
 * with zeros to a multiple of N * align_elems and rank r holds its elements
 * [r S_u, (r+1) S_u); a rank's shard buffer is its slices of units 0..U-1 in
 * order. Units are numbered in forward order; the two-unit peak takes the
 * largest pair of adjacent units (the next unit prefetched while one runs).
 * units: n_units entries or NULL; slot_tensor: n_tensors entries or NULL
 * (tensor ids unit by unit); tensor_offset: n_tensors entries or NULL
 * (offset of tensor k inside its gathered unit). Returns 0 or -1. */
int orc_unit_plan_make(const int64_t* numels, int32_t n_tensors, const int32_t* unit_of_tensor,
                       int32_t n_units, int32_t n_ranks, int32_t align_elems,
                       orc_unit_plan* out, orc_unit* units, int32_t* slot_tensor,
                       int64_t* tensor_offset);

/* The all-gather of one unit ([Z3] "Just-in-time all-gather": every rank
 * reconstructs the layer's full parameters): full[r S_u + j] =
 * shards[r][shard_offset_u + j] for every rank r and j < S_u. */
void orc_gather_unit(const orc_unit* u, int32_t n_ranks, const uint16_t* const* shards,
                     uint16_t* full);

/* The inverse: rank r keeps full[r S_u .. (r+1) S_u) at shard_offset_u of its
 * shard buffer ([ZF] "FSDP: the same idea, one unit at a time": the unit's
 * flattened parameters are sharded across the GPUs). */
void orc_shard_unit(const orc_unit* u, int32_t n_ranks, const uint16_t* full,
                    uint16_t* const* shards);

/* Sharding strategies: [ZF] "FSDP: the same idea, one unit at a time" (FULL_SHARD
 * is stage 3, SHARD_GRAD_OP is close to stage 2, NO_SHARD is ordinary DDP,
 * HYBRID_SHARD shards inside a node and replicates across nodes); [SB] "What
 * does each stage cost on the wire?" (Llama 3: states and gradients sharded,
 * parameters not resharded after the forward pass -- stage 3's memory,
 * stage 2's traffic). */
enum {
  ORC_FULL_SHARD = 0,
  ORC_SHARD_GRAD_OP = 1,
  ORC_NO_SHARD = 2,
  ORC_HYBRID_SHARD = 3,
  ORC_NO_RESHARD_AFTER_FORWARD = 4
};

typedef struct orc_strategy_cost {
  double persistent_bytes;  /* model states held between steps, per rank */
  double peak_bytes;        /* persistent + the largest gathered-parameter transient */
  double comm_elems;        /* elements per rank per step, the pages' counting */
  double comm_elems_inter;  /* of which between shard groups (HYBRID_SHARD) */
  double ring_bytes;        /* bytes each rank sends per step over rings */
  double ring_bytes_inter;  /* of which between shard groups */
  int32_t shard_ranks;      /* ranks one copy of the states is sharded over */
  int32_t gathers_per_unit; /* all-gathers of each unit per step */
} orc_strategy_cost;

/* Per-rank cost of one step under a strategy, for a unit plan whose n_ranks
 * is the shard group g; n_replicas R is the number of shard groups (HYBRID_SHARD
 * only; every other strategy takes R = 1). With psi, psi_pad P, held elements
 * S and largest unit U of the plan, 16-bit parameters and gradients and
 * K = 12:
 *   FULL_SHARD     16S; +2U; 3P elements; ring 3 (g-1) S x 2 bytes; 2 gathers
 *   SHARD_GRAD_OP  2P + 14S; no transient; 2P; ring 2 (g-1) S x 2; 1 gather
 *   NO_SHARD       16 psi; 2 psi; ring all-reduce 2 (g-1)/g x 2 psi; 0 gathers
 *   HYBRID_SHARD   FULL_SHARD inside the group, plus an all-reduce of each
 *                  rank's S gradient elements over the R groups: 2S elements
 *                  and 2 (R-1)/R x 2S bytes between groups (none when R = 1)
 *   NO_RESHARD_AFTER_FORWARD  16S; +2P (every unit gathered in the forward
 *                  pass is kept for its backward); 2P; ring 2 (g-1) S x 2;
 *                  1 gather
 * Returns 0, or -1 for an unknown strategy or R < 1 (R != 1 outside
 * HYBRID_SHARD). */
int orc_strategy_cost_make(const orc_unit_plan* p, int32_t strategy, int32_t n_replicas,
                           orc_strategy_cost* out);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_ORACLE_H */
