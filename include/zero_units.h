/*
 * zero_units.h -- stage-3 FSDP units in libzero: the per-unit layout of the
 * sharded parameters and the just-in-time all-gather of a unit.
 *
 * What it computes.
 *   Layout: the model's tensors are grouped into units (typically one
 *   transformer block each, plus a root unit for embeddings and head). Unit
 *   u's tensors, in list order, are flattened into one vector of psi_u
 *   elements, padded with zeros to psi_pad_u, a multiple of N * align_elems,
 *   and cut into N equal slices of S_u = psi_pad_u / N elements; rank r holds
 *   slice r. A rank's shard buffer is its slices of units 0, 1, ..., U-1 back
 *   to back: unit u's slice starts at shard_offset_u = S_0 + ... + S_{u-1}.
 *   All-gather of unit u: full_u[r * S_u + j] = shard_r[shard_offset_u + j]
 *   for every rank r and j < S_u -- every rank rebuilds the unit's full
 *   parameters before the unit runs. The inverse (shard) writes a full unit
 *   back into the N slices.
 *   Accounting per rank (K = 12, 16 bytes per held element): persistent
 *   bytes; the peak with one gathered unit, with two adjacent ones (the next
 *   unit prefetched while one computes) and in the backward pass (the unit's
 *   parameters plus its full gradient before the reduce-scatter); wire volume
 *   3 psi elements per step (all-gather forward, all-gather backward,
 *   reduce-scatter). Activations are not counted: they need a model.
 *
 * Sources (page title, section):
 *   "Training models too big for one GPU: ZeRO & FSDP": "FSDP: the same idea,
 *     one unit at a time" (units, per-unit flatten and shard, gather / run /
 *     free, peak = shards + one or two gathered units);
 *   "ZeRO Stage 3 Math": "Just-in-time all-gather: how the weights reappear",
 *     "Peak transient memory" (peak = persistent 16 psi / N + one layer's full
 *     parameters + activations; unit granularity trades peak memory against
 *     collective size);
 *   "Stop Replicating What You Can Shard: ZeRO and FSDP": "FSDP: the same
 *     idea, layer-native" (3 psi = forward gather + backward gather +
 *     reduce-scatter; root unit for embeddings and head);
 *   "How far does splitting the batch get you?": "What does stage 3 actually
 *     do per layer?", "What does each stage cost on the wire?".
 *
 * One GPU holds all N ranks: the N shard buffers are resident HBM buffers
 * and the all-gather is one copy kernel over every rank's slice.
 *
 * Conventions are those of zero.h: int status returns (ZERO_OK or a negative
 * zero_status), caller-owned device memory, asynchronous calls on the given
 * stream, 16-byte aligned device pointers, immutable plans, int64 element
 * indices. Elements are 16-bit (bf16 or fp16; the copy does not look at
 * them).
 */
#ifndef ZERO_UNITS_H
#define ZERO_UNITS_H

#include "zero.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest alignment grain (elements) a unit plan accepts. */
#define ZERO_UNIT_MAX_ALIGN 4096

typedef struct zero_unit_plan zero_unit_plan;

/* One unit of a plan (56 bytes). */
typedef struct zero_unit {
  int64_t psi;           /* parameters of the unit's tensors */
  int64_t pad;           /* zeros appended: psi_pad is a multiple of N * align_elems */
  int64_t psi_pad;       /* elements of the gathered unit */
  int64_t shard_elems;   /* S_u = psi_pad / N, elements of the unit each rank holds */
  int64_t shard_offset;  /* start of the unit's slice in every rank's shard buffer */
  int64_t flat_offset;   /* start of the unit in the concatenation of all padded units */
  int32_t n_tensors;     /* tensors of the unit */
  int32_t first_slot;    /* first entry of the unit in the slot list (zero_unit_plan_tensors) */
} zero_unit;

/* Plan totals and accounting (120 bytes). Bytes are per rank; GB = 1e9. */
typedef struct zero_unit_plan_info {
  int64_t psi;               /* all parameters */
  int64_t psi_pad;           /* sum of the units' psi_pad */
  int64_t shard_elems;       /* elements each rank holds: sum of the units' shard_elems */
  int64_t max_unit_psi_pad;  /* largest gathered unit */
  int32_t n_units, n_ranks, n_tensors, align_elems;
  double persistent_bytes;   /* 16 * shard_elems: 2 weight + 2 gradient + 12 optimizer */
  double peak_one_bytes;     /* persistent + 2 * max psi_pad_u (one gathered unit) */
  double peak_two_bytes;     /* persistent + 2 * max (psi_pad_u + psi_pad_{u+1}) (prefetch) */
  double peak_backward_bytes;/* persistent + 4 * max psi_pad_u (parameters + full gradient) */
  double max_unit_fraction;  /* max psi_u / psi */
  double comm_elems;         /* 3 * psi_pad per step */
  double comm_bytes;         /* 2 * comm_elems (16-bit elements) */
  double ring_bytes;         /* per rank per step over a ring: 3 * (N - 1) * shard_elems * 2 */
  int32_t n_gathers;         /* 2 * n_units all-gathers per step (forward and backward) */
  int32_t reserved;
} zero_unit_plan_info;

/* Build a unit plan. numels[k] (>= 0) is tensor k's size; unit_of_tensor[k]
 * in [0, n_units) names its unit; units are numbered in forward order and
 * each needs at least one tensor. n_ranks in [1, ZERO_MAX_RANKS];
 * align_elems in [1, ZERO_UNIT_MAX_ALIGN] (1: pad each unit to a multiple of
 * N only; 8: every slice starts on a 16-byte boundary, the fast copy).
 * Host only. Returns ZERO_EINVAL on bad arguments, ZERO_ERANGE for more than
 * ZERO_MAX_RANKS ranks or an alignment above ZERO_UNIT_MAX_ALIGN, ZERO_ENOMEM. */
ZERO_API int zero_unit_plan_create(const int64_t* numels, int32_t n_tensors,
                                   const int32_t* unit_of_tensor, int32_t n_units,
                                   int32_t n_ranks, int32_t align_elems, zero_unit_plan** out);
ZERO_API void zero_unit_plan_destroy(zero_unit_plan* plan);
ZERO_API int zero_unit_plan_get_info(const zero_unit_plan* plan, zero_unit_plan_info* out);
/* out: capacity >= n_units entries (ZERO_ERANGE otherwise). */
ZERO_API int zero_unit_plan_units(const zero_unit_plan* plan, zero_unit* out, int32_t capacity);
/* slot_tensor (may be NULL): tensor ids unit by unit, in list order within a
 * unit (unit u's are entries first_slot .. first_slot + n_tensors - 1).
 * tensor_offset (may be NULL): tensor k's offset inside its gathered unit.
 * Both need capacity >= n_tensors entries (ZERO_ERANGE otherwise). */
ZERO_API int zero_unit_plan_tensors(const zero_unit_plan* plan, int32_t* slot_tensor,
                                    int64_t* tensor_offset, int32_t capacity);

/* Sharding strategies ("Training models too big for one GPU: ZeRO & FSDP",
 * "FSDP: the same idea, one unit at a time": FULL_SHARD is stage 3,
 * SHARD_GRAD_OP is close to stage 2, NO_SHARD is ordinary DDP, HYBRID_SHARD
 * shards inside a node and replicates across nodes; "How far does splitting
 * the batch get you?", "What does each stage cost on the wire?": Llama 3 kept
 * the gathered parameters from the forward pass for the backward pass --
 * stage 3's memory for the forward, stage 2's traffic). */
typedef enum zero_strategy {
  ZERO_FULL_SHARD = 0,
  ZERO_SHARD_GRAD_OP = 1,
  ZERO_NO_SHARD = 2,
  ZERO_HYBRID_SHARD = 3,
  ZERO_NO_RESHARD_AFTER_FORWARD = 4
} zero_strategy;

/* Per-rank cost of one step under a strategy (56 bytes). */
typedef struct zero_strategy_cost {
  double persistent_bytes;  /* model states held between steps */
  double peak_bytes;        /* persistent + the largest gathered-parameter transient */
  double comm_elems;        /* elements sent per step, counted as the pages count them */
  double comm_elems_inter;  /* of which between shard groups (HYBRID_SHARD) */
  double ring_bytes;        /* bytes sent per step when every collective is a ring */
  double ring_bytes_inter;  /* of which between shard groups */
  int32_t shard_ranks;      /* ranks one copy of the states is sharded over */
  int32_t gathers_per_unit; /* all-gathers of each unit per step */
} zero_strategy_cost;

/* Cost of a step under `strategy` for the plan's layout. The plan's n_ranks
 * is the shard group g; n_replicas R >= 1 is the number of groups holding
 * replicas of the same shards (HYBRID_SHARD; R must be 1 for every other
 * strategy). With the plan's psi, psi_pad P, held elements S and largest
 * unit U, 16-bit parameters and gradients, K = 12:
 *   FULL_SHARD     persistent 16S, peak +2U, 3P elements, ring 3(g-1)S x 2 bytes,
 *                  2 gathers per unit;
 *   SHARD_GRAD_OP  persistent 2P + 14S, no transient, 2P elements,
 *                  ring 2(g-1)S x 2, 1 gather;
 *   NO_SHARD       persistent 16 psi, 2 psi elements, ring 2(g-1)/g x 2 psi, 0 gathers;
 *   HYBRID_SHARD   FULL_SHARD inside the group plus, for R > 1, an all-reduce
 *                  of each rank's S reduced gradient elements over the R groups:
 *                  2S elements and 2(R-1)/R x 2S bytes between groups;
 *   NO_RESHARD_AFTER_FORWARD  persistent 16S, peak +2P (every unit gathered in
 *                  the forward pass is held until its backward), 2P elements,
 *                  ring 2(g-1)S x 2, 1 gather.
 * Host only. Returns ZERO_EINVAL for a NULL argument, an unknown strategy or
 * a bad n_replicas. */
ZERO_API int zero_unit_plan_strategy_cost(const zero_unit_plan* plan, int32_t strategy,
                                          int32_t n_replicas, zero_strategy_cost* out);

/* All-gather of units [unit_lo, unit_hi) (a forward or backward prefetch
 * window), one kernel launch per 256 slices (N slices per unit). A window
 * larger than half of L2 is written with evict-first stores, a smaller one
 * normally (the unit's layer reads it next).
 *   unit_buffers[u - unit_lo][r * S_u + j] = shards[r][shard_offset_u + j].
 * shards: n_ranks device pointers, rank r's shard buffer of shard_elems
 *   16-bit elements; read only. The copy may read the rest of the 16-byte
 *   block that holds a buffer's last element, so allocate each shard buffer
 *   to a multiple of 16 bytes (any cudaMalloc'd buffer is).
 * unit_buffers: unit_hi - unit_lo device pointers, unit u's buffer of
 *   psi_pad_u 16-bit elements; written entirely (its padding elements receive
 *   the shards' padding elements).
 * Buffers must not overlap. Asynchronous on stream. Returns ZERO_EINVAL (bad
 * plan, range or NULL pointer), ZERO_EALIGN (pointer not 16-byte aligned),
 * ZERO_ECUDA (launch failure). */
ZERO_API int zero_gather_units(const zero_unit_plan* plan, int32_t unit_lo, int32_t unit_hi,
                               const void* const* shards, void* const* unit_buffers,
                               void* stream);

/* The inverse: shards[r][shard_offset_u + j] = unit_buffers[u - unit_lo][r * S_u + j]
 * for units [unit_lo, unit_hi) (placing a full unit, e.g. initial weights,
 * into the N slices). Same pointer rules with the roles swapped; the rest of
 * every shard buffer is left as it was. */
ZERO_API int zero_shard_units(const zero_unit_plan* plan, int32_t unit_lo, int32_t unit_hi,
                              const void* const* unit_buffers, void* const* shards,
                              void* stream);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_UNITS_H */
