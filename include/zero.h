/*
 * zero.h -- C ABI of libzero: the per-shard ZeRO step of mixed-precision
 * AdamW on one GB300 (sm_103a).
 *
 * What the library computes. N data-parallel ranks hold N gradient replicas
 * of one flattened parameter vector. Rank i owns the 1/N slice
 * [i*S, (i+1)*S) of the padded flat vector and, for every element j it owns:
 *   1. reduce-scatter: g = (sum of the N replicas' values in ring order
 *      i+1, i+2, ..., N-1, 0, ..., i, accumulated in fp32) * fp32(1/(S_l*N)),
 *      S_l the loss scale; a non-finite g raises the bucket's flag and the
 *      step's overflow word;
 *   2. optional global-norm clip: g *= c when c = max_norm/(||g||_2 + 1e-6) < 1;
 *   3. AdamW on the fp32 master/m/v shard (decoupled weight decay);
 *   4. cast of the updated master to the bf16/fp16 working copy, written into
 *      its slot of the gathered flat parameter buffer;
 * and a step that saw any non-finite g is skipped as a whole (no state
 * changes, t kept, dynamic loss scale halved).
 *
 * Sources (page title, section):
 *   "Training models too big for one GPU: ZeRO & FSDP": "Adam, and why it's
 *     expensive" (update equations), "Mixed-precision training" (fp32 master,
 *     loss scaling, skip on overflow), "Data parallelism and the all-reduce"
 *     (averaging; reduce-scatter leaves GPU i with the sum of chunk i),
 *     "ZeRO stages 1, 2 and 3" (each GPU updates its own 1/N slice, then the
 *     updated weights are gathered), "FSDP: the same idea, one unit at a time"
 *     (parameters flattened and sharded), "The memory bill: 16 bytes per
 *     parameter" (K = 12 optimizer bytes);
 *   "How far does splitting the batch get you?": "Why does the all-reduce not
 *     get more expensive with more ranks?" (ring reduce-scatter, 2(d-1)M/d
 *     bytes), "How does the collective hide behind the backward pass?"
 *     (gradient buckets), "What does gradient accumulation actually buy?"
 *     (fp32 reduce-scatter), "What does each stage cost on the wire?";
 *   "ZeRO Stage 3 Math": "Stage 3: divide everything by N";
 *   "Stop Replicating What You Can Shard: ZeRO and FSDP": "The three stages
 *     of ZeRO" (per-stage memory).
 * The global-norm clip is not on the pages; its convention is stated at
 * zero_grad_norm.
 *
 * One GPU holds all N ranks: the N replicas are N resident HBM buffers, a
 * single launch covers every rank's slice, and the all-gather is implicit
 * (rank i writes its slot of the one flat parameter buffer).
 *
 * Conventions.
 *   - Every function returns an int status: ZERO_OK (0) or a negative
 *     zero_status. No call aborts or throws.
 *   - The library allocates no device memory. Device buffers (replicas,
 *     optimizer shards, reduced-gradient shards, flat parameters, the
 *     scaler, bucket flags, workspace) are owned by the caller.
 *   - Device calls are asynchronous on the given cudaStream_t (passed as
 *     void*; NULL = legacy default stream) and never synchronize the host.
 *     Decisions (skip, clip coefficient, loss scale) stay on the device in
 *     zero_scaler.
 *   - Every device pointer must be 16-byte aligned (ZERO_EALIGN otherwise).
 *   - Plans are immutable after creation and the library keeps no global
 *     state (the one exception is the fixed device array behind
 *     zero_grad_norm_noalloc), so concurrent calls on different streams and
 *     buffers are safe. Calls that share a scaler or buffers must be ordered
 *     by the caller.
 *   - Element indices are int64 (N * psi may exceed 2^31).
 *   - Kernels are launched with programmatic stream serialization: each
 *     waits for the previous grid in the stream before touching memory and
 *     lets the next one be scheduled early. A caller kernel launched after a
 *     library call behaves as with any launch, unless the caller gives it
 *     that launch attribute too; then it must wait (griddepcontrol.wait)
 *     before reading the library's results.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ZERO_API __attribute__((visibility("default")))
#else
#define ZERO_API
#endif

/* Largest number of simulated data-parallel ranks one plan may have. */
#define ZERO_MAX_RANKS 64

/* Elements per norm tile: the squared-gradient partial sums are formed over
 * tiles of this many elements inside each segment (see zero_grad_norm). */
#define ZERO_TILE_ELEMS 4096

typedef enum zero_status {
  ZERO_OK = 0,
  ZERO_EINVAL = -1,   /* invalid argument (NULL pointer, bad range, bad size) */
  ZERO_EALIGN = -2,   /* a device pointer is not 16-byte aligned */
  ZERO_ERANGE = -3,   /* a size exceeds a library limit (e.g. ZERO_MAX_RANKS) */
  ZERO_ECUDA = -4,    /* a CUDA launch or runtime call failed */
  ZERO_ENOMEM = -5,   /* host allocation failed */
  ZERO_ESTATE = -6    /* call order violated (e.g. clip without zero_grad_norm) */
} zero_status;

typedef enum zero_dtype { ZERO_BF16 = 0, ZERO_FP16 = 1 } zero_dtype;

/* ------------------------------------------------------------------ plan -- */

typedef struct zero_plan zero_plan; /* opaque, host memory, immutable */

/* Flat range [lo, hi) of one bucket owned by one rank. Segments are ordered
 * by lo, i.e. bucket-major with ranks ascending. */
typedef struct zero_segment {
  int64_t lo, hi;
  int32_t rank;
  int32_t bucket;
} zero_segment;

/* Bucket k: flat range [lo, hi) and its segments
 * [seg_first, seg_first + seg_count) of the plan's segment list. */
typedef struct zero_bucket {
  int64_t lo, hi;
  int32_t seg_first, seg_count;
} zero_bucket;

typedef struct zero_plan_info {
  int64_t psi;            /* parameters: sum of the tensor sizes */
  int64_t pad;            /* zeros appended: (N - psi mod N) mod N */
  int64_t psi_pad;        /* psi + pad, a multiple of N */
  int64_t shard_elems;    /* S = psi_pad / N: elements each rank owns */
  int64_t bucket_elems;   /* bucket size in elements (0 = one bucket) */
  int64_t n_tiles;        /* norm tiles over all segments */
  int32_t n_ranks;        /* N */
  int32_t n_buckets;
  int32_t n_segments;
  int32_t n_tensors;
  int32_t grad_dtype;     /* zero_dtype of gradients and working parameters */
  int32_t reserved;
  /* Per-device model-state bytes of mixed-precision Adam (K = 12), from the
   * unpadded psi: DDP 16 psi, ZeRO-1 4 psi + 12 psi/N, ZeRO-2 2 psi + 14 psi/N,
   * ZeRO-3 16 psi/N ("ZeRO stages 1, 2 and 3"; "ZeRO Stage 3 Math",
   * "Stage 3: divide everything by N"). */
  double bill_ddp, bill_z1, bill_z2, bill_z3;
  /* Ring all-reduce of the 2 psi bytes of 16-bit gradients: bytes each rank
   * sends, 2(N-1)M/N, and sequential hops 2(N-1) ("Why does the all-reduce
   * not get more expensive with more ranks?"). */
  double ring_bytes_per_rank, ring_hops;
  /* Communication per step in elements: 2 psi (DDP, ZeRO-1, ZeRO-2) and
   * 3 psi (ZeRO-3) ("What does each stage cost on the wire?"). */
  double comm_elems_ddp, comm_elems_z1, comm_elems_z2, comm_elems_z3;
  /* HBM bytes per parameter of one whole-group step on one GPU:
   * fused (no clip) 2N + 26; two-pass (clip) 2N + 34. */
  double step_bytes_fused, step_bytes_two_pass;
} zero_plan_info;

/* Build a plan: flatten the tensor list (tensor k starts at the sum of the
 * previous sizes, no per-tensor alignment), pad to a multiple of n_ranks,
 * give rank i the slice [i*S, (i+1)*S), cut the padded buffer into buckets
 * of bucket_elems elements (0 = one bucket) and each bucket at the owners'
 * slice boundaries into segments.
 *   numels:       n_tensors sizes (>= 0), host memory, read only.
 *   n_ranks:      1 .. ZERO_MAX_RANKS (ZERO_ERANGE above).
 *   grad_dtype:   format of gradient replicas and working parameters.
 *   out:          receives a plan owned by the caller (zero_plan_destroy).
 * Errors: ZERO_EINVAL (NULL out, negative size or bucket, n_ranks < 1),
 * ZERO_ERANGE, ZERO_ENOMEM. */
ZERO_API int zero_plan_create(const int64_t* numels, int32_t n_tensors, int32_t n_ranks,
                              int64_t bucket_elems, zero_dtype grad_dtype, zero_plan** out);
ZERO_API void zero_plan_destroy(zero_plan* plan);
/* Copy the plan's sizes, bills and wire figures to *out (host memory).
 * zero_plan_info_get is the same call under a second name. */
ZERO_API int zero_plan_get_info(const zero_plan* plan, zero_plan_info* out);
ZERO_API int zero_plan_info_get(const zero_plan* plan, zero_plan_info* out);
/* out[k] = flat offset of tensor k (n_tensors entries). */
ZERO_API int zero_plan_tensor_offsets(const zero_plan* plan, int64_t* out);
/* Copies min(cap, n_segments) segments; ZERO_ERANGE if cap < n_segments. */
ZERO_API int zero_plan_segments(const zero_plan* plan, zero_segment* out, int32_t cap);
/* [lo, hi) of bucket k. */
ZERO_API int zero_plan_bucket_range(const zero_plan* plan, int32_t bucket, int64_t* lo,
                                    int64_t* hi);
/* All buckets and segments at once ("How far does splitting the batch get
 * you?", "How does the collective hide behind the backward pass?": the
 * gradients are reduced bucket by bucket). out: n_buckets entries, segs:
 * n_segments entries (host memory); either may be NULL. */
ZERO_API int zero_plan_buckets(const zero_plan* plan, zero_bucket* out, zero_segment* segs);
/* Device workspace bytes of a step. two_pass != 0 (a clipped step): the norm
 * records zero_reduce_scatter, zero_grad_norm and zero_grad_norm_local use,
 * one 16-byte record per tile plus ZERO_NORM_OWNER_BLOCKS per rank.
 * two_pass == 0: 0, the fused step uses no workspace. 0 for a NULL plan. */
#define ZERO_NORM_OWNER_BLOCKS 16
ZERO_API size_t zero_workspace_bytes(const zero_plan* plan, int32_t two_pass);

/* ---------------------------------------------------- hyperparameters -- */

typedef struct zero_hparams {
  double lr, beta1, beta2, eps, weight_decay;
  double max_grad_norm;     /* > 0: clip to this global L2 norm; <= 0: no clip */
  int32_t dynamic_scale;    /* 1: halve the loss scale on overflow (floor 1) and
                               double it after growth_interval good steps */
  int32_t growth_interval;  /* >= 1 */
  double init_scale;        /* initial loss scale (1 for bf16 without scaling) */
} zero_hparams;

/* Device-resident step state. Create it with zero_scaler_init on the host
 * and copy it to device memory (sizeof(zero_scaler) bytes, 16-byte aligned);
 * after that only the library's kernels write it. The host may read it back
 * at any time after synchronizing the stream. */
typedef struct zero_scaler {
  float scale;          /* loss scale S_l used to unscale this step's gradients */
  int32_t good_steps;   /* consecutive non-overflow steps since the last change */
  int32_t t;            /* optimizer steps applied so far */
  uint32_t pending;     /* OR of non-finite flags raised in the current step */
  uint32_t overflow;    /* 1 if the last finished step was skipped */
  int32_t state_index;  /* current optimizer state set (ping-pong), 0 or 1 */
  double beta1_pow;     /* beta1^t, formed by t successive products */
  double beta2_pow;     /* beta2^t */
  double norm_sq;       /* global sum of squared reduced gradients (last zero_grad_norm) */
  double norm;          /* sqrt(norm_sq) */
  float clip_coef;      /* coefficient applied by the last clipped step (1 = none) */
  int32_t clip_apply;   /* 1 if clip_coef < 1 applies */
  int32_t norm_step;    /* t + 1 of the step zero_grad_norm was computed for */
  int32_t n_skipped;    /* steps skipped so far */
  int32_t error;        /* device error word: 0 = ok, else a ZERO_DEVERR_* code */
  uint32_t finish_count;/* library-internal CTA counter of the step's last kernel; 0 between calls */
} zero_scaler;

/* device error codes written to zero_scaler.error (first error wins) */
#define ZERO_DEVERR_STATE_INDEX 1   /* state_index outside the given sets */
#define ZERO_DEVERR_NO_NORM 2       /* clip requested but zero_grad_norm not run */
#define ZERO_DEVERR_TIMEOUT 3       /* a pipeline wait expired (2 s); results invalid */

/* Fill *out (host memory) with the initial scaler: scale = init_scale,
 * t = 0, beta powers 1, state set 0, all flags clear. */
ZERO_API int zero_scaler_init(const zero_hparams* hp, zero_scaler* out);

/* -------------------------------------------------------------- the step -- */

/* Pointer conventions shared by the calls below.
 *   replicas:     host array of N device pointers; replicas[r] points at
 *                 flat element `window_base` of rank r's 16-bit gradient, and
 *                 must cover every element of the processed ranks' slices.
 *                 Padding elements (j >= psi) must hold zeros. The step
 *                 may read the rest of the 16-byte block that holds the
 *                 window's last element (at most 14 bytes past it; the
 *                 values are not used), so that block must be allocated:
 *                 any buffer from cudaMalloc that holds the element is.
 *   window_base:  flat index that replicas[r] and flat_params point at
 *                 (0 for full buffers; i*S when only rank i's slice is held).
 *   flat_params:  device pointer at flat element window_base of the 16-bit
 *                 working parameters; rank i writes its slot [i*S, (i+1)*S).
 *   grad_shards:  host array of N device pointers; grad_shards[i][k] is the
 *                 fp32 reduced gradient of flat element i*S + k (S floats).
 *   master, exp_avg, exp_avg_sq: host arrays of n_sets*N device pointers;
 *                 entry [s*N + i] is rank i's fp32 shard (S floats) of state
 *                 set s. Entries of ranks outside [rank_lo, rank_hi) may be NULL.
 *   rank_lo, rank_hi: the owners processed, 0 <= rank_lo < rank_hi <= N.
 *   d_scaler:     device pointer to the zero_scaler.
 *   d_bucket_flags: device array of n_buckets uint32 (may be NULL); each
 *                 call ORs 1 into the flag of every bucket in which it finds
 *                 a non-finite reduced gradient. The caller clears them.
 */

/* Reduce-scatter (two-pass path, step 1) ("How far does splitting the batch
 * get you?", "Why does the all-reduce not get more expensive with more
 * ranks?": chunk i is summed hop by hop around the ring and is complete at
 * rank i; "What does gradient accumulation actually buy?": the reduction is
 * fp32; "Training models too big for one GPU: ZeRO & FSDP", "Mixed-precision
 * training": divide by the loss scale, skip the step on overflow, and "Data
 * parallelism and the all-reduce": average over the replicas): for the owners [rank_lo, rank_hi)
 * and bucket `bucket` (-1 = all buckets), write the unscaled, unclipped
 * reduced gradient to grad_shards, OR non-finite flags into d_bucket_flags
 * and d_scaler->pending, and, when d_workspace is not NULL, store the
 * per-tile squared-norm partial sums there for zero_grad_norm.
 * Reads 2N bytes and writes 4 bytes per element. */
ZERO_API int zero_reduce_scatter(const zero_plan* plan, int32_t bucket, int32_t rank_lo,
                                 int32_t rank_hi, const void* const* replicas,
                                 int64_t window_base, float* const* grad_shards,
                                 zero_scaler* d_scaler, uint32_t* d_bucket_flags,
                                 void* d_workspace, void* stream);

/* Global gradient norm and clip coefficient (two-pass path, step 2).
 * The pages give no clipping rule; the convention is the common one: L2 norm
 * of the unscaled, averaged gradient over the processed owners' elements;
 * c = max_norm / (norm + 1e-6) in fp64, applied (rounded to fp32) by the next
 * zero_step only if c < 1. Squares are accumulated in fp32 float-float pairs
 * (exact products, two-sum additions) in a fixed order that depends only on
 * the plan: per tile; per owner over a fixed partition of its tiles; the
 * owners' records in ascending owner order; fp64 for the final value. So the
 * result does not depend on the grid, and a window of owners gives the same
 * owner records as any other call that covers those owners (see
 * zero_grad_norm_local).
 * grad_shards == NULL: use the partials zero_reduce_scatter left in
 * d_workspace (it must have covered all segments of [rank_lo, rank_hi) in
 * this step). Otherwise recompute the partials from grad_shards (4 bytes
 * read per element). Writes norm_sq, norm, clip_coef, clip_apply and
 * norm_step to d_scaler. hp->max_grad_norm must be > 0. */
ZERO_API int zero_grad_norm(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                            const float* const* grad_shards, const zero_hparams* hp,
                            zero_scaler* d_scaler, void* d_workspace, void* stream);

/* ------------------------------------------- scalars across processes --
 * "Training models too big for one GPU: ZeRO & FSDP", "ZeRO stages 1, 2 and
 * 3": each rank updates only its own slice, so when the owners are split
 * over processes (each holding the N replicas of its owners' slices) only
 * the step's global scalars have to cross: whether any owner saw a
 * non-finite gradient (the step is skipped everywhere), and, when clipping,
 * the sum of squares behind the global norm.
 *
 * Protocol, per step, for processes whose windows [rank_lo, rank_hi)
 * partition [0, N):
 *   two-pass: zero_reduce_scatter -> zero_grad_norm_local -> sum the
 *     zero_exchange blobs of all processes -> zero_grad_norm_apply ->
 *     zero_step (instead of zero_grad_norm);
 *   fused: zero_step_update -> zero_grad_norm_local -> sum ->
 *     zero_grad_norm_apply -> zero_step_finish.
 * "Sum" is an element-wise integer sum of the blobs viewed as 260 int32
 * words (any all-reduce with SUM over int32, e.g. NCCL or gloo): each owner
 * record is non-zero in exactly one process, so the sum reproduces it
 * bit for bit, and the overflow words add up to the number of windows that
 * saw one. Every process then holds the same norm, clip coefficient and skip
 * decision as one process running zero_grad_norm over all N owners, bit for
 * bit. The per-bucket flags stay per process (OR them if needed). */

/* One owner's squared-norm record: hi + lo is the float-float sum of the
 * squares of its reduced gradients with |g| < 2^56; 2^192 (big_hi + big_lo)
 * is the sum of the rest (non-finite if a g was). */
typedef struct zero_norm_record {
  float hi, lo, big_hi, big_lo;
} zero_norm_record;

/* The scalars one process contributes to a step (1040 bytes, device memory,
 * 16-byte aligned). */
typedef struct zero_exchange {
  uint32_t overflow;        /* 1 if this window's step saw a non-finite value */
  uint32_t reserved[3];     /* 0 */
  zero_norm_record owner[ZERO_MAX_RANKS];  /* owners of the window; zeros elsewhere */
} zero_exchange;

/* Export: write *d_exchange from this process's window: overflow =
 * (d_scaler->pending != 0) after this step's reduce (two-pass) or update
 * (fused) pass; with clipping (hp->max_grad_norm > 0) the owner records of
 * [rank_lo, rank_hi), from the records zero_reduce_scatter left in
 * d_workspace (grad_shards NULL) or recomputed from grad_shards; zeros for
 * every other owner. Without clipping d_workspace and grad_shards are not
 * used (may be NULL). Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA. */
ZERO_API int zero_grad_norm_local(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                                  const float* const* grad_shards, const zero_hparams* hp,
                                  zero_scaler* d_scaler, void* d_workspace,
                                  zero_exchange* d_exchange, void* stream);

/* Import the summed exchange: a non-zero overflow word sets the step's
 * overflow (d_scaler->pending); with clipping, the norm fields of d_scaler
 * (norm_sq, norm, clip_coef, clip_apply, norm_step) from the records of all
 * N owners merged in ascending owner order, as zero_grad_norm computes them.
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA. */
ZERO_API int zero_grad_norm_apply(const zero_plan* plan, const zero_exchange* d_exchange,
                                  const zero_hparams* hp, zero_scaler* d_scaler, void* stream);

/* One optimizer step for the owners [rank_lo, rank_hi); call it once per
 * step: it ends by updating the loss scale, t and the skip bookkeeping.
 * Sources: "Training models too big for one GPU: ZeRO & FSDP", "ZeRO stages
 * 1, 2 and 3" (rank i updates its own slice of the optimizer state, then the
 * new weights are gathered), "Adam, and why it's expensive" (the update,
 * with eps outside the square root of the bias-corrected second moment;
 * AdamW's decoupled weight decay), "Mixed-precision training" (fp32 master
 * rounded to the 16-bit working copy; skip on overflow; dynamic loss scale).
 *
 * Fused path (grad_shards == NULL, needs n_sets == 2, no clip): one pass
 * reads the N replicas and the current state set (d_scaler->state_index),
 * reduces, unscales, checks, runs AdamW and writes the other state set and
 * the 16-bit parameters (2N + 26 bytes per element). If any element was
 * non-finite the step is skipped: the state index stays, and the parameters
 * are re-cast from the kept master (6 more bytes per element).
 *
 * Two-pass path (grad_shards != NULL, after zero_reduce_scatter and, when
 * hp->max_grad_norm > 0, zero_grad_norm): if the step's overflow word is set
 * nothing is written; otherwise AdamW runs on the reduced gradients (times
 * the clip coefficient when it applies) and the parameters are written
 * (30 bytes per element). n_sets == 2: the current set is read and the
 * other one written, and the finish makes it current (measured about 4 %
 * faster on GB300 than updating in place); n_sets == 1: the one set is
 * updated in place (12 bytes per element less memory).
 *
 * Errors: ZERO_EINVAL (bad ranges or NULL pointers, fused with clip or with
 * n_sets != 2), ZERO_EALIGN, ZERO_ECUDA. */
ZERO_API int zero_step(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                       float* const* master, float* const* exp_avg, float* const* exp_avg_sq,
                       int32_t n_sets, const float* const* grad_shards,
                       const void* const* replicas, int64_t window_base, void* flat_params,
                       const zero_hparams* hp, zero_scaler* d_scaler,
                       uint32_t* d_bucket_flags, void* stream);

/* zero_step in two calls, for callers that want to place their own work (or
 * timing events) between the update and the bookkeeping. zero_step(...)
 * gives exactly the results of zero_step_update(...) followed by
 * zero_step_finish(...) with the same arguments. (A fused zero_step whose
 * pass is one launch over at most 2^22 elements folds the finish into the
 * pass: the last CTA to finish does the bookkeeping and, if the step
 * overflowed, re-casts the parameters; one launch instead of two. At most
 * 2^20 elements with N <= 16 and one micro-batch it runs a kernel without the
 * copy pipeline, measured faster there.)
 * zero_step_update launches the update kernel of the chosen path (fused or
 * two-pass) and nothing else. zero_step_finish re-casts the parameters from
 * the kept master set if the fused step overflowed, then updates the loss
 * scale, t, the state index and the skip count. grad_shards only selects
 * the path (NULL = fused) in zero_step_finish; replicas may be NULL there. */
ZERO_API int zero_step_update(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                              float* const* master, float* const* exp_avg,
                              float* const* exp_avg_sq, int32_t n_sets,
                              const float* const* grad_shards, const void* const* replicas,
                              int64_t window_base, void* flat_params, const zero_hparams* hp,
                              zero_scaler* d_scaler, uint32_t* d_bucket_flags, void* stream);
ZERO_API int zero_step_finish(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                              float* const* master, int32_t n_sets,
                              const float* const* grad_shards, int64_t window_base,
                              void* flat_params, const zero_hparams* hp, zero_scaler* d_scaler,
                              void* stream);

/* ---------------------------------------------- micro-batch accumulation --
 * "How far does splitting the batch get you?", "What does gradient
 * accumulation actually buy?": run k micro-batches, accumulate each rank's
 * gradients locally in fp32, then reduce once (an fp32 reduce-scatter).
 *
 * zero_accumulate: for every replica r (all N) and every element j of the
 * window [rank_lo*S, rank_hi*S): accum[r][j] = first ? widen(micro[r][j])
 *   : accum[r][j] + widen(micro[r][j]) (fp32, round to nearest even).
 *   micro: N device pointers (16-bit, at flat element window_base);
 *   accum: N device pointers (fp32, same window). 10 bytes per replica and
 *   element (6 when first).
 * zero_reduce_scatter_accum / zero_step_accum / zero_step_update_accum: as
 *   the calls without the suffix, for a step of n_micro >= 1 micro-batches.
 *   `replicas` holds the last micro-batch's 16-bit gradients and, when
 *   n_micro > 1, `accum` the fp32 sums of the earlier n_micro - 1 (from
 *   zero_accumulate). Each replica's value is accum + widen(replica), one
 *   rounding, added in ring order; the unscale becomes fp32(1/(S_l*N*n_micro))
 *   (the average over every micro-batch of every rank). The accumulators are
 *   read, never written: the fused step reads 6N + 26 bytes per element.
 *   As with the replicas, the step may read the rest of the 16-byte block
 *   that holds an accumulator window's last element (at most 12 bytes past
 *   it), so that block must be allocated.
 *   With n_micro == 1 they equal the calls without the suffix (accum may be
 *   NULL). zero_step_accum's accumulators only matter on the fused path. */
ZERO_API int zero_accumulate(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                             const void* const* micro, float* const* accum, int64_t window_base,
                             int32_t first, void* stream);
ZERO_API int zero_reduce_scatter_accum(const zero_plan* plan, int32_t bucket, int32_t rank_lo,
                                       int32_t rank_hi, const void* const* replicas,
                                       const float* const* accum, int32_t n_micro,
                                       int64_t window_base, float* const* grad_shards,
                                       zero_scaler* d_scaler, uint32_t* d_bucket_flags,
                                       void* d_workspace, void* stream);
ZERO_API int zero_step_accum(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                             float* const* master, float* const* exp_avg,
                             float* const* exp_avg_sq, int32_t n_sets,
                             const float* const* grad_shards, const void* const* replicas,
                             const float* const* accum, int32_t n_micro, int64_t window_base,
                             void* flat_params, const zero_hparams* hp, zero_scaler* d_scaler,
                             uint32_t* d_bucket_flags, void* stream);
ZERO_API int zero_step_update_accum(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                                    float* const* master, float* const* exp_avg,
                                    float* const* exp_avg_sq, int32_t n_sets,
                                    const float* const* grad_shards, const void* const* replicas,
                                    const float* const* accum, int32_t n_micro,
                                    int64_t window_base, void* flat_params,
                                    const zero_hparams* hp, zero_scaler* d_scaler,
                                    uint32_t* d_bucket_flags, void* stream);

/* -------------------------------------- ring reduce-scatter across processes --
 * "How far does splitting the batch get you?", "Why does the all-reduce not
 * get more expensive with more ranks?": when the N ranks are N processes,
 * each with its own 16-bit gradient (the whole padded flat vector), the
 * reduce-scatter is a ring. Chunk i is owner i's slice [i*S, (i+1)*S): rank
 * i+1 starts it with its own values, each rank on the way adds its own, and
 * after N - 1 hops rank i adds its own last, so the sum is taken in the ring
 * order i+1, ..., N-1, 0, ..., i of zero_reduce_scatter, bit for bit. The
 * partial sums stay fp32 on the wire ("What does gradient accumulation
 * actually buy?": an fp32 reduce-scatter), 4 bytes per element per hop.
 *
 * zero_ring_hop: this rank's part of hop `hop` (1 .. N) of one step, for
 * chunk c = (rank - hop) mod N:
 *   hop 1:        out[k] = widen(grad[c*S + k]); recv must be NULL;
 *   1 < hop < N:  out[k] = recv[k] + widen(grad[c*S + k]) (fp32, one rounding);
 *   hop N:        c = rank; out[k] = (recv[k] + widen(grad[c*S + k])) *
 *                 fp32(1/(S_l*N)), S_l = d_scaler->scale: the unscaled
 *                 reduced gradient of this rank's slice (grad_shards[rank] of
 *                 zero_grad_norm_local / zero_step); a non-finite value ORs 1
 *                 into its bucket's flag and d_scaler->pending.
 *   (N = 1: hop 1 is the last hop, recv NULL.)
 * After hops 1 .. N-1 the caller sends `out` to rank (rank + 1) mod N and
 * receives the next hop's `recv` from rank (rank - 1) mod N (for example with
 * torch.distributed send/recv; NCCL keeps it on the stream).
 *   grad: device pointer at flat element 0 of this rank's gradient (psi_pad
 *         elements, padding zeros); recv, out: S floats each (device).
 * Reads 2 (+4 when recv) and writes 4 bytes per element. The rest of the
 * step runs as on one process with the window [rank, rank + 1):
 * zero_grad_norm_local / zero_grad_norm_apply across processes, then
 * zero_step; the new parameters are all-gathered by the caller.
 * Errors: ZERO_EINVAL (bad rank or hop, recv given on hop 1 or missing
 * after it, NULL pointers), ZERO_EALIGN, ZERO_ECUDA. */
ZERO_API int zero_ring_hop(const zero_plan* plan, int32_t rank, int32_t hop, const void* grad,
                           const float* recv, float* out, zero_scaler* d_scaler,
                           uint32_t* d_bucket_flags, void* stream);

/* Write the 16-bit working copy of the owners' slices from one fp32 master
 * set (round to nearest even): master[i] is rank i's shard (N entries).
 * Used to initialise the parameters; 6 bytes per element. */
ZERO_API int zero_cast_params(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                              const float* const* master, void* flat_params,
                              int64_t window_base, void* stream);

/* Self-test of the failure detection: launches one CTA that waits on a
 * pipeline barrier nobody ever completes, with the same bounded wait the
 * step kernels use but a limit of limit_ns nanoseconds (1e3 .. 1e10). When
 * the wait expires the kernel writes ZERO_DEVERR_TIMEOUT to d_scaler->error
 * and returns, leaving the context usable. Returns ZERO_EINVAL for a limit
 * outside the range. */
ZERO_API int zero_selftest_wait_timeout(zero_scaler* d_scaler, int64_t limit_ns, void* stream);

/* Checked builds (libzero_checked.so, compiled with -DZERO_CHECKED) test
 * every global and shared-memory range a kernel is about to touch against
 * the extents the plan gives (the call's window, the shard length, the
 * workspace's records, the stage slot); a failing test skips that access,
 * counts a violation and keeps the first one, and nothing traps.
 * zero_checked_status synchronizes `stream`, returns the count and the
 * first violation (site << 48 | low 48 bits of the offending index; sites:
 * 1 self-test, 2 scalar element, 3 vector element, 4 replica copy,
 * 5 accumulator copy, 6 state copy, 7 stage slot, 8 store, 9 norm record,
 * 10 micro-batch accumulation, 11 unit gather / shard, zero_units.h,
 * 12 reload of a reduced gradient for the norm's big-square path)
 * and clears both. zero_selftest_check plants one violation (site 1,
 * index 42). In the release build both return ZERO_ESTATE (and
 * zero_checked_status zeroes its outputs). */
ZERO_API int zero_checked_status(int64_t* violations, int64_t* first, void* stream);
ZERO_API int zero_selftest_check(void* stream);

/* Kernels launched per call, for accounting (L = ceil(segments processed /
 * 128), empty launches skipped): fused zero_step L + L (update; overflow
 * re-cast check merged with the bookkeeping in the last), or 1 when it folds
 * the finish into the pass (L == 1, at most 2^22 elements), two-pass zero_step
 * L + 1, zero_reduce_scatter L, zero_grad_norm 2 (+ L when it recomputes the
 * records), zero_grad_norm_local 2 with clipping (+ L when it recomputes),
 * 1 without, zero_grad_norm_apply 1, zero_cast_params L. */

/* Maximum number of norm tiles (ZERO_TILE_ELEMS elements each, counted per
 * segment) that one zero_grad_norm_noalloc call may cover: 2^19 tiles, about
 * 2.1e9 elements; the array is 8 MiB + 16 KiB of device memory. */
#define ZERO_NOALLOC_MAX_TILES (1 << 19)

/* zero_grad_norm_noalloc -- the global norm and clip coefficient of
 * zero_grad_norm (grad_shards form), without a caller-provided workspace.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: code running inside a host framework whose
 * allocator owns all of the GPU's memory, plugins and embedded runtimes that
 * are not allowed to call cudaMalloc themselves, and callers with a fixed
 * memory budget that cannot grow by a workspace sized from the model.
 * It allocates nothing: the per-tile records live in one fixed device
 * array of ZERO_NOALLOC_MAX_TILES + 64 * ZERO_NORM_OWNER_BLOCKS 16-byte
 * records inside the library, which every GPU that loads the library holds
 * until the process exits.
 *   grad_shards: as for zero_grad_norm, required (not NULL).
 *   Result: norm_sq, norm, clip_coef, clip_apply and norm_step in d_scaler,
 *   equal to what zero_grad_norm computes from the same gradients.
 * The first call on each device resolves the array's device address with
 * that device current; make that first call before any stream capture. The
 * address is kept for the life of the process: after cudaDeviceReset (or any
 * other destruction of the device's context) do not call it again.
 * All calls share the array and it keeps the last call's contents (each call
 * rewrites every record it reads). Calls that overlap on the GPU race on
 * it: order them on one stream.
 * Errors: ZERO_EINVAL (NULL arguments, bad ranks, max_grad_norm <= 0),
 * ZERO_EALIGN, ZERO_ERANGE (the owners' slices need more than
 * ZERO_NOALLOC_MAX_TILES tiles), ZERO_ECUDA. */
ZERO_API int zero_grad_norm_noalloc(const zero_plan* plan, int32_t rank_lo, int32_t rank_hi,
                                    const float* const* grad_shards, const zero_hparams* hp,
                                    zero_scaler* d_scaler, void* stream);

ZERO_API const char* zero_strerror(int status);
/* Library version: major * 10000 + minor * 100 + patch. */
ZERO_API int zero_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_H */
