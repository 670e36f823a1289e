/*
 * plan.cpp -- host planner: flatten, pad, shard, bucket, segment, account.
 *
 * "Training models too big for one GPU: ZeRO & FSDP", "FSDP: the same idea,
 * one unit at a time": a unit's parameters are flattened and sharded across
 * the GPUs; "ZeRO stages 1, 2 and 3": GPU i updates only its 1/N slice.
 * "How far does splitting the batch get you?", "How does the collective hide
 * behind the backward pass?": gradients are reduced in buckets.
 *
 * Layout: one flat buffer, padded once to a multiple of N; rank i owns
 * [i*S, (i+1)*S); bucket k is [k*B, min((k+1)*B, psi_pad)); a segment is a
 * maximal range inside one bucket and one rank's slice. Segments are found by
 * merging the sorted cut points {k*B} and {i*S}.
 */
#include <algorithm>
#include <new>

#include "zero_internal.h"

static_assert(sizeof(zero_scaler) == 80, "zero_scaler layout is part of the ABI");
static_assert(sizeof(zero_plan_info) == 168, "zero_plan_info layout is part of the ABI");
static_assert(sizeof(zero_hparams) == 64, "zero_hparams layout is part of the ABI");
static_assert(sizeof(zero_segment) == 24, "zero_segment layout is part of the ABI");

extern "C" {

ZERO_API int zero_plan_create(const int64_t* numels, int32_t n_tensors, int32_t n_ranks,
                              int64_t bucket_elems, zero_dtype grad_dtype, zero_plan** out) {
  if (!out) return ZERO_EINVAL;
  *out = nullptr;
  if (n_tensors < 0 || (n_tensors > 0 && !numels) || bucket_elems < 0 || n_ranks < 1)
    return ZERO_EINVAL;
  if (grad_dtype != ZERO_BF16 && grad_dtype != ZERO_FP16) return ZERO_EINVAL;
  if (n_ranks > ZERO_MAX_RANKS) return ZERO_ERANGE;

  zero_plan* p = new (std::nothrow) zero_plan();
  if (!p) return ZERO_ENOMEM;
  try {
    p->offsets.resize(static_cast<size_t>(n_tensors));
    int64_t psi = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
      if (numels[k] < 0) {
        delete p;
        return ZERO_EINVAL;
      }
      p->offsets[k] = psi;
      psi += numels[k];
    }
    const int64_t N = n_ranks;
    const int64_t rem = psi % N;
    const int64_t pad = rem == 0 ? 0 : N - rem;
    const int64_t psi_pad = psi + pad;
    const int64_t S = psi_pad / N;

    zero_plan_info& I = p->info;
    I = zero_plan_info{};
    I.psi = psi;
    I.pad = pad;
    I.psi_pad = psi_pad;
    I.shard_elems = S;
    I.bucket_elems = bucket_elems;
    I.n_ranks = n_ranks;
    I.n_tensors = n_tensors;
    I.grad_dtype = grad_dtype;
    I.n_buckets = psi_pad == 0 ? 0
                  : bucket_elems == 0 ? 1
                                      : static_cast<int32_t>((psi_pad - 1) / bucket_elems + 1);

    // merge the bucket and shard cut points and emit the ranges between them
    p->rank_seg0.assign(static_cast<size_t>(N) + 1, 0);
    int64_t pos = 0;
    int64_t next_bucket_cut = bucket_elems == 0 ? psi_pad : bucket_elems;
    int32_t bucket = 0;
    int32_t rank = 0;
    int64_t tiles = 0;
    while (pos < psi_pad) {
      int64_t rank_end = (rank + 1) * S;
      int64_t end = std::min(std::min(next_bucket_cut, rank_end), psi_pad);
      zero_segment s{pos, end, rank, bucket};
      p->segs.push_back(s);
      int64_t nt = (end - pos + ZERO_TILE_ELEMS - 1) / ZERO_TILE_ELEMS;
      p->seg_tile0.push_back(tiles);
      p->seg_tiles.push_back(nt);
      tiles += nt;
      pos = end;
      if (pos == rank_end) {
        ++rank;
        if (rank < N) p->rank_seg0[rank] = static_cast<int32_t>(p->segs.size());
      }
      if (pos == next_bucket_cut && bucket_elems != 0) {
        ++bucket;
        next_bucket_cut += bucket_elems;
      }
    }
    for (int32_t r = rank + 1; r <= N; ++r) p->rank_seg0[r] = static_cast<int32_t>(p->segs.size());
    p->rank_seg0[N] = static_cast<int32_t>(p->segs.size());
    I.n_segments = static_cast<int32_t>(p->segs.size());
    I.n_tiles = tiles;

    // accounting (unpadded psi, K = 12 bytes of fp32 master + m + v)
    const double dpsi = static_cast<double>(psi);
    const double dN = static_cast<double>(N);
    I.bill_ddp = 16.0 * dpsi;
    I.bill_z1 = 4.0 * dpsi + 12.0 * dpsi / dN;
    I.bill_z2 = 2.0 * dpsi + 14.0 * dpsi / dN;
    I.bill_z3 = 16.0 * dpsi / dN;
    const double grad_bytes = 2.0 * dpsi;
    I.ring_bytes_per_rank = 2.0 * (dN - 1.0) * grad_bytes / dN;
    I.ring_hops = 2.0 * (dN - 1.0);
    I.comm_elems_ddp = 2.0 * dpsi;
    I.comm_elems_z1 = 2.0 * dpsi;
    I.comm_elems_z2 = 2.0 * dpsi;
    I.comm_elems_z3 = 3.0 * dpsi;
    I.step_bytes_fused = 2.0 * dN + 26.0;
    I.step_bytes_two_pass = 2.0 * dN + 34.0;
  } catch (...) {
    delete p;
    return ZERO_ENOMEM;
  }
  *out = p;
  return ZERO_OK;
}

ZERO_API void zero_plan_destroy(zero_plan* plan) { delete plan; }

ZERO_API int zero_plan_get_info(const zero_plan* plan, zero_plan_info* out) {
  if (!plan || !out) return ZERO_EINVAL;
  *out = plan->info;
  return ZERO_OK;
}

ZERO_API int zero_plan_info_get(const zero_plan* plan, zero_plan_info* out) {
  return zero_plan_get_info(plan, out);
}

ZERO_API int zero_plan_tensor_offsets(const zero_plan* plan, int64_t* out) {
  if (!plan || (!out && !plan->offsets.empty())) return ZERO_EINVAL;
  std::copy(plan->offsets.begin(), plan->offsets.end(), out);
  return ZERO_OK;
}

ZERO_API int zero_plan_segments(const zero_plan* plan, zero_segment* out, int32_t cap) {
  if (!plan || cap < 0 || (!out && cap > 0)) return ZERO_EINVAL;
  const int32_t n = plan->info.n_segments;
  const int32_t c = std::min(n, cap);
  std::copy(plan->segs.begin(), plan->segs.begin() + c, out);
  return cap < n ? ZERO_ERANGE : ZERO_OK;
}

ZERO_API int zero_plan_buckets(const zero_plan* plan, zero_bucket* out, zero_segment* segs) {
  if (!plan) return ZERO_EINVAL;
  if (segs) std::copy(plan->segs.begin(), plan->segs.end(), segs);
  if (!out) return ZERO_OK;
  const int32_t nb = plan->info.n_buckets;
  for (int32_t b = 0; b < nb; ++b) {
    int64_t lo = 0, hi = 0;
    zero_plan_bucket_range(plan, b, &lo, &hi);
    out[b].lo = lo;
    out[b].hi = hi;
    out[b].seg_first = 0;
    out[b].seg_count = 0;
  }
  // segments are ordered by lo, so each bucket's segments are one run
  for (int32_t s = plan->info.n_segments - 1; s >= 0; --s) {
    zero_bucket& b = out[plan->segs[s].bucket];
    b.seg_first = s;
    b.seg_count += 1;
  }
  return ZERO_OK;
}

ZERO_API int zero_plan_bucket_range(const zero_plan* plan, int32_t bucket, int64_t* lo,
                                    int64_t* hi) {
  if (!plan || !lo || !hi || bucket < 0 || bucket >= plan->info.n_buckets) return ZERO_EINVAL;
  const int64_t B = plan->info.bucket_elems;
  if (B == 0) {
    *lo = 0;
    *hi = plan->info.psi_pad;
  } else {
    *lo = static_cast<int64_t>(bucket) * B;
    *hi = std::min(*lo + B, plan->info.psi_pad);
  }
  return ZERO_OK;
}

ZERO_API size_t zero_workspace_bytes(const zero_plan* plan, int32_t two_pass) {
  if (!plan || !two_pass) return 0;
  // one 16-byte norm record per tile, then the norm finish's share records
  const size_t records = static_cast<size_t>(plan->info.n_tiles) +
                         static_cast<size_t>(plan->info.n_ranks) * zero_detail::kNormOwnerBlocks;
  return (records * 16 + 255) & ~static_cast<size_t>(255);
}

ZERO_API int zero_scaler_init(const zero_hparams* hp, zero_scaler* out) {
  if (!hp || !out) return ZERO_EINVAL;
  if (!(hp->init_scale > 0.0) || hp->growth_interval < 1) return ZERO_EINVAL;
  *out = zero_scaler{};
  out->scale = static_cast<float>(hp->init_scale);
  out->beta1_pow = 1.0;
  out->beta2_pow = 1.0;
  out->clip_coef = 1.0f;
  return ZERO_OK;
}

ZERO_API const char* zero_strerror(int status) {
  switch (status) {
    case ZERO_OK: return "ok";
    case ZERO_EINVAL: return "invalid argument";
    case ZERO_EALIGN: return "device pointer not 16-byte aligned";
    case ZERO_ERANGE: return "size exceeds a library limit";
    case ZERO_ECUDA: return "CUDA launch or runtime error";
    case ZERO_ENOMEM: return "host allocation failed";
    case ZERO_ESTATE: return "call order violated";
    default: return "unknown status";
  }
}

ZERO_API int zero_version(void) { return 100; }

}  // extern "C"
