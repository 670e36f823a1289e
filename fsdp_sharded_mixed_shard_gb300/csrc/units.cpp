/*
 * units.cpp -- host planner for the stage-3 FSDP unit layout.
 *
 * "Training models too big for one GPU: ZeRO & FSDP", "FSDP: the same idea,
 * one unit at a time": the model is wrapped into units and each unit's
 * parameters are flattened and sharded across the GPUs; peak memory is the
 * shards plus one or two gathered units. "ZeRO Stage 3 Math", "Peak
 * transient memory": peak = persistent 16 psi / N + one layer's full
 * parameters (+ activations, not counted here). "How far does splitting the
 * batch get you?", "What does each stage cost on the wire?": stage 3 moves
 * 3 psi elements per step.
 *
 * Tensors are grouped by a stable counting sort on their unit id; each unit
 * is padded to a multiple of N * align and cut into N slices; a rank's shard
 * buffer stacks its slices unit after unit.
 */
#include <algorithm>
#include <new>
#include <vector>

#include "zero_units_internal.h"

static_assert(sizeof(zero_unit) == 56, "zero_unit layout is part of the ABI");
static_assert(sizeof(zero_unit_plan_info) == 120, "zero_unit_plan_info layout is part of the ABI");
static_assert(sizeof(zero_strategy_cost) == 56, "zero_strategy_cost layout is part of the ABI");

extern "C" {

ZERO_API int zero_unit_plan_create(const int64_t* numels, int32_t n_tensors,
                                   const int32_t* unit_of_tensor, int32_t n_units,
                                   int32_t n_ranks, int32_t align_elems, zero_unit_plan** out) {
  if (!out) return ZERO_EINVAL;
  *out = nullptr;
  if (!numels || !unit_of_tensor || n_tensors < 1 || n_units < 1 || n_ranks < 1 ||
      align_elems < 1)
    return ZERO_EINVAL;
  if (n_ranks > ZERO_MAX_RANKS || align_elems > ZERO_UNIT_MAX_ALIGN) return ZERO_ERANGE;
  for (int32_t k = 0; k < n_tensors; ++k)
    if (numels[k] < 0 || unit_of_tensor[k] < 0 || unit_of_tensor[k] >= n_units)
      return ZERO_EINVAL;

  zero_unit_plan* p = new (std::nothrow) zero_unit_plan();
  if (!p) return ZERO_ENOMEM;
  try {
    // stable counting sort of the tensors by unit
    std::vector<int32_t> count(static_cast<size_t>(n_units) + 1, 0);
    for (int32_t k = 0; k < n_tensors; ++k) ++count[unit_of_tensor[k] + 1];
    for (int32_t u = 0; u < n_units; ++u) {
      if (count[u + 1] == 0) {  // a unit without tensors
        delete p;
        return ZERO_EINVAL;
      }
      count[u + 1] += count[u];
    }
    p->slot_tensor.resize(static_cast<size_t>(n_tensors));
    p->tensor_offset.resize(static_cast<size_t>(n_tensors));
    p->units.resize(static_cast<size_t>(n_units));
    std::vector<int32_t> fill(count.begin(), count.end() - 1);
    for (int32_t k = 0; k < n_tensors; ++k) p->slot_tensor[fill[unit_of_tensor[k]]++] = k;

    const int64_t N = n_ranks;
    const int64_t grain = N * align_elems;
    zero_unit_plan_info& I = p->info;
    I = zero_unit_plan_info{};
    I.n_units = n_units;
    I.n_ranks = n_ranks;
    I.n_tensors = n_tensors;
    I.align_elems = align_elems;
    int64_t flat = 0, held = 0, largest_psi = 0, largest_pad = 0, best_pair = 0, prev = 0;
    for (int32_t u = 0; u < n_units; ++u) {
      zero_unit& U = p->units[u];
      U = zero_unit{};
      U.first_slot = count[u];
      U.n_tensors = count[u + 1] - count[u];
      int64_t off = 0;
      for (int32_t s = count[u]; s < count[u + 1]; ++s) {
        const int32_t k = p->slot_tensor[s];
        p->tensor_offset[k] = off;
        off += numels[k];
      }
      U.psi = off;
      const int64_t rem = off % grain;
      U.pad = rem == 0 ? 0 : grain - rem;
      U.psi_pad = off + U.pad;
      U.shard_elems = U.psi_pad / N;
      U.shard_offset = held;
      U.flat_offset = flat;
      held += U.shard_elems;
      flat += U.psi_pad;
      I.psi += U.psi;
      largest_psi = std::max(largest_psi, U.psi);
      largest_pad = std::max(largest_pad, U.psi_pad);
      best_pair = std::max(best_pair, prev + U.psi_pad);
      prev = U.psi_pad;
    }
    I.psi_pad = flat;
    I.shard_elems = held;
    I.max_unit_psi_pad = largest_pad;
    I.persistent_bytes = 16.0 * static_cast<double>(held);
    I.peak_one_bytes = I.persistent_bytes + 2.0 * static_cast<double>(largest_pad);
    I.peak_two_bytes = I.persistent_bytes + 2.0 * static_cast<double>(best_pair);
    I.peak_backward_bytes = I.persistent_bytes + 4.0 * static_cast<double>(largest_pad);
    I.max_unit_fraction =
        I.psi > 0 ? static_cast<double>(largest_psi) / static_cast<double>(I.psi) : 0.0;
    I.comm_elems = 3.0 * static_cast<double>(flat);
    I.comm_bytes = 2.0 * I.comm_elems;
    I.ring_bytes = 6.0 * static_cast<double>(N - 1) * static_cast<double>(held);
    I.n_gathers = 2 * n_units;
  } catch (...) {
    delete p;
    return ZERO_ENOMEM;
  }
  *out = p;
  return ZERO_OK;
}

ZERO_API void zero_unit_plan_destroy(zero_unit_plan* plan) { delete plan; }

ZERO_API int zero_unit_plan_get_info(const zero_unit_plan* plan, zero_unit_plan_info* out) {
  if (!plan || !out) return ZERO_EINVAL;
  *out = plan->info;
  return ZERO_OK;
}

ZERO_API int zero_unit_plan_units(const zero_unit_plan* plan, zero_unit* out, int32_t capacity) {
  if (!plan || !out) return ZERO_EINVAL;
  if (capacity < plan->info.n_units) return ZERO_ERANGE;
  std::copy(plan->units.begin(), plan->units.end(), out);
  return ZERO_OK;
}

ZERO_API int zero_unit_plan_tensors(const zero_unit_plan* plan, int32_t* slot_tensor,
                                    int64_t* tensor_offset, int32_t capacity) {
  if (!plan) return ZERO_EINVAL;
  if ((slot_tensor || tensor_offset) && capacity < plan->info.n_tensors) return ZERO_ERANGE;
  if (slot_tensor) std::copy(plan->slot_tensor.begin(), plan->slot_tensor.end(), slot_tensor);
  if (tensor_offset)
    std::copy(plan->tensor_offset.begin(), plan->tensor_offset.end(), tensor_offset);
  return ZERO_OK;
}

ZERO_API int zero_unit_plan_strategy_cost(const zero_unit_plan* plan, int32_t strategy,
                                          int32_t n_replicas, zero_strategy_cost* out) {
  if (!plan || !out || n_replicas < 1) return ZERO_EINVAL;
  if (strategy != ZERO_HYBRID_SHARD && n_replicas != 1) return ZERO_EINVAL;
  const zero_unit_plan_info& I = plan->info;
  const double g = I.n_ranks, reps = n_replicas;
  const double held = static_cast<double>(I.shard_elems);
  const double padded = static_cast<double>(I.psi_pad);
  const double params = static_cast<double>(I.psi);
  const double largest = static_cast<double>(I.max_unit_psi_pad);
  zero_strategy_cost c{};
  c.shard_ranks = I.n_ranks;
  switch (strategy) {
    case ZERO_FULL_SHARD:
    case ZERO_HYBRID_SHARD:
      // stage 3 in the group: gathered for the forward and again for the
      // backward, reduce-scattered after it
      c.persistent_bytes = 16.0 * held;
      c.peak_bytes = c.persistent_bytes + 2.0 * largest;
      c.comm_elems = 3.0 * padded;
      c.ring_bytes = 6.0 * (g - 1.0) * held;
      c.gathers_per_unit = 2;
      if (strategy == ZERO_HYBRID_SHARD && n_replicas > 1) {
        // the groups are replicas: all-reduce each rank's reduced shard
        c.comm_elems_inter = 2.0 * held;
        c.ring_bytes_inter = 4.0 * held * (reps - 1.0) / reps;
        c.comm_elems += c.comm_elems_inter;
        c.ring_bytes += c.ring_bytes_inter;
      }
      break;
    case ZERO_SHARD_GRAD_OP:
      // stage 2: the 16-bit weights stay resident
      c.persistent_bytes = 2.0 * padded + 14.0 * held;
      c.peak_bytes = c.persistent_bytes;
      c.comm_elems = 2.0 * padded;
      c.ring_bytes = 4.0 * (g - 1.0) * held;
      c.gathers_per_unit = 1;
      break;
    case ZERO_NO_SHARD:
      c.persistent_bytes = 16.0 * params;
      c.peak_bytes = c.persistent_bytes;
      c.comm_elems = 2.0 * params;
      c.ring_bytes = 2.0 * (g - 1.0) * (2.0 * params) / g;
      c.shard_ranks = 1;
      c.gathers_per_unit = 0;
      break;
    case ZERO_NO_RESHARD_AFTER_FORWARD:
      // one gather per unit, kept from its forward to its backward
      c.persistent_bytes = 16.0 * held;
      c.peak_bytes = c.persistent_bytes + 2.0 * padded;
      c.comm_elems = 2.0 * padded;
      c.ring_bytes = 4.0 * (g - 1.0) * held;
      c.gathers_per_unit = 1;
      break;
    default:
      return ZERO_EINVAL;
  }
  *out = c;
  return ZERO_OK;
}

}  // extern "C"
