/*
 * units.c -- CPU checker for the stage-3 FSDP unit layout and its all-gather.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h). Plain loops, one statement per
 * step of the definition; shares no code with the CUDA library.
 */
#include <string.h>

#include "oracle.h"

int orc_unit_plan_make(const int64_t* numels, int32_t n_tensors, const int32_t* unit_of_tensor,
                       int32_t n_units, int32_t n_ranks, int32_t align_elems,
                       orc_unit_plan* out, orc_unit* units, int32_t* slot_tensor,
                       int64_t* tensor_offset) {
  if (!out || n_tensors < 1 || n_units < 1 || n_ranks < 1 || align_elems < 1) return -1;
  if (!numels || !unit_of_tensor) return -1;
  for (int32_t k = 0; k < n_tensors; ++k)
    if (numels[k] < 0 || unit_of_tensor[k] < 0 || unit_of_tensor[k] >= n_units) return -1;
  memset(out, 0, sizeof(*out));
  out->n_units = n_units;
  out->n_ranks = n_ranks;
  out->n_tensors = n_tensors;
  out->align_elems = align_elems;

  const int64_t grain = (int64_t)n_ranks * align_elems;
  int64_t flat = 0, held = 0, slot = 0;
  double best_one = 0.0, best_pair = 0.0, prev = 0.0, biggest = 0.0;
  for (int32_t u = 0; u < n_units; ++u) {
    /* flatten the unit: its tensors in list order, back to back */
    int64_t psi_u = 0;
    int32_t count = 0;
    int32_t first = (int32_t)slot;
    for (int32_t k = 0; k < n_tensors; ++k) {
      if (unit_of_tensor[k] != u) continue;
      if (tensor_offset) tensor_offset[k] = psi_u;
      if (slot_tensor) slot_tensor[slot] = k;
      ++slot;
      ++count;
      psi_u += numels[k];
    }
    if (count == 0) return -1;
    /* pad to a multiple of N * align and cut into N equal slices */
    int64_t pad = (grain - psi_u % grain) % grain;
    int64_t psi_pad = psi_u + pad;
    int64_t shard = psi_pad / n_ranks;
    if (units) {
      units[u].psi = psi_u;
      units[u].pad = pad;
      units[u].psi_pad = psi_pad;
      units[u].shard = shard;
      units[u].shard_offset = held;
      units[u].flat_offset = flat;
      units[u].n_tensors = count;
      units[u].first_slot = first;
    }
    out->psi += psi_u;
    if ((double)psi_u > biggest) biggest = (double)psi_u;
    flat += psi_pad;
    held += shard;
    if (psi_pad > out->max_unit_psi_pad) out->max_unit_psi_pad = psi_pad;
    /* gathered bytes: 2 per element (bf16 or fp16 working copy) */
    double gathered = 2.0 * (double)psi_pad;
    if (gathered > best_one) best_one = gathered;
    double pair = u == 0 ? gathered : prev + gathered;
    if (pair > best_pair) best_pair = pair;
    prev = gathered;
  }
  out->psi_pad = flat;
  out->shard = held;

  /* [Z3] "Peak transient memory": the persistent share is 16 bytes per held
   * element (2 weight + 2 gradient + 12 optimizer state); the transient is
   * the gathered unit(s). [ZF] "FSDP: the same idea, one unit at a time":
   * one or two gathered units. Backward: the unit's full gradient exists
   * beside its gathered parameters until it is reduce-scattered. */
  out->persistent_bytes = 16.0 * (double)held;
  out->peak_one_bytes = out->persistent_bytes + best_one;
  out->peak_two_bytes = out->persistent_bytes + best_pair;
  out->peak_backward_bytes = out->persistent_bytes + 2.0 * best_one;
  out->max_unit_fraction = out->psi > 0 ? biggest / (double)out->psi : 0.0;

  /* [SB] "What does each stage cost on the wire?": a forward all-gather, a
   * backward all-gather and a reduce-scatter, psi elements each; a ring
   * moves (N-1) slices per rank for each of them. */
  out->comm_elems = 3.0 * (double)flat;
  out->comm_bytes = 2.0 * out->comm_elems;
  out->ring_bytes = 3.0 * 2.0 * (double)(n_ranks - 1) * (double)held;
  out->n_gathers = 2 * n_units;
  return 0;
}

void orc_gather_unit(const orc_unit* u, int32_t n_ranks, const uint16_t* const* shards,
                     uint16_t* full) {
  for (int32_t r = 0; r < n_ranks; ++r)
    for (int64_t j = 0; j < u->shard; ++j)
      full[(int64_t)r * u->shard + j] = shards[r][u->shard_offset + j];
}

void orc_shard_unit(const orc_unit* u, int32_t n_ranks, const uint16_t* full,
                    uint16_t* const* shards) {
  for (int32_t r = 0; r < n_ranks; ++r)
    for (int64_t j = 0; j < u->shard; ++j)
      shards[r][u->shard_offset + j] = full[(int64_t)r * u->shard + j];
}

int orc_strategy_cost_make(const orc_unit_plan* p, int32_t strategy, int32_t n_replicas,
                           orc_strategy_cost* out) {
  if (!p || !out || n_replicas < 1) return -1;
  if (strategy != ORC_HYBRID_SHARD && n_replicas != 1) return -1;
  memset(out, 0, sizeof(*out));
  const double g = (double)p->n_ranks;
  const double R = (double)n_replicas;
  const double psi = (double)p->psi;
  const double P = (double)p->psi_pad;
  const double S = (double)p->shard;
  const double U = (double)p->max_unit_psi_pad;
  switch (strategy) {
    case ORC_FULL_SHARD:
    case ORC_HYBRID_SHARD:
      /* stage 3 inside the shard group: gather before the forward and again
       * before the backward, reduce-scatter after it */
      out->persistent_bytes = 16.0 * S;
      out->peak_bytes = out->persistent_bytes + 2.0 * U;
      out->comm_elems = 3.0 * P;
      out->ring_bytes = 3.0 * (g - 1.0) * S * 2.0;
      out->shard_ranks = p->n_ranks;
      out->gathers_per_unit = 2;
      if (strategy == ORC_HYBRID_SHARD && n_replicas > 1) {
        /* the groups hold replicas of the same shard: all-reduce each
         * rank's S reduced gradient elements across the R groups */
        out->comm_elems_inter = 2.0 * S;
        out->ring_bytes_inter = 2.0 * (R - 1.0) / R * (2.0 * S);
        out->comm_elems += out->comm_elems_inter;
        out->ring_bytes += out->ring_bytes_inter;
      }
      return 0;
    case ORC_SHARD_GRAD_OP:
      /* stage 2: 16-bit parameters resident, gradients and optimizer states
       * sharded; reduce-scatter, then all-gather of the updated parameters */
      out->persistent_bytes = 2.0 * P + 14.0 * S;
      out->peak_bytes = out->persistent_bytes;
      out->comm_elems = 2.0 * P;
      out->ring_bytes = 2.0 * (g - 1.0) * S * 2.0;
      out->shard_ranks = p->n_ranks;
      out->gathers_per_unit = 1;
      return 0;
    case ORC_NO_SHARD:
      /* plain data parallelism: everything replicated, one all-reduce */
      out->persistent_bytes = 16.0 * psi;
      out->peak_bytes = out->persistent_bytes;
      out->comm_elems = 2.0 * psi;
      out->ring_bytes = orc_ring_bytes(2.0 * psi, p->n_ranks);
      out->shard_ranks = 1;
      out->gathers_per_unit = 0;
      return 0;
    case ORC_NO_RESHARD_AFTER_FORWARD:
      /* stage-3 shards; each unit gathered once, in the forward pass, and
       * kept until its backward: at the turn every unit is gathered */
      out->persistent_bytes = 16.0 * S;
      out->peak_bytes = out->persistent_bytes + 2.0 * P;
      out->comm_elems = 2.0 * P;
      out->ring_bytes = 2.0 * (g - 1.0) * S * 2.0;
      out->shard_ranks = p->n_ranks;
      out->gathers_per_unit = 1;
      return 0;
    default:
      return -1;
  }
}
