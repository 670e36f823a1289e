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
