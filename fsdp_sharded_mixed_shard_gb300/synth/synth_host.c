/*
 * synth_host.c -- host build of the synthetic input generator (synth.h).
 * Fills fp32 arrays; the caller converts to the gradient's 16-bit format.
 * Built with -ffp-contract=off so the fp32 steps match the GPU build.
 */
#include "synth.h"

uint64_t zs_host_u64(uint64_t seed, uint32_t tag, uint32_t step, uint32_t rank,
                     uint64_t elem) {
  return zs_u64(zs_key(seed, tag, step, rank), elem);
}

uint64_t zs_host_mix64(uint64_t z) { return zs_mix64(z); }

float zs_host_normal(uint64_t h) { return zs_normal(h); }

/* out[k] = gradient value of flat element elem0 + k, k in [0, n). */
void zs_host_fill_grad(float* out, int64_t n, int64_t elem0, const zs_grad_spec* spec,
                       uint32_t step, uint32_t rank) {
  for (int64_t k = 0; k < n; ++k) out[k] = zs_grad_value(spec, step, rank, elem0 + k);
}

/* out[k] = initial master weight of flat element elem0 + k. */
void zs_host_fill_master(float* out, int64_t n, int64_t elem0, uint64_t seed, int64_t psi) {
  for (int64_t k = 0; k < n; ++k) out[k] = zs_master_value(seed, psi, elem0 + k);
}

/* same values through the per-(step, rank) stream */
void zs_host_fill_grad_stream(float* out, int64_t n, int64_t elem0, const zs_grad_spec* spec,
                              uint32_t step, uint32_t rank) {
  zs_grad_stream s = zs_grad_stream_make(spec, step, rank);
  for (int64_t k = 0; k < n; ++k) out[k] = zs_grad_stream_value(&s, elem0 + k);
}

/* gradient values at arbitrary flat indices */
void zs_host_grad_at(float* out, const int64_t* elems, int64_t n, const zs_grad_spec* spec,
                     uint32_t step, uint32_t rank) {
  for (int64_t k = 0; k < n; ++k) out[k] = zs_grad_value(spec, step, rank, elems[k]);
}

/* initial master weights at arbitrary flat indices */
void zs_host_master_at(float* out, const int64_t* elems, int64_t n, uint64_t seed, int64_t psi) {
  for (int64_t k = 0; k < n; ++k) out[k] = zs_master_value(seed, psi, elems[k]);
}

int64_t zs_host_spec_size(void) { return (int64_t)sizeof(zs_grad_spec); }
