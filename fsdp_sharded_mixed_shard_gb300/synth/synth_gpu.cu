/*
 * synth_gpu.cu -- device build of the synthetic input generator (synth.h).
 * Harness only: fills gradient replicas (cast to bf16/fp16 with CUDA's
 * round-to-nearest-even conversions) and master weights in HBM before a run.
 * Never part of a timed step.
 */
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include "synth.h"

#define ZS_EXPORT __attribute__((visibility("default")))

namespace {

template <bool kBf16>
__global__ void fill_grad_kernel(uint16_t* __restrict__ dst, int64_t n, int64_t elem0,
                                 zs_grad_stream st) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
    float x = zs_grad_stream_value(&st, elem0 + k);
    if (kBf16) {
      __nv_bfloat16 h = __float2bfloat16_rn(x);
      dst[k] = *reinterpret_cast<uint16_t*>(&h);
    } else {
      __half h = __float2half_rn(x);
      dst[k] = *reinterpret_cast<uint16_t*>(&h);
    }
  }
}

__global__ void fill_master_kernel(float* __restrict__ dst, int64_t n, int64_t elem0,
                                   uint64_t seed, int64_t psi) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
    dst[k] = zs_master_value(seed, psi, elem0 + k);
}

int grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  if (b > 152 * 32) b = 152 * 32;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

extern "C" {

/* dst[k] = 16-bit cast of gradient element elem0 + k; is_bf16 selects bf16 or fp16.
 * Returns 0 or the CUDA error code. */
ZS_EXPORT int zs_gpu_fill_grad(void* dst, int64_t n, int64_t elem0, const zs_grad_spec* spec,
                     uint32_t step, uint32_t rank, int32_t is_bf16, void* stream) {
  if (n <= 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  zs_grad_stream st = zs_grad_stream_make(spec, step, rank);
  if (is_bf16)
    fill_grad_kernel<true><<<grid_for(n), 256, 0, s>>>((uint16_t*)dst, n, elem0, st);
  else
    fill_grad_kernel<false><<<grid_for(n), 256, 0, s>>>((uint16_t*)dst, n, elem0, st);
  return (int)cudaGetLastError();
}

ZS_EXPORT int zs_gpu_fill_master(float* dst, int64_t n, int64_t elem0, uint64_t seed, int64_t psi,
                       void* stream) {
  if (n <= 0) return 0;
  fill_master_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(dst, n, elem0, seed, psi);
  return (int)cudaGetLastError();
}

ZS_EXPORT int64_t zs_gpu_spec_size(void) { return (int64_t)sizeof(zs_grad_spec); }

}  // extern "C"
