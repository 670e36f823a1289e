// pdl.cuh -- programmatic dependent launch between this library's kernels.
//
// Each kernel is launched with programmatic stream serialization, so the
// next kernel in the stream may be scheduled before the previous one ends
// (its launch and CTA start-up overlap the previous kernel's tail). Every
// kernel's first statement waits for the previous grid to complete and its
// memory to be visible (griddepcontrol.wait, a no-op when there is no
// programmatic dependency), so no kernel reads or writes anything early;
// then it allows its own dependents to be scheduled. A dependent grid is
// scheduled only after every CTA of this grid has executed the trigger or
// exited, so a waiting dependent never holds resources the grid still needs.
#ifndef ZERO_PDL_CUH
#define ZERO_PDL_CUH

#include <cuda_runtime.h>

#include <utility>

constexpr bool kProgrammaticLaunch = true;

__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KernelArgs, typename... Actual>
cudaError_t launch_pdl(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Actual&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Actual>(args)...);
}

// An ordinary stream-ordered launch (no programmatic dependency) that
// returns the launch's own status, so a caller's earlier sticky error is
// neither consumed nor reported as this launch's.
template <typename... KernelArgs, typename... Actual>
cudaError_t launch_plain(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Actual&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Actual>(args)...);
}

#endif
