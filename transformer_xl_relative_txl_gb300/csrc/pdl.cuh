// Programmatic dependent launch: a kernel launched behind another on the
// same stream with the programmatic-serialisation attribute may start its
// CTAs while the kernel before it is still running, once every CTA of that
// kernel has started or signalled.  Such a kernel does only CTA-local set-up
// (shared memory, barriers) before grid_dep_wait(), which returns once the
// kernel before it has completed and its memory operations are visible; it
// touches global memory and tensor memory only after it.  Launched without
// the attribute (or first on its stream), grid_dep_wait() returns at once.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace txl {

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the kernel launched behind this one start its CTAs (they then wait in
// grid_dep_wait until this kernel completes).
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` on `stream` with programmatic stream serialisation.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace txl
