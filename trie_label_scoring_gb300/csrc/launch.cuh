// Kernel launch with programmatic dependent launch (PDL): a kernel may be
// launched while the previous kernel in its stream is still finishing, so the
// gap between dependent kernels shrinks. Every kernel of this library calls
// grid_dependency_wait() before it touches global memory, which keeps the
// usual stream order for all data: the wait returns once the grids it depends
// on have completed and their writes are visible.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace quail {

// A no-op for a kernel that was launched without the programmatic attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace quail
