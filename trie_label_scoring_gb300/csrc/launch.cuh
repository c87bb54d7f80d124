// Kernel launch with programmatic dependent launch (PDL): a kernel may be
// launched while the previous kernel in its stream is still finishing, so the
// gap between dependent kernels shrinks. Every kernel of this library calls
// grid_dependency_wait() before it touches what an earlier kernel wrote, and
// every thread calls it before exiting, which keeps the usual stream order for
// all data: the wait returns once the grids it depends on have completed and
// their writes are visible. (The mma.sync doc attention reads the call's
// inputs and the node q rows before its wait; see grid_launch_dependents.)
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace quail {

// A no-op for a kernel that was launched without the programmatic attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream launch before this one finishes; it
// launches once every block of this grid has executed this or exited. Called
// after this kernel's own grid_dependency_wait, so everything before this
// kernel is complete when the next one starts, and the next one need wait
// only before it reads this kernel's outputs. Only kernels that hold no
// tensor memory call it.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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
