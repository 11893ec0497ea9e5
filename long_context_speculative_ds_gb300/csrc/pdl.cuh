// Programmatic dependent launch for the three kernels of one verify call
// (split pass -> combine -> finalize -> the next call's split pass).
//
// Each of these kernels is launched with programmatic stream serialisation
// and begins with griddepcontrol.wait, before it touches global memory: the
// wait returns once the preceding kernel of the stream has completed and its
// writes are visible, so the data dependencies are exactly those of plain
// stream order.  What the launch attribute buys is that the dependent grid
// is already scheduled when that happens (its launch latency overlaps the
// tail of the preceding grid); each kernel signals launch_dependents as soon
// as it starts.  In a kernel launched without the attribute
// griddepcontrol.wait returns at once; a dependent of a kernel that never
// signals is launched when that kernel completes.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace ds {

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
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

}  // namespace ds
