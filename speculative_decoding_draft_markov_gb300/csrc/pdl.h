// Programmatic dependent launch for the small kernels of the step: the next kernel in the
// stream is scheduled while the current one runs, so its launch latency hides behind the
// current kernel's tail.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace dspark {

// First statement of a kernel launched with launch_pdl: wait until the previous kernel in the
// stream has completed and its writes are visible (nothing this kernel reads or writes can race
// a predecessor), then let the next kernel be scheduled.  A no-op for a plain launch.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dspark
