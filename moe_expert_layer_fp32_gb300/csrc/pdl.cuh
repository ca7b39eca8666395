// Programmatic dependent launch between the kernels of one layer call.
//
// A kernel launched with pdl_attr() may start while the kernel before it in the
// stream is still running.  Rules every such kernel follows:
//  - before pdl_wait() it reads nothing the previous kernel writes and writes
//    nothing the previous kernel reads or writes;
//  - it calls pdl_launch_dependents() only after its own pdl_wait(), so a kernel
//    that starts early has every kernel but its direct predecessor complete.
// pdl_wait() returns at once when the kernel was launched without the attribute
// or its predecessor has finished; a kernel that never calls
// pdl_launch_dependents() lets its dependent start when it completes.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline void pdl_attr(cudaLaunchAttribute& a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
}

// <<<grid, block, smem, s>>> with the attribute
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  pdl_attr(attr[0]);
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace moe
