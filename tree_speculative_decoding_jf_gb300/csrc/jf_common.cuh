// jf_common.cuh -- host/device helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "jf.h"

namespace jf {

inline bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline jf_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

// Number of SMs of the current device (cached per device id); 0 if it cannot be queried.
int current_sm_count();

__device__ __forceinline__ void report(int32_t* dev_err, int32_t bits) {
  if (dev_err != nullptr) atomicOr(dev_err, bits);
}

// Programmatic dependent launch: every kernel of the library is launched so that it may
// start while the previous kernel of the stream finishes; it calls grid_dependency_wait()
// before its first global-memory access (which returns once the previous grid has
// completed and its writes are visible) and grid_dependents_launch() once it no longer
// needs its SM slot exclusively.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace jf
