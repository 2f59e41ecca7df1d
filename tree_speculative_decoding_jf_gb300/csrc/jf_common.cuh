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

}  // namespace jf
