// jf_api.cu -- status strings, version and the device-property cache.
#include <mutex>

#include "jf_common.cuh"

namespace jf {

int current_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace jf

extern "C" const char* jf_status_string(int status) {
  switch (status) {
    case JF_OK: return "JF_OK";
    case JF_ERR_INVALID_ARGUMENT: return "JF_ERR_INVALID_ARGUMENT";
    case JF_ERR_INVALID_TREE: return "JF_ERR_INVALID_TREE";
    case JF_ERR_UNSUPPORTED: return "JF_ERR_UNSUPPORTED";
    case JF_ERR_WORKSPACE_TOO_SMALL: return "JF_ERR_WORKSPACE_TOO_SMALL";
    case JF_ERR_CUDA: return "JF_ERR_CUDA";
    case JF_ERR_TIMEOUT: return "JF_ERR_TIMEOUT";
    case JF_ERR_MISALIGNED: return "JF_ERR_MISALIGNED";
    case JF_ERR_SCRATCH_CAPACITY: return "JF_ERR_SCRATCH_CAPACITY";
    default: return "JF_ERR_UNKNOWN";
  }
}

extern "C" int jf_version(void) { return 100; }   // 0.1.0
