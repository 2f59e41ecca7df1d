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

// Rows of sequence b in a call's per-node arrays.  Padded calls (cu == nullptr): rows
// b * N .. b * N + N - 1, of which the first n are the tree (n = N, or tree_len[b]
// clamped to [1, N] for ragged calls; the rest is padding).  Packed calls (cu = cumulative
// node counts, cu[0] = 0, cu[B] = T): rows cu[b] .. cu[b + 1] - 1, no padding.  A packed
// span that is empty, longer than N or outside [0, T) is not ok: it gets n = 0 (nothing
// of the sequence is read or written) and the caller reports JF_DEVERR_BAD_TREE_LEN.
struct SeqSpan {
  long long row0;   // first row
  int n;            // tree nodes
  int rows;         // rows the sequence owns: N padded, n packed
  bool ok;
};
__device__ __forceinline__ SeqSpan seq_span(const int32_t* cu, const int32_t* tree_len, int b,
                                            int N, long long T) {
  SeqSpan s;
  if (cu == nullptr) {
    s.row0 = static_cast<long long>(b) * N;
    s.rows = N;
    s.n = N;
    s.ok = true;
    if (tree_len != nullptr) {
      const int raw = tree_len[b];
      s.n = max(1, min(raw, N));
      s.ok = raw == s.n;
    }
  } else {
    const long long r0 = cu[b], r1 = cu[b + 1];
    s.ok = r0 >= 0 && r1 <= T && r1 - r0 >= 1 && r1 - r0 <= N;
    s.row0 = s.ok ? r0 : 0;
    s.n = s.ok ? static_cast<int>(r1 - r0) : 0;
    s.rows = s.n;
  }
  return s;
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
