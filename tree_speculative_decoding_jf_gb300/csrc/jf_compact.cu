// jf_compact.cu -- accepted-path KV compaction.
//
// After greedy verification the accepted root path [0, path[1], .., path[a]] of sequence b
// becomes part of its context: the K/V rows at logical positions P + path[k] move to
// P + k (k = 1..a) and the prefix grows to P + a + 1 (JetFlow explainer, technical
// summary §2 "Method": tree nodes hold their K/V after the prefix; the accepted branch is
// the context the target continues from).
//
// One CTA per (sequence, kv-head) moves that head's rows; they are disjoint from every
// other CTA's.  Sources and destinations of one sequence overlap, but along the path
// path[k] >= k rises strictly, so taking the nodes in increasing chunks and, within a
// chunk, reading every source into shared memory before writing any destination gives
// the sequential result: a destination of chunk c lies below every source of chunks > c,
// and a source of chunk c lies above every destination of chunks < c.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kCompactThreads = 256;
constexpr int kCompactChunk = 32;          // nodes per read/write phase
constexpr int kPage = 16;

template <int D>
__global__ void __launch_bounds__(kCompactThreads)
    compact_kernel(uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                   const int32_t* __restrict__ block_table, const int32_t* __restrict__ prefix_len,
                   const int32_t* __restrict__ path, const int32_t* __restrict__ accept_len, int N,
                   int Hkv, int max_pages, int num_pages, int32_t* __restrict__ new_prefix_len,
                   int32_t* dev_err) {
  constexpr int kVec = D * 2 / 16;                       // 16-byte vectors per row
  __shared__ uint4 s_rows[2][kCompactChunk][kVec];       // [K|V][node][vector]
  __shared__ int s_path[JF_MAX_NODES];
  grid_dependency_wait();
  const int b = blockIdx.x, g = blockIdx.y;
  const int32_t* bt = block_table + static_cast<size_t>(b) * max_pages;
  const int P = prefix_len[b];
  const int a = accept_len[b];
  const int32_t* pth = path + static_cast<size_t>(b) * N;
  int bits = 0;
  if (P < 0 || static_cast<long long>(P) + N > static_cast<long long>(max_pages) * kPage)
    bits |= JF_DEVERR_BAD_PREFIX;
  if (a < 0 || a > N - 1) bits |= JF_DEVERR_BAD_PATH;
  if (bits == 0) {
    for (int k = threadIdx.x; k <= a; k += blockDim.x) {
      const int v = pth[k];
      s_path[k] = v;
      if (k == 0 ? v != 0 : (v <= pth[k - 1] || v >= N)) bits |= JF_DEVERR_BAD_PATH;
      // pages of the source (P + v) and of the destination (P + k)
      const int ps = bt[(P + (v >= 0 && v < N ? v : 0)) / kPage];
      const int pd = bt[(P + k) / kPage];
      if (ps < 0 || ps >= num_pages || pd < 0 || pd >= num_pages) bits |= JF_DEVERR_BAD_PAGE;
    }
  }
  // Every thread learns the union of the bits (uniform branch below).
  const int any_bad = __syncthreads_or(bits != 0);
  if (any_bad) {
    if (bits != 0 && g == 0) report(dev_err, bits);
    if (threadIdx.x == 0 && g == 0) new_prefix_len[b] = P;
    grid_dependents_launch();
    return;
  }
  if (threadIdx.x == 0 && g == 0) new_prefix_len[b] = P + a + 1;
  auto row = [&](uint16_t* cache, int t) -> uint4* {
    const int page = bt[t / kPage];
    return reinterpret_cast<uint4*>(cache + ((static_cast<size_t>(page) * kPage + t % kPage) * Hkv + g) * D);
  };
  for (int k0 = 1; k0 <= a; k0 += kCompactChunk) {
    const int n = min(kCompactChunk, a + 1 - k0);
    // read every source row of the chunk (K and V)
    for (int e = threadIdx.x; e < 2 * n * kVec; e += blockDim.x) {
      const int kv = e / (n * kVec), rem = e % (n * kVec);
      const int k = rem / kVec, q = rem % kVec;
      const int t = P + s_path[k0 + k];
      s_rows[kv][k][q] = row(kv ? v_cache : k_cache, t)[q];
    }
    __syncthreads();
    // then write every destination row
    for (int e = threadIdx.x; e < 2 * n * kVec; e += blockDim.x) {
      const int kv = e / (n * kVec), rem = e % (n * kVec);
      const int k = rem / kVec, q = rem % kVec;
      row(kv ? v_cache : k_cache, P + k0 + k)[q] = s_rows[kv][k][q];
    }
    __syncthreads();
  }
  grid_dependents_launch();
}

}  // namespace
}  // namespace jf

extern "C" jf_status jf_compact_accepted_kv(void* k_cache, void* v_cache, const int32_t* block_table,
                                            const int32_t* prefix_len, const int32_t* path,
                                            const int32_t* accept_len, int32_t B, int32_t N,
                                            int32_t Hkv, int32_t D, int32_t page_size,
                                            int32_t max_pages, int32_t num_pages,
                                            int32_t* new_prefix_len, int32_t* dev_err,
                                            jf_stream_t stream) {
  if (k_cache == nullptr || v_cache == nullptr || block_table == nullptr || prefix_len == nullptr ||
      path == nullptr || accept_len == nullptr || new_prefix_len == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || Hkv < 1 || max_pages < 1 || num_pages < 1) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES || (D != 64 && D != 128) || page_size != jf::kPage) return JF_ERR_UNSUPPORTED;
  if (B > 65535 * 1024 || Hkv > 65535) return JF_ERR_UNSUPPORTED;
  if (!jf::aligned_to(k_cache, 16) || !jf::aligned_to(v_cache, 16)) return JF_ERR_MISALIGNED;
  if (new_prefix_len == prefix_len) return JF_ERR_INVALID_ARGUMENT;
  const dim3 grid(static_cast<unsigned>(B), static_cast<unsigned>(Hkv));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* kc = static_cast<uint16_t*>(k_cache);
  uint16_t* vc = static_cast<uint16_t*>(v_cache);
  const cudaError_t e =
      D == 128 ? jf::launch_pdl(jf::compact_kernel<128>, grid, dim3(jf::kCompactThreads), 0, s, kc, vc,
                                block_table, prefix_len, path, accept_len, N, Hkv, max_pages,
                                num_pages, new_prefix_len, dev_err)
               : jf::launch_pdl(jf::compact_kernel<64>, grid, dim3(jf::kCompactThreads), 0, s, kc, vc,
                                block_table, prefix_len, path, accept_len, N, Hkv, max_pages,
                                num_pages, new_prefix_len, dev_err);
  return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}
