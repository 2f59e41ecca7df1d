// jf_mask.cu -- tree-causal attention mask builder.
//
// JetFlow explainer, technical summary §2 ("Tree-Causal Attention Mask"): each draft node
// sees the prefix and its own ancestors, never descendants or unrelated sibling branches.
// The mask row of node i is the ancestor-or-self set packed LSB-first into W = ceil(N/64)
// uint64 words.
//
// One CTA per sequence.  The sequence's parent array is staged in shared memory and
// validated once; then each thread owns (node i, word w) pairs and walks i's ancestor
// chain, setting the bits that fall into word w and stopping as soon as the chain drops
// below the word's first node (ancestor ids decrease strictly).  The w == 0 walk reaches
// the root, so it also yields depth and position id.  Ragged calls give sequence b only
// n_b nodes: rows of padding nodes (i >= n_b) get zero words and depth = pos = -1.
// Packed calls hold sequence b's n_b nodes at rows cu[b] .. cu[b + 1] - 1 of every
// per-node array, with no padding rows.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kMaskThreads = 256;

__global__ void __launch_bounds__(kMaskThreads)
    tree_mask_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ prefix_len,
                     const int32_t* __restrict__ tree_len, const int32_t* __restrict__ cu,
                     long long T, int N, int W, uint64_t* __restrict__ mask,
                     int32_t* __restrict__ depth, int32_t* __restrict__ pos, int32_t* dev_err) {
  extern __shared__ int32_t s_par[];   // [N]; malformed entries replaced by -1
  grid_dependency_wait();
  const int b = blockIdx.x;
  const SeqSpan sp = seq_span(cu, tree_len, b, N, T);
  if (!sp.ok && threadIdx.x == 0) report(dev_err, JF_DEVERR_BAD_TREE_LEN);
  const int32_t* par = parent + sp.row0;
  const int n = sp.n;                  // nodes of this sequence's tree
  const int rows = sp.rows;            // rows it owns (padding included)
  int bad = 0;
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    if (i >= n) {                      // padding: never read, never an ancestor
      s_par[i] = -1;
      continue;
    }
    int p = par[i];
    const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
    if (!ok) {
      bad = 1;
      p = -1;
    }
    s_par[i] = p;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) report(dev_err, JF_DEVERR_BAD_PARENT);

  const int P = prefix_len[b];
  uint64_t* mrow = mask + sp.row0 * W;
  const int pairs = rows * W;
  for (int e = threadIdx.x; e < pairs; e += blockDim.x) {
    const int i = e / W;
    const int w = e - i * W;
    if (i >= n) {
      mrow[e] = 0ull;
      if (w == 0) {
        if (depth != nullptr) depth[sp.row0 + i] = -1;
        if (pos != nullptr) pos[sp.row0 + i] = -1;
      }
      continue;
    }
    const int lo = w * 64;
    uint64_t word = 0;
    int count = 0;
    int a = i;
    // Bits above the word are skipped; the walk ends below the word's first node unless
    // w == 0, whose walk runs to the root to count the depth.
    while (a >= lo) {
      if (a < lo + 64) word |= 1ull << (a - lo);
      ++count;
      a = s_par[a];
    }
    mrow[e] = word;
    if (w == 0) {
      const int d = count - 1;
      if (depth != nullptr) depth[sp.row0 + i] = d;
      if (pos != nullptr) pos[sp.row0 + i] = P + d;
    }
  }
  grid_dependents_launch();
}

}  // namespace
}  // namespace jf

namespace {

jf_status build_mask(const int32_t* parent, const int32_t* prefix_len, const int32_t* tree_len,
                     const int32_t* cu, int32_t T, int32_t B, int32_t N, uint64_t* mask,
                     int32_t* depth, int32_t* pos, int32_t* dev_err, jf_stream_t stream) {
  if (parent == nullptr || prefix_len == nullptr || mask == nullptr) return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1) return JF_ERR_INVALID_ARGUMENT;
  if (cu != nullptr && T < 1) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES) return JF_ERR_UNSUPPORTED;
  if (!jf::aligned_to(mask, 8)) return JF_ERR_MISALIGNED;
  const int W = (N + 63) / 64;
  const size_t smem = sizeof(int32_t) * static_cast<size_t>(N);
  const cudaError_t e = jf::launch_pdl(jf::tree_mask_kernel, dim3(B), dim3(jf::kMaskThreads), smem,
                                       reinterpret_cast<cudaStream_t>(stream), parent,
                                       prefix_len, tree_len, cu, static_cast<long long>(T), N, W,
                                       mask, depth, pos, dev_err);
  return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

}  // namespace

extern "C" jf_status jf_build_tree_mask(const int32_t* parent, const int32_t* prefix_len,
                                        int32_t B, int32_t N, uint64_t* mask, int32_t* depth,
                                        int32_t* pos, int32_t* dev_err, jf_stream_t stream) {
  return build_mask(parent, prefix_len, nullptr, nullptr, 0, B, N, mask, depth, pos, dev_err,
                    stream);
}

extern "C" jf_status jf_build_tree_mask_ragged(const int32_t* parent, const int32_t* prefix_len,
                                               const int32_t* tree_len, int32_t B, int32_t N,
                                               uint64_t* mask, int32_t* depth, int32_t* pos,
                                               int32_t* dev_err, jf_stream_t stream) {
  if (tree_len == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return build_mask(parent, prefix_len, tree_len, nullptr, 0, B, N, mask, depth, pos, dev_err,
                    stream);
}

extern "C" jf_status jf_build_tree_mask_packed(const int32_t* parent, const int32_t* prefix_len,
                                               const int32_t* cu_seqlens, int32_t B, int32_t N_max,
                                               int32_t T, uint64_t* mask, int32_t* depth,
                                               int32_t* pos, int32_t* dev_err, jf_stream_t stream) {
  if (cu_seqlens == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return build_mask(parent, prefix_len, nullptr, cu_seqlens, T, B, N_max, mask, depth, pos,
                    dev_err, stream);
}
