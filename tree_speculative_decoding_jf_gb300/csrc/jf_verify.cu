// jf_verify.cu -- greedy tree verification: per-node vocabulary argmax, then the longest
// accepted root path.
//
// The target model checks all drafted nodes in one pass and keeps the drafted prefix it
// agrees with (qxai.app commentary on JetFlow, "まず、何が問題なのか"; the explainer's §4
// counts the accepted tokens tau).  Greedy reading: child c of p is accepted iff
// draft[c] == argmax(logits[p]).
//
// Kernel 1 (HBM-bound): each CTA scans one chunk of one logits row with 16-byte loads and
// writes a packed 64-bit key (order-preserving value bits << 32 | ~index) into the
// workspace; max over keys gives the largest value and, among equal values, the smallest
// index.  Chunks per row are chosen so that rows x chunks fills the GPU.
// Kernel 2 (one CTA per sequence): merges the chunk keys into argmax (shared atomicMax),
// finds depths by pointer jumping, computes accepted-subtree lengths level by level from
// the deepest level up with shared-memory atomicMax on (len + 1) << 16 | (0xFFFF - child),
// and walks the best children from the root.  Trees of at most 64 nodes take a one-warp
// version of the same steps with no block barriers.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxUnroll = 4;
constexpr int kWalkThreads = 512;
constexpr int kMinChunkElems = 8192;

// Order-preserving map of a float to uint32 (larger float -> larger integer); -0 -> +0.
__device__ __forceinline__ uint32_t ordered_bits(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t pack_key(float v, int idx) {
  return (static_cast<uint64_t>(ordered_bits(v)) << 32) |
         static_cast<uint64_t>(~static_cast<uint32_t>(idx));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<uint16_t>(uint16_t x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }

struct Best {
  float v;
  int i;
  __device__ __forceinline__ void take(float x, int idx) {
    if (x > v) { v = x; i = idx; }   // indices arrive in increasing order per thread
  }
};

__device__ __forceinline__ void take_vec(Best& b, uint4 q, int idx, uint16_t) {
  b.take(bf16_lo(q.x), idx + 0); b.take(bf16_hi(q.x), idx + 1);
  b.take(bf16_lo(q.y), idx + 2); b.take(bf16_hi(q.y), idx + 3);
  b.take(bf16_lo(q.z), idx + 4); b.take(bf16_hi(q.z), idx + 5);
  b.take(bf16_lo(q.w), idx + 6); b.take(bf16_hi(q.w), idx + 7);
}
__device__ __forceinline__ void take_vec(Best& b, uint4 q, int idx, float) {
  b.take(__uint_as_float(q.x), idx + 0); b.take(__uint_as_float(q.y), idx + 1);
  b.take(__uint_as_float(q.z), idx + 2); b.take(__uint_as_float(q.w), idx + 3);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t other = __shfl_xor_sync(0xffffffffu, k, o);
    k = other > k ? other : k;
  }
  return k;
}

template <typename T>
__global__ void __launch_bounds__(kArgmaxThreads)
    argmax_chunk_kernel(const T* __restrict__ logits, long long V, int chunks, int chunk_len,
                        uint64_t* __restrict__ part, int idx_off) {
  constexpr int kVec = 16 / sizeof(T);
  grid_dependency_wait();
  const long long row = blockIdx.x / chunks;
  const int c = blockIdx.x - static_cast<int>(row * chunks);
  const long long s = static_cast<long long>(c) * chunk_len;
  const long long e = min(V, s + chunk_len);
  const T* base = logits + row * V;

  // Split [s, e) into a scalar head up to the first 16-byte boundary, a vector body and
  // a scalar tail; every thread sees its indices in increasing order.
  const uintptr_t addr = reinterpret_cast<uintptr_t>(base + s);
  long long head = ((16 - (addr & 15)) & 15) / sizeof(T);
  if (head > e - s) head = e - s;
  const long long body0 = s + head;
  const long long nvec = (e - body0) / kVec;
  const long long body1 = body0 + nvec * kVec;

  Best best{-INFINITY, -1};
  int first = -1;   // first index this thread looked at (for all -inf rows)
  if (threadIdx.x < head) {
    const long long idx = s + threadIdx.x;
    best.take(to_f<T>(base[idx]), static_cast<int>(idx));
    first = static_cast<int>(idx);
  }
  const uint4* vb = reinterpret_cast<const uint4*>(base + body0);
  for (long long v0 = threadIdx.x; v0 < nvec; v0 += kArgmaxThreads * kArgmaxUnroll) {
    uint4 q[kArgmaxUnroll];
#pragma unroll
    for (int u = 0; u < kArgmaxUnroll; ++u) {
      const long long vi = v0 + static_cast<long long>(u) * kArgmaxThreads;
      if (vi < nvec) q[u] = __ldcs(vb + vi);
    }
#pragma unroll
    for (int u = 0; u < kArgmaxUnroll; ++u) {
      const long long vi = v0 + static_cast<long long>(u) * kArgmaxThreads;
      if (vi < nvec) {
        const int idx = static_cast<int>(body0 + vi * kVec);
        if (first < 0) first = idx;
        take_vec(best, q[u], idx, T());
      }
    }
  }
  if (threadIdx.x < e - body1) {
    const long long idx = body1 + threadIdx.x;
    best.take(to_f<T>(base[idx]), static_cast<int>(idx));
    if (first < 0) first = static_cast<int>(idx);
  }
  if (best.i < 0 && first >= 0) best.i = first;   // every value it saw was -inf
  // keys carry vocabulary indices: the row's own plus idx_off (a shard's first token)
  uint64_t key = best.i < 0 ? 0ull : pack_key(best.v, best.i + idx_off);

  __shared__ uint64_t s_keys[kArgmaxThreads / 32];
  key = warp_max_u64(key);
  if ((threadIdx.x & 31) == 0) s_keys[threadIdx.x >> 5] = key;
  __syncthreads();
  if (threadIdx.x < 32) {
    key = threadIdx.x < kArgmaxThreads / 32 ? s_keys[threadIdx.x] : 0ull;
    key = warp_max_u64(key);
    if (threadIdx.x == 0) part[blockIdx.x] = key;
  }
  grid_dependents_launch();
}

// Threads of a walk block: the tree rounded up to whole warps, at least four warps (the
// chunk-key merge wants loads in flight) and at most kWalkThreads, so small trees pay for
// cheap barriers.  With fewer than kWalkThreads threads, N fits in one pass of the block.
inline int walk_threads(int N) { return std::min(kWalkThreads, std::max(128, (N + 31) / 32 * 32)); }

__global__ void __launch_bounds__(kWalkThreads)
    tree_walk_kernel(const uint64_t* __restrict__ part, int chunks,
                     const int32_t* __restrict__ draft, const int32_t* __restrict__ parent,
                     const int32_t* __restrict__ tree_len, const int32_t* __restrict__ cu,
                     long long T, int N, int V, int32_t* __restrict__ argmax_out,
                     int32_t* __restrict__ accept_len, int32_t* __restrict__ path,
                     int32_t* __restrict__ bonus, int32_t* dev_err) {
  extern __shared__ uint64_t sm64[];
  unsigned long long* s_best = reinterpret_cast<unsigned long long*>(sm64);   // [N] best key
  int32_t* sm = reinterpret_cast<int32_t*>(sm64 + N);
  int32_t* s_par = sm;            // [N] parent, malformed -> -1
  int32_t* s_am = s_par + N;      // [N] argmax
  int32_t* s_dep = s_am + N;      // [N] depth (pointer jumping)
  int32_t* s_anc = s_dep + N;     // [N] ancestor pointer (pointer jumping)
  uint32_t* s_key = reinterpret_cast<uint32_t*>(s_anc + N);   // [N] best accepted child
  int32_t* s_path = reinterpret_cast<int32_t*>(s_key + N);    // [N]
  int32_t* s_draft = s_path + N;                               // [N]
  __shared__ int s_flag;
  __shared__ int s_len;

  grid_dependency_wait();
  const int b = blockIdx.x;
  // Ragged calls: nodes >= nt are padding, never read and never accepted.  Packed calls:
  // the sequence's rows start at cu[b] and it owns no padding rows.
  const SeqSpan sp = seq_span(cu, tree_len, b, N, T);
  if (!sp.ok && threadIdx.x == 0) report(dev_err, JF_DEVERR_BAD_TREE_LEN);
  const size_t rb = static_cast<size_t>(sp.row0);
  const int nt = sp.n;
  const int rows = sp.rows;
  // The block is sized to the tree (threadIdx.x + k * blockDim.x covers every node for
  // k < kPer).  Parents and drafts are requested first and stay in flight while the
  // chunk keys are merged, so both arrive in one memory round trip.
  constexpr int kPer = (JF_MAX_NODES + kWalkThreads - 1) / kWalkThreads;
  int r_par[kPer], r_draft[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < nt) {
      r_par[k] = parent[rb + i];
      r_draft[k] = draft[rb + i];
    }
  }
  // Chunk keys of every row, all loads in flight together: (row, chunk) pairs spread over
  // the block, combined per row with a shared-memory 64-bit atomicMax.
  for (int i = threadIdx.x; i < N; i += blockDim.x) s_best[i] = 0ull;
  __syncthreads();
  {
    // Keys are fetched kKeyBatch per thread before any is merged, so a block of 128
    // threads has 1024 of them in flight per round trip.
    constexpr int kKeyBatch = 8;
    const int total = rows * chunks;
    const uint64_t* pk = part + rb * chunks;
    for (int e0 = threadIdx.x; e0 < total; e0 += blockDim.x * kKeyBatch) {
      uint64_t kv[kKeyBatch];
#pragma unroll
      for (int u = 0; u < kKeyBatch; ++u) {
        const int e = e0 + u * static_cast<int>(blockDim.x);
        kv[u] = e < total ? pk[e] : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kKeyBatch; ++u) {
        const int e = e0 + u * static_cast<int>(blockDim.x);
        if (e < total) atomicMax(&s_best[e / chunks], kv[u]);
      }
    }
  }
  int bad_parent = 0, bad_token = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < N) {
      int p = i < nt ? r_par[k] : -1;
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
      if (!ok && i < nt) bad_parent = 1;
      if (!ok) p = -1;
      s_par[i] = p;
      s_anc[i] = p;
      s_dep[i] = p >= 0 ? 1 : 0;
      s_key[i] = 0u;
      const int d = i < nt ? r_draft[k] : -1;
      s_draft[i] = d;
      if (i > 0 && i < nt && (d < 0 || d >= V)) bad_token = 1;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int am = static_cast<int>(~static_cast<uint32_t>(s_best[i] & 0xFFFFFFFFull));
    s_am[i] = am;
    if (argmax_out != nullptr && i < rows) argmax_out[rb + i] = am;
  }
  bad_parent = __syncthreads_or(bad_parent);
  bad_token = __syncthreads_or(bad_token);
  if (threadIdx.x == 0) {
    if (bad_parent) report(dev_err, JF_DEVERR_BAD_PARENT);
    if (bad_token) report(dev_err, JF_DEVERR_BAD_TOKEN);
  }

  // Depth by pointer jumping: dep[i] += dep[anc[i]], anc[i] = anc[anc[i]].
  for (int round = 0; round < 32; ++round) {
    int nd[kPer], na[kPer];
    int any = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < N) {
        const int a = s_anc[i];
        nd[k] = s_dep[i];
        na[k] = a;
        if (a >= 0) {
          nd[k] += s_dep[a];
          na[k] = s_anc[a];
          any = 1;
        }
      }
    }
    if (!__syncthreads_or(any)) break;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < N) { s_dep[i] = nd[k]; s_anc[i] = na[k]; }
    }
    __syncthreads();
  }
  int maxd = 0;
  for (int i = threadIdx.x; i < N; i += blockDim.x) maxd = max(maxd, s_dep[i]);
  if (threadIdx.x == 0) s_flag = 0;
  __syncthreads();
  atomicMax(&s_flag, maxd);
  __syncthreads();
  maxd = s_flag;

  // Accepted-subtree lengths, deepest level first: a node's key is final once every
  // node one level below has been processed.
  for (int d = maxd; d >= 1; --d) {
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
      const int p = s_par[i];
      if (s_dep[i] == d && p >= 0 && s_draft[i] == s_am[p]) {
        const uint32_t len = (s_key[i] >> 16) + 1u;
        atomicMax(&s_key[p], (len << 16) | static_cast<uint32_t>(0xFFFF - i));
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int cur = 0, n = 0;
    s_path[0] = 0;
    while (s_key[cur] != 0u && n < N - 1) {
      cur = 0xFFFF - static_cast<int>(s_key[cur] & 0xFFFFu);
      s_path[++n] = cur;
    }
    s_len = n;
    accept_len[b] = n;
    bonus[b] = s_am[cur];
  }
  __syncthreads();
  const int n = s_len;
  for (int k = threadIdx.x; k < N; k += blockDim.x)
    path[static_cast<size_t>(b) * N + k] = k <= n ? s_path[k] : -1;
  grid_dependents_launch();
}

// Small trees (N <= 64) in one warp: no block barriers, so a deep chain costs a few dozen
// cycles per level instead of a __syncthreads each.  Lane q owns nodes q and q + 32.  Every
// chunk key of a lane's rows is requested before any is merged (at most kSmallWalkKeys
// loads in flight per lane), so the merge costs one memory round trip.  Depths come from
// pointer jumping through shared memory, accepted-subtree lengths from shared-memory
// atomicMax level by level (deepest first, a __syncwarp between levels), then lane 0
// follows the best children from the root.
constexpr int kSmallWalkNodes = 64;
constexpr int kSmallWalkKeys = 48;    // keys per lane: 48 chunks of one row, or 24 of two

inline bool small_walk_fits(int N, int chunks) {
  return N <= kSmallWalkNodes &&
         (N <= 32 ? chunks <= kSmallWalkKeys : chunks <= kSmallWalkKeys / 2);
}

__global__ void __launch_bounds__(32)
    tree_walk_small_kernel(const uint64_t* __restrict__ part, int chunks,
                           const int32_t* __restrict__ draft, const int32_t* __restrict__ parent,
                           const int32_t* __restrict__ tree_len, const int32_t* __restrict__ cu,
                           long long T, int N, int V,
                           int32_t* __restrict__ argmax_out, int32_t* __restrict__ accept_len,
                           int32_t* __restrict__ path, int32_t* __restrict__ bonus,
                           int32_t* dev_err) {
  constexpr int H = kSmallWalkKeys / 2;
  __shared__ int s_par[kSmallWalkNodes], s_am[kSmallWalkNodes], s_dep[kSmallWalkNodes],
      s_anc[kSmallWalkNodes], s_path[kSmallWalkNodes];
  __shared__ uint32_t s_key[kSmallWalkNodes];
  grid_dependency_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  const SeqSpan sp = seq_span(cu, tree_len, b, N, T);
  if (!sp.ok && lane == 0) report(dev_err, JF_DEVERR_BAD_TREE_LEN);
  const size_t rb = static_cast<size_t>(sp.row0);
  const int nt = sp.n;
  const int rows = sp.rows;
  const bool two = N > 32;                          // two rows per lane
  int r_par[2] = {-1, -1}, r_draft[2] = {-1, -1};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < nt) {
      r_par[k] = parent[rb + i];
      r_draft[k] = draft[rb + i];
    }
  }
  // One lane's keys: row lane's chunks 0..47, or rows lane and lane + 32 with 24 each.
  uint64_t kv[kSmallWalkKeys];
#pragma unroll
  for (int u = 0; u < kSmallWalkKeys; ++u) {
    const int i = two ? lane + 32 * (u / H) : lane;
    const int c = two ? u % H : u;
    kv[u] = (i < rows && c < chunks) ? part[(rb + i) * chunks + c] : 0ull;
  }
  uint64_t best[2] = {0ull, 0ull};
#pragma unroll
  for (int u = 0; u < kSmallWalkKeys; ++u) {
    const int k = two ? u / H : 0;
    best[k] = kv[u] > best[k] ? kv[u] : best[k];
  }
  int bad_parent = 0, bad_token = 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < N) {
      const int am = static_cast<int>(~static_cast<uint32_t>(best[k] & 0xFFFFFFFFull));
      s_am[i] = am;
      if (argmax_out != nullptr && i < rows) argmax_out[rb + i] = am;
      int p = i < nt ? r_par[k] : -1;
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
      if (!ok && i < nt) bad_parent = 1;
      if (!ok) p = -1;
      s_par[i] = p;
      s_anc[i] = p;
      s_dep[i] = p >= 0 ? 1 : 0;
      s_key[i] = 0u;
      if (i > 0 && i < nt && (r_draft[k] < 0 || r_draft[k] >= V)) bad_token = 1;
    }
  }
  if (__any_sync(0xffffffffu, bad_parent) && lane == 0) report(dev_err, JF_DEVERR_BAD_PARENT);
  if (__any_sync(0xffffffffu, bad_token) && lane == 0) report(dev_err, JF_DEVERR_BAD_TOKEN);
  __syncwarp();
  // depth by pointer jumping: dep[i] += dep[anc[i]], anc[i] = anc[anc[i]]
  for (int round = 0; round < 7; ++round) {
    int nd[2], na[2], any = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      nd[k] = 0; na[k] = -1;
      if (i < N) {
        const int a = s_anc[i];
        nd[k] = s_dep[i];
        na[k] = a;
        if (a >= 0) {
          nd[k] += s_dep[a];
          na[k] = s_anc[a];
          any = 1;
        }
      }
    }
    if (!__any_sync(0xffffffffu, any)) break;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < N) { s_dep[i] = nd[k]; s_anc[i] = na[k]; }
    }
    __syncwarp();
  }
  int maxd = 0;
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (lane + 32 * k < N) maxd = max(maxd, s_dep[lane + 32 * k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxd = max(maxd, __shfl_xor_sync(0xffffffffu, maxd, o));
  // accepted-subtree lengths, deepest level first
  int acc[2], dep[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    const int p = i < N ? s_par[i] : -1;
    dep[k] = i < N ? s_dep[i] : -1;
    acc[k] = (p >= 0 && i < nt && r_draft[k] == s_am[p]) ? 1 : 0;
  }
  for (int d = maxd; d >= 1; --d) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (dep[k] == d && acc[k]) {
        const uint32_t len = (s_key[i] >> 16) + 1u;
        atomicMax(&s_key[s_par[i]], (len << 16) | static_cast<uint32_t>(0xFFFF - i));
      }
    }
    __syncwarp();
  }
  if (lane == 0) {
    int cur = 0, n = 0;
    s_path[0] = 0;
    while (s_key[cur] != 0u && n < N - 1) {
      cur = 0xFFFF - static_cast<int>(s_key[cur] & 0xFFFFu);
      s_path[++n] = cur;
    }
    s_dep[0] = n;                     // reused: the accepted length for the other lanes
    accept_len[b] = n;
    bonus[b] = s_am[cur];
  }
  __syncwarp();
  const int n = s_dep[0];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = lane + 32 * k;
    if (i < N) path[static_cast<size_t>(b) * N + i] = i <= n ? s_path[i] : -1;
  }
  grid_dependents_launch();
}

struct VerifyPlan {
  int chunks;
  int chunk_len;
};

// Chunks per logit row for `rows` rows of V logits.
bool plan_verify_rows(long long rows, int V, VerifyPlan* p) {
  if (rows < 1 || V < 1) return false;
  const int sms = current_sm_count() > 0 ? current_sm_count() : 148;
  const long long target = static_cast<long long>(sms) * 4;   // CTAs to keep HBM busy
  long long c = (target + rows - 1) / rows;
  const long long cmax = std::max<long long>(1, (V + kMinChunkElems - 1) / kMinChunkElems);
  c = std::min(std::max<long long>(c, 1), cmax);
  long long len = (V + c - 1) / c;
  len = (len + 7) / 8 * 8;
  c = (V + len - 1) / len;
  p->chunks = static_cast<int>(c);
  p->chunk_len = static_cast<int>(len);
  return true;
}

bool plan_verify(int B, int N, int V, VerifyPlan* p) {
  if (B < 1 || N < 1 || N > JF_MAX_NODES || V < 1) return false;
  return plan_verify_rows(static_cast<long long>(B) * N, V, p);
}

// Launches the walk over the argmax keys in `part`: one warp per sequence for small trees,
// else the block-wide walk.  Both are programmatic dependents of the argmax grid.
// Packed calls pass cu (cumulative node counts) and T = cu[B]; others nullptr and 0.
jf_status launch_walk(const uint64_t* part, int chunks, const int32_t* draft,
                      const int32_t* parent, const int32_t* tree_len, int B, int N, int V,
                      int32_t* argmax, int32_t* accept_len, int32_t* path, int32_t* bonus,
                      int32_t* dev_err, cudaStream_t s, const int32_t* cu = nullptr,
                      long long T = 0) {
  cudaError_t e;
  if (small_walk_fits(N, chunks)) {
    e = launch_pdl(tree_walk_small_kernel, dim3(B), dim3(32), 0, s, part, chunks, draft, parent,
                   tree_len, cu, T, N, V, argmax, accept_len, path, bonus, dev_err);
  } else {
    const size_t smem = static_cast<size_t>(N) * (7 * sizeof(int32_t) + sizeof(uint64_t));
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(tree_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return JF_ERR_CUDA;
    e = launch_pdl(tree_walk_kernel, dim3(B), dim3(walk_threads(N)), smem, s, part, chunks, draft,
                   parent, tree_len, cu, T, N, V, argmax, accept_len, path, bonus, dev_err);
  }
  return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

// Chunks of the stochastic verification: fixed 8192-logit chunks, so the bonus draw scans
// one chunk of 32 logits per thread (the argmax plan may give a whole row to one CTA).
constexpr int kSampleChunk = 8192;

inline int sampled_chunks(int V) { return (V + kSampleChunk - 1) / kSampleChunk; }

}  // namespace
}  // namespace jf

extern "C" size_t jf_tree_verify_workspace_size(int32_t B, int32_t N, int32_t V) {
  jf::VerifyPlan p;
  if (!jf::plan_verify(B, N, V, &p)) return static_cast<size_t>(-1);
  const size_t rows = static_cast<size_t>(B) * N;
  return std::max(rows * p.chunks * sizeof(uint64_t),                       // argmax keys
                  rows * jf::sampled_chunks(V) * sizeof(float2));          // sampling stats
}

namespace {

// Packed calls (cu != nullptr) hold T = cu[B] logit rows; the others B * N.
jf_status tree_verify_call(const void* logits, int32_t dtype, const int32_t* draft,
                           const int32_t* parent, const int32_t* tree_len, const int32_t* cu,
                           int32_t T, int32_t B, int32_t N, int32_t V, int32_t* argmax,
                           int32_t* accept_len, int32_t* path, int32_t* bonus, void* workspace,
                           size_t workspace_bytes, int32_t* dev_err, jf_stream_t stream) {
  if (logits == nullptr || draft == nullptr || parent == nullptr || accept_len == nullptr ||
      path == nullptr || bonus == nullptr || workspace == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (dtype != JF_DTYPE_BF16 && dtype != JF_DTYPE_F32) return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || V < 1) return JF_ERR_INVALID_ARGUMENT;
  if (cu != nullptr && T < 1) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES) return JF_ERR_UNSUPPORTED;
  const long long rows = cu != nullptr ? static_cast<long long>(T) : static_cast<long long>(B) * N;
  jf::VerifyPlan p;
  if (!jf::plan_verify_rows(rows, V, &p)) return JF_ERR_UNSUPPORTED;
  const size_t need = static_cast<size_t>(rows) * p.chunks * sizeof(uint64_t);
  if (workspace_bytes < need) return JF_ERR_WORKSPACE_TOO_SMALL;
  if (!jf::aligned_to(workspace, 8)) return JF_ERR_MISALIGNED;
  if (!jf::aligned_to(logits, dtype == JF_DTYPE_BF16 ? 2 : 4)) return JF_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint64_t* part = static_cast<uint64_t*>(workspace);
  const long long grid = rows * p.chunks;
  if (grid > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  const long long Vl = V;
  const cudaError_t ea =
      dtype == JF_DTYPE_BF16
          ? jf::launch_pdl(jf::argmax_chunk_kernel<uint16_t>, dim3(static_cast<unsigned>(grid)),
                           dim3(jf::kArgmaxThreads), 0, s, static_cast<const uint16_t*>(logits),
                           Vl, p.chunks, p.chunk_len, part, 0)
          : jf::launch_pdl(jf::argmax_chunk_kernel<float>, dim3(static_cast<unsigned>(grid)),
                           dim3(jf::kArgmaxThreads), 0, s, static_cast<const float*>(logits), Vl,
                           p.chunks, p.chunk_len, part, 0);
  if (ea != cudaSuccess) return JF_ERR_CUDA;
  return jf::launch_walk(part, p.chunks, draft, parent, tree_len, B, N, V, argmax, accept_len, path,
                         bonus, dev_err, s, cu, T);
}

}  // namespace

extern "C" jf_status jf_tree_verify(const void* logits, int32_t dtype, const int32_t* draft,
                                    const int32_t* parent, int32_t B, int32_t N, int32_t V,
                                    int32_t* argmax, int32_t* accept_len, int32_t* path,
                                    int32_t* bonus, void* workspace, size_t workspace_bytes,
                                    int32_t* dev_err, jf_stream_t stream) {
  return tree_verify_call(logits, dtype, draft, parent, nullptr, nullptr, 0, B, N, V, argmax,
                          accept_len, path, bonus, workspace, workspace_bytes, dev_err, stream);
}

extern "C" jf_status jf_tree_verify_ragged(const void* logits, int32_t dtype, const int32_t* draft,
                                           const int32_t* parent, const int32_t* tree_len,
                                           int32_t B, int32_t N, int32_t V, int32_t* argmax,
                                           int32_t* accept_len, int32_t* path, int32_t* bonus,
                                           void* workspace, size_t workspace_bytes,
                                           int32_t* dev_err, jf_stream_t stream) {
  if (tree_len == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return tree_verify_call(logits, dtype, draft, parent, tree_len, nullptr, 0, B, N, V, argmax,
                          accept_len, path, bonus, workspace, workspace_bytes, dev_err, stream);
}

extern "C" size_t jf_tree_verify_packed_workspace_size(int32_t T, int32_t V) {
  jf::VerifyPlan p;
  if (T < 1 || !jf::plan_verify_rows(T, V, &p)) return static_cast<size_t>(-1);
  return std::max(static_cast<size_t>(T) * p.chunks * sizeof(uint64_t),              // argmax keys
                  static_cast<size_t>(T) * jf::sampled_chunks(V) * sizeof(float2));  // sampling stats
}

extern "C" jf_status jf_tree_verify_packed(const void* logits, int32_t dtype, const int32_t* draft,
                                           const int32_t* parent, const int32_t* cu_seqlens,
                                           int32_t B, int32_t N_max, int32_t T, int32_t V,
                                           int32_t* argmax, int32_t* accept_len, int32_t* path,
                                           int32_t* bonus, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_err,
                                           jf_stream_t stream) {
  if (cu_seqlens == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return tree_verify_call(logits, dtype, draft, parent, nullptr, cu_seqlens, T, B, N_max, V,
                          argmax, accept_len, path, bonus, workspace, workspace_bytes, dev_err,
                          stream);
}

// ------------------------------------------------------------------------ allocation-free
// jf_tree_verify_static: the argmax partial keys live in a fixed array compiled into the
// library instead of a caller workspace.  Host code only ever passes the array's device
// address (looked up per device); the symbol itself is a host-side stand-in.
static __device__ __align__(256) uint64_t g_verify_static_scratch[JF_VERIFY_STATIC_SCRATCH_KEYS];

namespace jf {
namespace {

// Device address of g_verify_static_scratch on the current device, looked up once per
// device with that device current; null if the lookup fails.
uint64_t* verify_static_scratch() {
  static std::mutex mu;
  static uint64_t* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<uint64_t*>(p);
  }
  return addr[dev];
}

}  // namespace
}  // namespace jf

extern "C" jf_status jf_tree_verify_static(const void* logits, int32_t dtype,
                                           const int32_t* draft, const int32_t* parent,
                                           int32_t B, int32_t N, int32_t V, int32_t* argmax,
                                           int32_t* accept_len, int32_t* path, int32_t* bonus,
                                           int32_t* dev_err, jf_stream_t stream) {
  if (logits == nullptr || draft == nullptr || parent == nullptr || accept_len == nullptr ||
      path == nullptr || bonus == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (dtype != JF_DTYPE_BF16 && dtype != JF_DTYPE_F32) return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || V < 1) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES) return JF_ERR_UNSUPPORTED;
  jf::VerifyPlan p;
  if (!jf::plan_verify(B, N, V, &p)) return JF_ERR_UNSUPPORTED;
  const unsigned long long keys = static_cast<unsigned long long>(B) * N * p.chunks;
  if (keys > JF_VERIFY_STATIC_SCRATCH_KEYS) return JF_ERR_SCRATCH_CAPACITY;
  if (!jf::aligned_to(logits, dtype == JF_DTYPE_BF16 ? 2 : 4)) return JF_ERR_MISALIGNED;
  uint64_t* part = jf::verify_static_scratch();
  if (part == nullptr) return JF_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(keys);
  const long long Vl = V;
  const cudaError_t ea =
      dtype == JF_DTYPE_BF16
          ? jf::launch_pdl(jf::argmax_chunk_kernel<uint16_t>, dim3(grid), dim3(jf::kArgmaxThreads),
                           0, s, static_cast<const uint16_t*>(logits), Vl, p.chunks, p.chunk_len,
                           part, 0)
          : jf::launch_pdl(jf::argmax_chunk_kernel<float>, dim3(grid), dim3(jf::kArgmaxThreads), 0,
                           s, static_cast<const float*>(logits), Vl, p.chunks, p.chunk_len, part, 0);
  if (ea != cudaSuccess) return JF_ERR_CUDA;
  return jf::launch_walk(part, p.chunks, draft, parent, nullptr, B, N, V, argmax, accept_len, path,
                         bonus, dev_err, s);
}

// ------------------------------------------------------------- vocabulary-sharded verify
// A target model whose output layer is split by vocabulary gives each GPU the logits of
// one vocabulary range.  The argmax keys (value, ~global index) of every range are
// exchanged (an all-gather the caller runs) and the walk runs on their maximum: the keys
// order by value and then by lower index, so the maximum over all ranges is the
// unsharded argmax.

namespace jf {
namespace {

// keys [S][rows][chunks] -> merged [rows]: one thread per row.
__global__ void __launch_bounds__(256)
    merge_shard_keys_kernel(const uint64_t* __restrict__ keys, int S, long long rows, int chunks,
                            uint64_t* __restrict__ merged) {
  grid_dependency_wait();
  const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r < rows) {
    uint64_t k = 0ull;
    for (int sh = 0; sh < S; ++sh)
      for (int c = 0; c < chunks; ++c) {
        const uint64_t v = keys[(static_cast<long long>(sh) * rows + r) * chunks + c];
        k = v > k ? v : k;
      }
    merged[r] = k;
  }
  grid_dependents_launch();
}

}  // namespace
}  // namespace jf

extern "C" int32_t jf_tree_verify_shard_chunks(int32_t B, int32_t N, int32_t V_shard) {
  jf::VerifyPlan p;
  if (!jf::plan_verify(B, N, V_shard, &p)) return -1;
  return p.chunks;
}

extern "C" jf_status jf_tree_verify_shard_keys(const void* logits_shard, int32_t dtype, int32_t B,
                                               int32_t N, int32_t V_shard, int32_t vocab_offset,
                                               int32_t chunks, uint64_t* keys,
                                               jf_stream_t stream) {
  if (logits_shard == nullptr || keys == nullptr) return JF_ERR_INVALID_ARGUMENT;
  if (dtype != JF_DTYPE_BF16 && dtype != JF_DTYPE_F32) return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || V_shard < 1 || chunks < 1 || vocab_offset < 0) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES) return JF_ERR_UNSUPPORTED;
  if (static_cast<long long>(vocab_offset) + V_shard > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  if (!jf::aligned_to(keys, 8)) return JF_ERR_MISALIGNED;
  if (!jf::aligned_to(logits_shard, dtype == JF_DTYPE_BF16 ? 2 : 4)) return JF_ERR_MISALIGNED;
  // chunks of at least 8 logits; trailing chunks past the shard end write key 0
  long long len = (static_cast<long long>(V_shard) + chunks - 1) / chunks;
  len = (len + 7) / 8 * 8;
  const long long grid = static_cast<long long>(B) * N * chunks;
  if (grid > 0x7FFFFFFFll || len > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long Vl = V_shard;
  const int cl = static_cast<int>(len);
  const cudaError_t e =
      dtype == JF_DTYPE_BF16
          ? jf::launch_pdl(jf::argmax_chunk_kernel<uint16_t>, dim3(static_cast<unsigned>(grid)),
                           dim3(jf::kArgmaxThreads), 0, s, static_cast<const uint16_t*>(logits_shard),
                           Vl, chunks, cl, keys, vocab_offset)
          : jf::launch_pdl(jf::argmax_chunk_kernel<float>, dim3(static_cast<unsigned>(grid)),
                           dim3(jf::kArgmaxThreads), 0, s, static_cast<const float*>(logits_shard),
                           Vl, chunks, cl, keys, vocab_offset);
  return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

extern "C" jf_status jf_tree_verify_from_keys(const uint64_t* keys, int32_t S, int32_t chunks,
                                              const int32_t* draft, const int32_t* parent, int32_t B,
                                              int32_t N, int32_t V, int32_t* argmax,
                                              int32_t* accept_len, int32_t* path, int32_t* bonus,
                                              void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, jf_stream_t stream) {
  if (keys == nullptr || draft == nullptr || parent == nullptr || accept_len == nullptr ||
      path == nullptr || bonus == nullptr || workspace == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (S < 1 || chunks < 1 || B < 1 || N < 1 || V < 1) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES) return JF_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * N;
  if (workspace_bytes < static_cast<size_t>(rows) * sizeof(uint64_t)) return JF_ERR_WORKSPACE_TOO_SMALL;
  if (!jf::aligned_to(workspace, 8) || !jf::aligned_to(keys, 8)) return JF_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint64_t* merged = static_cast<uint64_t*>(workspace);
  const long long blocks = (rows + 255) / 256;
  if (blocks > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  if (jf::launch_pdl(jf::merge_shard_keys_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                     keys, static_cast<int>(S), rows, static_cast<int>(chunks), merged) != cudaSuccess)
    return JF_ERR_CUDA;
  return jf::launch_walk(merged, 1, draft, parent, nullptr, B, N, V, argmax, accept_len, path, bonus,
                         dev_err, s);
}

// ------------------------------------------------------------------------ stochastic verify
// jf_tree_verify_sampled: lossless acceptance instead of argmax matching.  The target
// distribution of node u is p = softmax(logits[u] / T).  Children of u are tested in
// increasing node id: child c with token x is accepted iff uniform[c] * R < p(x), R the
// probability mass left after removing the tokens rejected so far at u (a point-mass
// draft's residual: SpecInfer's multi-step speculative sampling for deterministic
// candidates); with no acceptance the bonus token is drawn from the residual by inverse
// CDF with bonus_uniform.  Every emitted token then follows the target distribution.
//
// Kernel 1 (HBM-bound, one warp per (row, 8192-logit chunk)): the chunk's largest logit
// m_c and the Kahan-compensated sum s_c of exp((x - m_c) / T).  Kernel 2 (one CTA per
// sequence): per visited node, M = max_c m_c and Z = sum_c s_c exp((m_c - M) / T) (fp64
// sums), the node's children in id order (a block scan over contiguous node ranges), their
// target probabilities computed in parallel, then one thread takes the ordered acceptance
// decisions from them in fp64.  The bonus draw finds the first chunk where the residual CDF
// crosses the threshold (per-thread chunk masses and an fp64 block scan), then scans that
// one chunk: per-thread Kahan sums, an fp64 block scan, and one thread re-walks its segment.
namespace jf {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kPreStats = 64;             // trees up to this size get every row's statistics first

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct KahanSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

// Calls f(value) for every element of [s, e) of `base` that this thread owns, with 16-byte
// loads for the aligned body (the argmax kernel's split into head, body and tail).
template <typename T, typename F>
__device__ __forceinline__ void for_chunk(const T* base, long long s, long long e, F f) {
  constexpr int kVec = 16 / sizeof(T);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(base + s);
  long long head = ((16 - (addr & 15)) & 15) / sizeof(T);
  if (head > e - s) head = e - s;
  const long long body0 = s + head;
  const long long nvec = (e - body0) / kVec;
  const long long body1 = body0 + nvec * kVec;
  if (threadIdx.x < head) f(to_f<T>(base[s + threadIdx.x]));
  const uint4* vb = reinterpret_cast<const uint4*>(base + body0);
  for (long long v0 = threadIdx.x; v0 < nvec; v0 += blockDim.x) {
    const uint4 q = vb[v0];
    if constexpr (sizeof(T) == 2) {
      f(bf16_lo(q.x)); f(bf16_hi(q.x)); f(bf16_lo(q.y)); f(bf16_hi(q.y));
      f(bf16_lo(q.z)); f(bf16_hi(q.z)); f(bf16_lo(q.w)); f(bf16_hi(q.w));
    } else {
      f(__uint_as_float(q.x)); f(__uint_as_float(q.y)); f(__uint_as_float(q.z)); f(__uint_as_float(q.w));
    }
  }
  if (threadIdx.x < e - body1) f(to_f<T>(base[body1 + threadIdx.x]));
}

// Adds the exponentials of one 16-byte vector of logits to a thread's running (m, sum):
// k = log2(e) / T; the sum is kept relative to 2^(m k) and rescaled when m rises (once per
// vector at most).  The vector's own terms are summed pairwise in fp32 before a
// Kahan-compensated add, so the thread's sum stays within a few ulp.
template <int NV>
__device__ __forceinline__ void stats_add(const float (&x)[NV], float k, float& m, KahanSum& acc) {
  float vm = x[0];
#pragma unroll
  for (int e = 1; e < NV; ++e) vm = fmaxf(vm, x[e]);
  if (vm > m) {
    const float f = m == -INFINITY ? 0.f : fast_exp2((m - vm) * k);
    acc.s *= f;
    acc.c *= f;
    m = vm;
  }
  float part[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) part[e] = fast_exp2((x[e] - m) * k);   // x - m: exact near m
#pragma unroll
  for (int w = NV / 2; w > 0; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) part[e] += part[e + w];
  acc.add(part[0]);
}

// One warp per (row, chunk): lane-strided 16-byte vectors, kInFlight per lane in flight, each
// vector folded into the lane's running (m, Kahan sum) by stats_add; the warp then combines
// its lanes: M = max m, S = sum_lanes sum * 2^((m - M) k), in fp32 (GB300's fp64 rate is
// low; the lanes' sums are already compensated).  No block-wide barrier: the CTA's warps
// (up to kSampleThreads / 32; fewer when there are few chunks, so the CTAs still spread
// over the SMs) work on consecutive chunks independently.
template <typename T>
__global__ void __launch_bounds__(kSampleThreads)
    sample_stats_kernel(const T* __restrict__ logits, long long V, long long total_chunks, int chunks,
                        int chunk_len, float inv_t, float2* __restrict__ stats) {
  constexpr int kVec = 16 / sizeof(T);
  constexpr int kInFlight = 8;
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long gc = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gc < total_chunks) {
    const long long row = gc / chunks;
    const int c = static_cast<int>(gc - row * chunks);
    const long long s = static_cast<long long>(c) * chunk_len;
    const long long e = min(V, s + chunk_len);
    const T* base = logits + row * V;
    const float k = inv_t * 1.4426950408889634f;       // exp(y / T) = 2^(y * k)
    float m = -INFINITY;
    KahanSum acc;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(base + s);
    long long head = ((16 - (addr & 15)) & 15) / sizeof(T);
    if (head > e - s) head = e - s;
    const long long body0 = s + head;
    const int nvec = static_cast<int>((e - body0) / kVec);
    const long long body1 = body0 + static_cast<long long>(nvec) * kVec;
    if (lane < head) {
      const float x[1] = {to_f<T>(base[s + lane])};
      stats_add<1>(x, k, m, acc);
    }
    const uint4* vb = reinterpret_cast<const uint4*>(base + body0);
    for (int v0 = lane; v0 < nvec; v0 += 32 * kInFlight) {
      uint4 q[kInFlight];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int vi = v0 + u * 32;
        if (vi < nvec) q[u] = __ldcs(vb + vi);
      }
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int vi = v0 + u * 32;
        if (vi < nvec) {
          float x[kVec];
          if constexpr (sizeof(T) == 2) {
            x[0] = bf16_lo(q[u].x); x[1] = bf16_hi(q[u].x); x[2] = bf16_lo(q[u].y); x[3] = bf16_hi(q[u].y);
            x[4] = bf16_lo(q[u].z); x[5] = bf16_hi(q[u].z); x[6] = bf16_lo(q[u].w); x[7] = bf16_hi(q[u].w);
          } else {
            x[0] = __uint_as_float(q[u].x); x[1] = __uint_as_float(q[u].y);
            x[2] = __uint_as_float(q[u].z); x[3] = __uint_as_float(q[u].w);
          }
          stats_add<kVec>(x, k, m, acc);
        }
      }
    }
    if (lane < e - body1) {
      const float x[1] = {to_f<T>(base[body1 + lane])};
      stats_add<1>(x, k, m, acc);
    }
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float mine = (m == -INFINITY) ? 0.f : (acc.s - acc.c) * fast_exp2((m - M) * k);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0) stats[gc] = make_float2(M, mine);
  }
  grid_dependents_launch();
}

// Exclusive block scan of one int per thread; returns the thread's offset, total in *all.
__device__ __forceinline__ int block_excl_scan(int v, int* s_red, int* all) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) s_red[w] = x;
  __syncthreads();
  int base = 0, tot = 0;
  for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) {
    if (k < w) base += s_red[k];
    tot += s_red[k];
  }
  *all = tot;
  return base + x - v;
}

__device__ __forceinline__ double block_excl_scan_f64(double v, double* s_red, double* all) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) s_red[w] = x;
  __syncthreads();
  double base = 0.0, tot = 0.0;
  for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) {
    if (k < w) base += s_red[k];
    tot += s_red[k];
  }
  *all = tot;
  return base + x - v;
}

template <typename T>
__global__ void __launch_bounds__(kSampleThreads, 1)
    sampled_walk_kernel(const T* __restrict__ logits, const float2* __restrict__ stats, int chunks,
                        int chunk_len, const int32_t* __restrict__ draft,
                        const int32_t* __restrict__ parent, const float* __restrict__ uniform,
                        const float* __restrict__ bonus_uniform, float temperature, int N,
                        long long V, int32_t* __restrict__ accept_len, int32_t* __restrict__ path,
                        int32_t* __restrict__ bonus, int32_t* dev_err,
                        const int32_t* __restrict__ tree_len, const int32_t* __restrict__ cu,
                        long long total_rows) {
  extern __shared__ __align__(16) int32_t smw[];
  T* s_cv = reinterpret_cast<T*>(smw);  // [kSampleChunk] the bonus chunk's logits
  int32_t* s_par = smw + kSampleChunk * sizeof(T) / sizeof(int32_t);   // [N] parent (malformed -> -1)
  int32_t* s_draft = s_par + N;         // [N]
  int32_t* s_kids = s_draft + N;        // [N] children of the current node, id order
  int32_t* s_path = s_kids + N;         // [N]
  float* s_uni = reinterpret_cast<float*>(s_path + N);                   // [N] the children's uniforms
  float* s_tlg = s_uni + N;             // [N] node c's token's logit in its parent's row
  int32_t* s_rej = reinterpret_cast<int32_t*>(s_tlg + N);                 // [N] rejected tokens
  double* s_rejp = reinterpret_cast<double*>(                             // [N] their probabilities
      (reinterpret_cast<uintptr_t>(s_rej + N) + 7) & ~static_cast<uintptr_t>(7));
  double* s_pk = s_rejp + N;            // [N] target probabilities of the children's tokens
  __shared__ float s_aM[kPreStats];     // small trees: every row's maximum and normaliser
  __shared__ double s_aZ[kPreStats];
  __shared__ double s_redd[kSampleThreads / 32];
  __shared__ int s_redi[kSampleThreads / 32];
  __shared__ int s_next, s_nrej, s_chunk, s_y;
  __shared__ double s_rejmass, s_base, s_uZ;
  __shared__ float s_uM;

  grid_dependency_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Ragged calls: nodes >= nt are padding (never read, never anyone's child).  Packed
  // calls: the sequence's rows start at cu[b]; a bad span is reported and not read.
  const SeqSpan sp = seq_span(cu, tree_len, b, N, total_rows);
  if (!sp.ok && threadIdx.x == 0) report(dev_err, JF_DEVERR_BAD_TREE_LEN);
  if (sp.n == 0) {
    if (threadIdx.x == 0) {
      accept_len[b] = 0;
      bonus[b] = -1;
    }
    for (int k = threadIdx.x; k < N; k += blockDim.x)
      path[static_cast<size_t>(b) * N + k] = k == 0 ? 0 : -1;
    grid_dependents_launch();
    return;
  }
  const size_t rb = static_cast<size_t>(sp.row0);
  const int nt = sp.n;
  const double Td = temperature;
  const float inv_t = 1.f / temperature;
  int bad_parent = 0, bad_token = 0;
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    if (i >= nt) {
      s_par[i] = -1;
      s_draft[i] = -1;
      continue;
    }
    int p = parent[rb + i];
    const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
    if (!ok) { bad_parent = 1; p = -1; }
    s_par[i] = p;
    const int d = draft[rb + i];
    if (i > 0 && (d < 0 || d >= V)) bad_token = 1;
    s_draft[i] = (d >= 0 && d < V) ? d : -1;
  }
  bad_parent = __syncthreads_or(bad_parent);
  // every node's token logit in its parent's row, all requested at once (a walk step then
  // reads its children's from shared memory)
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    const int p = s_par[c], x = s_draft[c];
    s_tlg[c] = (p >= 0 && x >= 0) ? to_f<T>(logits[(rb + p) * V + x]) : -INFINITY;
  }
  bad_token = __syncthreads_or(bad_token);
  if (threadIdx.x == 0) {
    if (bad_parent) report(dev_err, JF_DEVERR_BAD_PARENT);
    if (bad_token) report(dev_err, JF_DEVERR_BAD_TOKEN);
    s_path[0] = 0;
  }
  // contiguous node range of this thread, for the ordered child lists
  const int per = (N + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
  const int c_lo = min(N, static_cast<int>(threadIdx.x) * per), c_hi = min(N, c_lo + per);
  int u = 0, n = 0;
  double M = 0.0, Z = 1.0, invZ = 1.0;
  const double invTd = 1.0 / Td;
  // M and Z of a row from its chunk statistics (fp64), by one warp (a row has a few dozen
  // chunks): fp64 sums of fp32 exponentials of fp64 arguments; exp's ~1e-7 relative error is
  // far below the 1e-5 margin the decisions are held to, and fp64 exp / division are slow
  // on this GPU (one division per node: the probabilities multiply by 1 / Z).
  auto row_stats = [&](int node, float* m_out, double* z_out) {
    const float2* st = stats + (rb + node) * chunks;
    float mloc = -INFINITY;
    for (int c = lane; c < chunks; c += 32) mloc = fmaxf(mloc, st[c].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    double zloc = 0.0;
    for (int c = lane; c < chunks; c += 32)
      zloc += static_cast<double>(st[c].y) *
              expf(static_cast<float>((static_cast<double>(st[c].x) - mloc) * invTd));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zloc += __shfl_xor_sync(0xffffffffu, zloc, o);
    if (lane == 0) {
      *m_out = mloc;
      *z_out = zloc;
    }
  };
  // Small trees: every row's M and Z up front, one warp per row, so a walk step waits on
  // no memory; larger ones find row u's when the walk reaches it.
  const bool all_stats = N <= kPreStats;
  if (all_stats)
    for (int k = warp; k < nt; k += static_cast<int>(blockDim.x >> 5)) row_stats(k, &s_aM[k], &s_aZ[k]);
  __syncthreads();
  for (;;) {
    if (all_stats) {
      if (threadIdx.x == 0) {
        s_uM = s_aM[u];
        s_uZ = s_aZ[u];
      }
    } else if (warp == 0) {
      row_stats(u, &s_uM, &s_uZ);
    }
    // children of u in id order (the scan's barriers publish M and Z)
    int cnt = 0;
    for (int c = c_lo; c < c_hi; ++c) cnt += (s_par[c] == u) ? 1 : 0;
    int nk = 0;
    int off = block_excl_scan(cnt, s_redi, &nk);
    M = s_uM;
    Z = s_uZ;
    invZ = 1.0 / Z;
    __syncthreads();                               // every thread has read M and Z
    for (int c = c_lo; c < c_hi; ++c)
      if (s_par[c] == u) s_kids[off++] = c;
    __syncthreads();
    // the children's target probabilities p(x) = exp((l_x - M) / T) / Z, one thread each
    // (fp64 is slow on this GPU: the ordered decisions below only read them)
    for (int k = threadIdx.x; k < nk; k += blockDim.x) {
      const int x = s_draft[s_kids[k]];
      const float lg = s_tlg[s_kids[k]];
      s_uni[k] = uniform[rb + s_kids[k]];
      s_pk[k] = x >= 0 ? static_cast<double>(expf(static_cast<float>((static_cast<double>(lg) - M) * invTd))) * invZ
                       : 0.0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double rej = 0.0;
      int next = -1, nrej = 0;
      for (int k = 0; k < nk; ++k) {
        const int c = s_kids[k];
        const int x = s_draft[c];
        bool seen = x < 0;
        for (int r = 0; r < nrej && !seen; ++r) seen = s_rej[r] == x;
        const double p = seen ? 0.0 : s_pk[k];
        if (static_cast<double>(s_uni[k]) * (1.0 - rej) < p) {
          next = c;
          break;
        }
        if (!seen) {
          s_rej[nrej] = x;
          s_rejp[nrej] = p;
          ++nrej;
          rej += p;
        }
      }
      s_next = next;
      s_nrej = nrej;
      s_rejmass = rej;
      if (next >= 0) s_path[n + 1] = next;
    }
    __syncthreads();
    if (s_next < 0) break;
    u = s_next;
    ++n;
  }
  // bonus token: inverse CDF of the residual at u
  const int nrej = s_nrej;
  const double target = static_cast<double>(bonus_uniform[b]) * (1.0 - s_rejmass);
  const T* row = logits + (rb + u) * V;
  const float2* st = stats + (rb + u) * chunks;
  // The chunk holding the threshold, in warp 0: residual chunk masses (the chunk's mass
  // minus its rejected tokens' probabilities) 32 chunks at a time, an fp64 warp scan, and
  // the first chunk c with (mass of the chunks before c) + w_c > target.  Masses can be a
  // rounding error below zero; with no crossing at all (rounding past the end) the last
  // chunk is taken, after the mass of all the others.
  if (warp == 0) {
    auto chunk_mass = [&](int c) -> double {
      const long long s0 = static_cast<long long>(c) * chunk_len, e0 = min(V, s0 + chunk_len);
      double w = static_cast<double>(st[c].y) *
                 expf(static_cast<float>((static_cast<double>(st[c].x) - M) * invTd)) * invZ;
      for (int r = 0; r < nrej; ++r)
        if (s_rej[r] >= s0 && s_rej[r] < e0) w -= s_rejp[r];
      return w;
    };
    double carry = 0.0, fbase = 0.0;
    int found = -1;
    for (int c0 = 0; c0 < chunks; c0 += 32) {
      const int c = c0 + lane;
      const double w = c < chunks ? chunk_mass(c) : 0.0;
      double incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned cross = __ballot_sync(0xffffffffu, c < chunks && carry + incl > target);
      if (cross != 0u) {
        const int L = __ffs(cross) - 1;
        found = c0 + L;
        fbase = carry + __shfl_sync(0xffffffffu, incl - w, L);
        break;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (found < 0) {
      found = chunks - 1;
      fbase = carry - chunk_mass(chunks - 1);
    }
    if (lane == 0) {
      s_chunk = found;
      s_base = fbase;
      s_y = -1;
    }
  }
  __syncthreads();
  // The chunk's logits are staged in shared memory by coalesced loads (16-byte vectors
  // when the chunk starts on a 16-byte boundary); then each thread takes 32 in token order.
  constexpr int kSeg = kSampleChunk / kSampleThreads;
  const long long cs0 = static_cast<long long>(s_chunk) * chunk_len;
  const long long ce0 = min(V, cs0 + chunk_len);
  const int clen = static_cast<int>(ce0 - cs0);
  {
    constexpr int kVec = 16 / sizeof(T);
    const T* src = row + cs0;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0u) {
      const int nv = clen / kVec;
      for (int v = threadIdx.x; v < nv; v += blockDim.x)
        reinterpret_cast<uint4*>(s_cv)[v] = __ldcs(reinterpret_cast<const uint4*>(src) + v);
      for (int e = nv * kVec + threadIdx.x; e < clen; e += blockDim.x) s_cv[e] = src[e];
    } else {
      for (int e = threadIdx.x; e < clen; e += blockDim.x) s_cv[e] = src[e];
    }
  }
  __syncthreads();
  const long long t0 = cs0 + static_cast<long long>(threadIdx.x) * kSeg;
  float ev[kSeg];
  {
    uint32_t rejm = 0u;                     // this thread's rejected tokens, one bit each
    for (int r = 0; r < nrej; ++r) {
      const long long d = static_cast<long long>(s_rej[r]) - t0;
      if (d >= 0 && d < kSeg) rejm |= 1u << d;
    }
    // exp((l - M) / T) of live tokens as 2^((l - M) log2(e) / T), else 0 (ex2.approx: ~2e-7
    // relative, inside the 1e-6 the bonus draw is held to)
    const float Mf = static_cast<float>(M);
    const float k2 = inv_t * 1.4426950408889634f;
    const int e0 = static_cast<int>(threadIdx.x) * kSeg;
#pragma unroll
    for (int e = 0; e < kSeg; ++e) {
      const bool live = e0 + e < clen && !((rejm >> e) & 1u);
      ev[e] = live ? fast_exp2((to_f<T>(s_cv[e0 + e]) - Mf) * k2) : 0.f;
    }
  }
  KahanSum ks;
#pragma unroll
  for (int e = 0; e < kSeg; ++e) ks.add(ev[e]);
  const double mine = (static_cast<double>(ks.s) - static_cast<double>(ks.c)) * invZ;
  double all = 0.0;
  const double before = s_base + block_excl_scan_f64(mine, s_redd, &all);
  if (mine > 0.0 && before <= target && target < before + mine) {
    // the crossing inside this thread's tokens, in fp32 and in the unnormalised units of
    // ev: the threshold's offset into the segment times Z (32 fp32 terms round to ~2e-6 of
    // the segment's own small mass)
    const float need = static_cast<float>((target - before) * Z);
    float cum = 0.f;
    int y = -1, last = -1;
#pragma unroll
    for (int e = 0; e < kSeg; ++e) {
      if (ev[e] > 0.f) last = e;
      cum += ev[e];
      if (y < 0 && cum > need) y = e;
    }
    s_y = static_cast<int>(t0) + (y >= 0 ? y : last);
  }
  __syncthreads();
  if (s_y < 0) {                               // rounding past the chunk's end: last live token
    int v = -1;
#pragma unroll
    for (int e = 0; e < kSeg; ++e)
      if (ev[e] > 0.f) v = static_cast<int>(t0) + e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s_redi[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
      int r = -1;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) r = max(r, s_redi[w]);
      s_y = r >= 0 ? r : static_cast<int>(cs0);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    accept_len[b] = n;
    bonus[b] = s_y;
  }
  for (int k = threadIdx.x; k < N; k += blockDim.x)
    path[static_cast<size_t>(b) * N + k] = k <= n ? s_path[k] : -1;
  grid_dependents_launch();
}

}  // namespace
}  // namespace jf

namespace {

// Packed calls (cu != nullptr) hold T = cu[B] logit rows; the others B * N.
jf_status tree_verify_sampled_call(const void* logits, int32_t dtype, const int32_t* draft,
                                   const int32_t* parent, const float* uniform,
                                   const float* bonus_uniform, float temperature, int32_t B,
                                   int32_t N, int32_t V, int32_t* accept_len, int32_t* path,
                                   int32_t* bonus, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_err, jf_stream_t stream, const int32_t* tree_len,
                                   const int32_t* cu, int32_t T) {
  if (logits == nullptr || draft == nullptr || parent == nullptr || uniform == nullptr ||
      bonus_uniform == nullptr || accept_len == nullptr || path == nullptr || bonus == nullptr ||
      workspace == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (dtype != JF_DTYPE_BF16 && dtype != JF_DTYPE_F32) return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || V < 1 || !(temperature > 0.f) || !std::isfinite(temperature))
    return JF_ERR_INVALID_ARGUMENT;
  if (cu != nullptr && T < 1) return JF_ERR_INVALID_ARGUMENT;
  if (N > JF_MAX_NODES) return JF_ERR_UNSUPPORTED;
  const long long rows = cu != nullptr ? static_cast<long long>(T) : static_cast<long long>(B) * N;
  jf::VerifyPlan p;
  p.chunk_len = jf::kSampleChunk;
  p.chunks = jf::sampled_chunks(V);
  const size_t need = static_cast<size_t>(rows) * p.chunks * sizeof(float2);
  if (workspace_bytes < need) return JF_ERR_WORKSPACE_TOO_SMALL;
  if (!jf::aligned_to(workspace, 8)) return JF_ERR_MISALIGNED;
  if (!jf::aligned_to(logits, dtype == JF_DTYPE_BF16 ? 2 : 4)) return JF_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float2* stats = static_cast<float2*>(workspace);
  const long long total = rows * p.chunks;                              // one warp each
  const int sms = jf::current_sm_count() > 0 ? jf::current_sm_count() : 148;
  int warps = jf::kSampleThreads / 32;
  while (warps > 1 && total < static_cast<long long>(warps) * 4 * sms) warps >>= 1;
  const long long grid = (total + warps - 1) / warps;
  if (grid > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  const long long Vl = V;
  const float inv_t = 1.f / temperature;
  const cudaError_t ea =
      dtype == JF_DTYPE_BF16
          ? jf::launch_pdl(jf::sample_stats_kernel<uint16_t>, dim3(static_cast<unsigned>(grid)),
                           dim3(32 * warps), 0, s, static_cast<const uint16_t*>(logits), Vl,
                           total, p.chunks, p.chunk_len, inv_t, stats)
          : jf::launch_pdl(jf::sample_stats_kernel<float>, dim3(static_cast<unsigned>(grid)),
                           dim3(32 * warps), 0, s, static_cast<const float*>(logits), Vl,
                           total, p.chunks, p.chunk_len, inv_t, stats);
  if (ea != cudaSuccess) return JF_ERR_CUDA;
  auto walk = [&](auto kern, const auto* lg) -> cudaError_t {
    // the bonus chunk's logits, then 7 int/float and 2 double arrays of N (+ alignment)
    const size_t smem = jf::kSampleChunk * sizeof(*lg) +
                        static_cast<size_t>(N) * (7 * sizeof(int32_t) + 2 * sizeof(double)) + 16;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
      return cudaErrorInvalidValue;
    return jf::launch_pdl(kern, dim3(B), dim3(jf::kSampleThreads), smem, s, lg,
                          static_cast<const float2*>(stats), p.chunks, p.chunk_len, draft, parent,
                          uniform, bonus_uniform, temperature, N, Vl, accept_len, path, bonus, dev_err,
                          tree_len, cu, static_cast<long long>(cu != nullptr ? T : 0));
  };
  const cudaError_t ew =
      dtype == JF_DTYPE_BF16
          ? walk(jf::sampled_walk_kernel<uint16_t>, static_cast<const uint16_t*>(logits))
          : walk(jf::sampled_walk_kernel<float>, static_cast<const float*>(logits));
  return ew == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

}  // namespace

extern "C" jf_status jf_tree_verify_sampled(const void* logits, int32_t dtype, const int32_t* draft,
                                            const int32_t* parent, const float* uniform,
                                            const float* bonus_uniform, float temperature,
                                            int32_t B, int32_t N, int32_t V, int32_t* accept_len,
                                            int32_t* path, int32_t* bonus, void* workspace,
                                            size_t workspace_bytes, int32_t* dev_err,
                                            jf_stream_t stream) {
  return tree_verify_sampled_call(logits, dtype, draft, parent, uniform, bonus_uniform,
                                  temperature, B, N, V, accept_len, path, bonus, workspace,
                                  workspace_bytes, dev_err, stream, nullptr, nullptr, 0);
}

extern "C" jf_status jf_tree_verify_sampled_ragged(
    const void* logits, int32_t dtype, const int32_t* draft, const int32_t* parent,
    const int32_t* tree_len, const float* uniform, const float* bonus_uniform, float temperature,
    int32_t B, int32_t N, int32_t V, int32_t* accept_len, int32_t* path, int32_t* bonus,
    void* workspace, size_t workspace_bytes, int32_t* dev_err, jf_stream_t stream) {
  if (tree_len == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return tree_verify_sampled_call(logits, dtype, draft, parent, uniform, bonus_uniform,
                                  temperature, B, N, V, accept_len, path, bonus, workspace,
                                  workspace_bytes, dev_err, stream, tree_len, nullptr, 0);
}

extern "C" jf_status jf_tree_verify_sampled_packed(
    const void* logits, int32_t dtype, const int32_t* draft, const int32_t* parent,
    const int32_t* cu_seqlens, const float* uniform, const float* bonus_uniform,
    float temperature, int32_t B, int32_t N_max, int32_t T, int32_t V, int32_t* accept_len,
    int32_t* path, int32_t* bonus, void* workspace, size_t workspace_bytes, int32_t* dev_err,
    jf_stream_t stream) {
  if (cu_seqlens == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return tree_verify_sampled_call(logits, dtype, draft, parent, uniform, bonus_uniform,
                                  temperature, B, N_max, V, accept_len, path, bonus, workspace,
                                  workspace_bytes, dev_err, stream, nullptr, cu_seqlens, T);
}
