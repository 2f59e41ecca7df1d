// jf_draft_tree.cu -- best-first draft-tree construction from per-depth draft logits.
//
// JetFlow explainer ("JetFlow: Breaking the Scaling Ceiling of Speculative Decoding with
// Parallel Tree Drafting"), technical summary §2 "Method", tree construction: at inference
// the draft head emits logits for every tree depth in one pass; nodes are ranked by a
// branch score, by default the cumulative draft log-probability, and a best-first
// expansion builds the candidate tree up to a token budget.
//
// Kernel 1, one CTA per (sequence, depth d): the K candidates of depth d are the K
// largest logits (lower token id on ties) with their log-probabilities
// logit - logsumexp(row), fp32.
// Kernel 2, one CTA per sequence: every node at depth d < Dmax has the K depth-(d+1)
// candidates as children, child score = fp32(parent score + candidate log-prob), root
// score 0.  Best-first expansion to N nodes pops nodes in the order of the key
// (score descending, depth ascending, rank path ascending), so the tree is the first N
// nodes of the candidate lattice in that order (a parent always precedes its children:
// its score is not lower and its depth is smaller).  The kernel finds them level by
// level: the level-d candidates are the children of the chosen level-(d-1) nodes (once
// N nodes are chosen, only those that beat the last of them), and the chosen set, kept
// sorted in shared memory, becomes the first N keys of (chosen so far + candidates): the
// candidates, sorted runs per parent, are merged pairwise into one sorted run, and each
// key's place is the number of keys below it.  A node is identified by its rank path
// packed into a 64-bit code (4 bits per level, first level in the top bits), so its
// parent's code is its own with the last digit cleared.
#include <algorithm>
#include <cmath>

#include <mutex>

#include "jf_common.cuh"
#include "jf_sm100.cuh"

namespace jf {
namespace {

constexpr int kTopThreads = 512;
constexpr int kTreeThreads = 1024;
constexpr int kMaxK = 8;
constexpr int kMaxDepth = 16;
constexpr int kMaxTreeN = 256;
constexpr int kCandMax = kMaxTreeN * kMaxK;   // candidates of one level, at most
constexpr int kCountMaxC = 64;           // up to this many candidates are ranked by counting
constexpr int kRowParts = 8;             // most CTAs (one cluster) per logit row
constexpr int kCandCap = 1024;           // filtered candidates a CTA keeps in shared memory

// ---------------------------------------------------------------- kernel 1: candidates
struct Cand {
  float v;
  int i;
};

template <typename T>
__device__ __forceinline__ float load_logit(const T* p, long long i);
template <>
__device__ __forceinline__ float load_logit<float>(const float* p, long long i) { return p[i]; }
template <>
__device__ __forceinline__ float load_logit<uint16_t>(const uint16_t* p, long long i) {
  return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}

// A warp keeps one sorted list of its kMaxK best logits, entry r in lane r (lanes >= kMaxK
// unused); thr is the list's last.  Every lane offers one logit per call; lanes whose
// logit beats thr are taken one at a time (lowest lane first): its rank p in the list is
// the number of entries that beat it, entries p.. move down one lane, and it lands in
// lane p.  After the first few hundred logits almost no lane qualifies, so the common
// case is one vote.
__device__ __forceinline__ void warp_offer(float v, int i, bool valid, Cand& wl, Cand& thr) {
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = static_cast<int>(threadIdx.x & 31);
  unsigned mask = __ballot_sync(kAll, valid && (v > thr.v || (v == thr.v && i < thr.i)));
  while (mask != 0u) {
    const int L = __ffs(mask) - 1;
    const float cv = __shfl_sync(kAll, v, L);
    const int ci = __shfl_sync(kAll, i, L);
    const bool ahead = lane < kMaxK && (wl.v > cv || (wl.v == cv && wl.i < ci));
    const int p = __popc(__ballot_sync(kAll, ahead));
    const float uv = __shfl_up_sync(kAll, wl.v, 1);
    const int ui = __shfl_up_sync(kAll, wl.i, 1);
    if (lane < kMaxK && lane > p) { wl.v = uv; wl.i = ui; }
    if (lane == p) { wl.v = cv; wl.i = ci; }
    thr.v = __shfl_sync(kAll, wl.v, kMaxK - 1);
    thr.i = __shfl_sync(kAll, wl.i, kMaxK - 1);
    mask &= ~(1u << L);
    mask &= __ballot_sync(kAll, valid && (v > thr.v || (v == thr.v && i < thr.i)));
  }
}

// State of one thread across the passes over its CTA's slice of a row.
struct PassState {
  float M;        // slice maximum (pass 2)
  float tau;      // candidate threshold (pass 2)
  float m;        // running maximum (pass 1)
  float sum;      // running sum of exp(x - M) (pass 2)
  Cand wl, thr;   // the warp's K-best list and its last entry (pass 3)
  Cand* cand;     // shared candidate buffer (pass 2)
  int* ncand;
};

// One pass over this CTA's slice of a row, warp-synchronously (every lane runs every
// step; lanes past the slice offer nothing).  PASS 1 folds the maximum into m.  PASS 2
// adds exp(x - M) into sum and appends every logit >= tau to the shared candidate buffer.
// PASS 3 (only when the buffer overflowed) offers every logit to the warp's K-best list.
// The row is read as 16-byte vectors, kUnroll per thread in flight, when it starts on a
// 16-byte boundary (bf16 passes 1 and 2 then work on packed pairs, see bf16_vec_pass);
// otherwise element by element.
template <int PASS>
__device__ __forceinline__ void take(float v, int i, bool valid, PassState& st) {
  if constexpr (PASS == 1) {
    if (valid) st.m = fmaxf(st.m, v);
  } else if constexpr (PASS == 2) {
    if (valid) {
      st.sum += __expf(v - st.M);
      if (v >= st.tau) {
        const int pos = atomicAdd(st.ncand, 1);
        if (pos < kCandCap) st.cand[pos] = Cand{v, i};
      }
    }
  } else {
    warp_offer(v, i, valid, st.wl, st.thr);
  }
}

// bf16 logits two to a 32-bit word (the lower-indexed one in the low half).  The maximum
// of packed pairs is exact, so the passes fold whole vectors with it.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16x8_max(const uint4& q) {
  return bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w));
}

// Passes 1 and 2 over 16-byte vectors of bf16 logits.  Pass 1 keeps the slice maximum as
// a packed pair.  Pass 2 sums exp(x - M) as 2^(x log2 e - M log2 e) over the eight logits
// and looks at them one by one only when the vector's maximum reaches tau.
template <int PASS>
__device__ __forceinline__ void bf16_vec_pass(const uint4* xv, int vb, int nvec, PassState& st) {
  constexpr int kUnroll = 4;
  constexpr float kLog2e = 1.4426950408889634f;
  uint32_t pm = 0xFF80FF80u;                    // (-inf, -inf)
  const float neg_ml = -st.M * kLog2e;
  float s0 = 0.f, s1 = 0.f;
  for (int v0 = vb + static_cast<int>(threadIdx.x); v0 < nvec; v0 += blockDim.x * kUnroll) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * blockDim.x;
      buf[u] = v < nvec ? __ldg(xv + v) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * blockDim.x;
      if (PASS == 1) {
        pm = bf16x2_max(pm, bf16x8_max(buf[u]));
      } else if (v < nvec) {
        const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s0 += fast_exp2(fmaf(bf16_lo(w[k]), kLog2e, neg_ml));
          s1 += fast_exp2(fmaf(bf16_hi(w[k]), kLog2e, neg_ml));
        }
        const uint32_t m2 = bf16x8_max(buf[u]);
        if (fmaxf(bf16_lo(m2), bf16_hi(m2)) >= st.tau) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float val = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
            if (val >= st.tau) {
              const int pos = atomicAdd(st.ncand, 1);
              if (pos < kCandCap) st.cand[pos] = Cand{val, v * 8 + e};
            }
          }
        }
      }
    }
  }
  if (PASS == 1) st.m = fmaxf(st.m, fmaxf(bf16_lo(pm), bf16_hi(pm)));
  else st.sum += s0 + s1;
}

template <typename T, int PASS>
__device__ __forceinline__ void row_pass(const T* x, int V, int part, int parts, PassState& st) {
  constexpr int kPer = 16 / sizeof(T);          // logits per vector
  constexpr int kUnroll = 4;
  const int lane0 = static_cast<int>(threadIdx.x) & ~31;   // first thread of this warp
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0u) {
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const int nvec_all = V / kPer;
    const int per = (nvec_all + parts - 1) / parts;
    const int vb = min(nvec_all, part * per);
    const int nvec = min(nvec_all, vb + per);
    if constexpr (sizeof(T) == 2 && PASS != 3) {
      bf16_vec_pass<PASS>(xv, vb, nvec, st);
    } else {
      // the warp loops while its first lane still has vectors, so all lanes step together
      for (int w0 = vb + lane0; w0 < nvec; w0 += blockDim.x * kUnroll) {
        const int v0 = w0 + (threadIdx.x & 31);
        uint4 buf[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * blockDim.x;
          buf[u] = v < nvec ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * blockDim.x;
          const bool valid = v < nvec;
          const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
          for (int e = 0; e < kPer; ++e) {
            float val;
            if constexpr (sizeof(T) == 2)
              val = __uint_as_float(((w[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu) << 16);
            else
              val = __uint_as_float(w[e]);
            take<PASS>(val, v * kPer + e, valid, st);
          }
        }
      }
    }
    if (part == parts - 1)
      for (int b0 = nvec_all * kPer + lane0; b0 < V; b0 += blockDim.x) {
        const int i = b0 + (threadIdx.x & 31);
        const bool valid = i < V;
        take<PASS>(valid ? load_logit<T>(x, i) : -INFINITY, i, valid, st);
      }
  } else {
    const int per = (V + parts - 1) / parts;
    const int ib = min(V, part * per), ie = min(V, ib + per);
    for (int b0 = ib + lane0; b0 < ie; b0 += blockDim.x) {
      const int i = b0 + (threadIdx.x & 31);
      const bool valid = i < ie;
      take<PASS>(valid ? load_logit<T>(x, i) : -INFINITY, i, valid, st);
    }
  }
}

// The k-th largest (k <= kMaxK) of one value per thread of the CTA, by repeated
// extraction: each warp takes its k largest, then warp 0 takes the k largest of those;
// the first of them is the CTA's maximum, returned in *mx.  Every thread of the CTA calls
// it; `scratch` holds kWarps * kMaxK floats.
__device__ float block_kth_largest(float x, int k, float* scratch, float* mx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int r = 0; r < k; ++r) {
    float b = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    const unsigned who = __ballot_sync(0xffffffffu, x == b);
    if (lane == __ffs(who) - 1) x = -INFINITY;
    if (lane == 0) scratch[warp * kMaxK + r] = b;
  }
  __syncthreads();
  float kth = -INFINITY, top = -INFINITY;
  if (warp == 0) {
    int head = 0;                                  // lane q < nwarps walks warp q's list
    for (int r = 0; r < k; ++r) {
      const float h = (lane < nwarps && head < k) ? scratch[lane * kMaxK + head] : -INFINITY;
      float b = h;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
      const unsigned who = __ballot_sync(0xffffffffu, lane < nwarps && head < k && h == b);
      if (lane == __ffs(who) - 1) ++head;
      if (r == 0) top = b;
      kth = b;
    }
    if (lane == 0) {
      scratch[0] = kth;
      scratch[1] = top;
    }
  }
  __syncthreads();
  kth = scratch[0];
  *mx = scratch[1];
  __syncthreads();
  return kth;
}

// A cluster of `parts` CTAs shares one row (parts <= kRowParts: the host splits rows only
// as far as it takes to fill the GPU); each makes two passes over its slice: the
// slice maximum m_c, then s_c = sum of exp(x - m_c) together with the slice's K best.
// The K best are found by filtering: the K-th largest of the threads' pass-1 maxima is a
// value at least K logits of the slice reach, so the slice's K best all lie at or above
// it; pass 2 keeps only those logits (a few dozen for real logits) and one warp ranks
// them.  When heavy ties push more than kCandCap logits over the threshold, a third pass
// ranks the whole slice per warp instead (exact either way).  The cluster's first CTA
// merges the slices through distributed shared memory: M = max m_c,
// S = sum s_c * exp(m_c - M), lse = M + log S, and the K best of the slices' lists.
// kMinBlocks: CTAs an SM must hold (3 caps registers at 40 and keeps a one-wave grid
// resident at once; 2 leaves the passes unconstrained and, on grids of several waves,
// keeps fewer rows in flight, so the second pass finds its slice in L2).
template <typename T, int kMinBlocks>
__global__ void __launch_bounds__(kTopThreads, kMinBlocks)
    draft_candidates_kernel(const T* __restrict__ logits, int V, int K, int parts,
                            int32_t* __restrict__ cand_token, float* __restrict__ cand_logp) {
  constexpr int kWarps = kTopThreads / 32;
  __shared__ Cand s_top[kWarps][kMaxK];
  __shared__ float s_red[kTopThreads];
  __shared__ float s_slice[2];                   // this slice's (max, sum)
  __shared__ Cand s_cand[kCandCap];
  __shared__ int s_ncand;
  grid_dependency_wait();
  const long long row = blockIdx.x / parts;
  const int part = static_cast<int>(cluster_ctarank());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* x = logits + row * V;
  PassState st;
  st.M = 0.f;
  st.tau = INFINITY;
  st.m = -INFINITY;
  st.sum = 0.f;
  st.wl = Cand{-INFINITY, 0x7fffffff};
  st.thr = Cand{-INFINITY, 0x7fffffff};
  st.cand = s_cand;
  st.ncand = &s_ncand;
  if (threadIdx.x == 0) s_ncand = 0;
  row_pass<T, 1>(x, V, part, parts, st);                      // slice maximum
  // threshold: the K-th largest thread maximum (-inf when the slice has fewer logits)
  float M;
  st.tau = block_kth_largest(st.m, K, s_red, &M);
  st.M = M;
  if (M != -INFINITY) row_pass<T, 2>(x, V, part, parts, st);
  __syncthreads();
  const int ncand = s_ncand;
  if (ncand <= kCandCap) {
    // rank the candidates in warp 0; the other warps' lists stay empty
    if (warp == 0)
      for (int j0 = 0; j0 < ncand; j0 += 32) {
        const int j = j0 + lane;
        const bool valid = j < ncand;
        const Cand c = valid ? s_cand[j] : Cand{-INFINITY, 0x7fffffff};
        warp_offer(c.v, c.i, valid, st.wl, st.thr);
      }
  } else if (M != -INFINITY) {
    row_pass<T, 3>(x, V, part, parts, st);                    // every logit, per warp
  }
  if (lane < kMaxK) s_top[warp][lane] = st.wl;
  float wsum = st.sum;                             // the slice's sum: per warp, then warp 0
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane == 0) s_red[warp] = wsum;
  __syncthreads();
  // merge the warps' lists: warp 0 takes the K best heads, one per round
  if (warp == 0) {
    int head = 0;                                  // lane q < kWarps walks list q
    Cand out = Cand{-INFINITY, 0x7fffffff};
    for (int r = 0; r < kMaxK; ++r) {
      const Cand h = (lane < kWarps && head < kMaxK) ? s_top[lane][head] : Cand{-INFINITY, 0x7fffffff};
      float bv = h.v;
      int bi = h.i;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane < kWarps && head < kMaxK && h.v == bv && h.i == bi) ++head;
      if (lane == r) out = Cand{bv, bi};
    }
    __syncwarp();
    if (lane < kMaxK) s_top[0][lane] = out;        // this slice's K best, in order
    if (lane == 0) {
      float sum = 0.f;
      for (int w = 0; w < kWarps; ++w) sum += s_red[w];
      s_slice[0] = M;
      s_slice[1] = sum;
    }
  }
  cluster_sync();                                // every slice's result is in place
  if (part == 0 && warp == 0) {
    // lane q < parts fetches slice q's (max, sum) and K-best list
    float mq = -INFINITY, sq = 0.f;
    Cand lst[kMaxK];
    if (lane < parts) {
      mq = dsmem_ld_f32(dsmem_addr(&s_slice[0], lane));
      sq = dsmem_ld_f32(dsmem_addr(&s_slice[1], lane));
#pragma unroll
      for (int r = 0; r < kMaxK; ++r) {
        const float2 c = dsmem_ld_f32x2(dsmem_addr(&s_top[0][r], lane));
        lst[r] = Cand{c.x, __float_as_int(c.y)};
      }
    } else {
#pragma unroll
      for (int r = 0; r < kMaxK; ++r) lst[r] = Cand{-INFINITY, 0x7fffffff};
    }
    float Mx = mq;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
    float S = mq == -INFINITY ? 0.f : sq * __expf(mq - Mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    int head = 0;
    for (int r = 0; r < K; ++r) {
      Cand h = Cand{-INFINITY, 0x7fffffff};
#pragma unroll
      for (int q = 0; q < kMaxK; ++q)
        if (q == head) h = lst[q];
      float bv = h.v;
      int bi = h.i;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (head < kMaxK && h.v == bv && h.i == bi) ++head;   // indices are unique
      if (lane == 0) {
        cand_token[row * K + r] = bi;
        cand_logp[row * K + r] = bv - (Mx + __logf(S));
      }
    }
  }
  cluster_sync();                                // no CTA leaves while the first reads it
  grid_dependents_launch();
}

// ---------------------------------------------------------------- kernel 2: best-first
// Sort key: hi = (descending-score bits << 32) | depth, lo = rank-path code; ascending.
__device__ __forceinline__ uint32_t desc_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // order-preserving
  return ~asc;
}
__device__ __forceinline__ float from_desc_bits(uint32_t d) {
  const uint32_t asc = ~d;
  const uint32_t u = (asc & 0x80000000u) ? (asc & 0x7fffffffu) : ~asc;
  return __uint_as_float(u);
}
__device__ __forceinline__ bool key_less(uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl) {
  return ah < bh || (ah == bh && al < bl);
}

// Number of the first n keys of a sorted array that are below (h, l).
__device__ __forceinline__ int lower_bound_key(const uint64_t* hi, const uint64_t* lo, int n, uint64_t h,
                                               uint64_t l) {
  int a = 0, c = n;
  while (a < c) {
    const int m = (a + c) >> 1;
    if (key_less(hi[m], lo[m], h, l)) a = m + 1;
    else c = m;
  }
  return a;
}

// Number of the first n keys of a sorted array that are at or below (h, l).
__device__ __forceinline__ int upper_bound_key(const uint64_t* hi, const uint64_t* lo, int n, uint64_t h,
                                               uint64_t l) {
  int a = 0, c = n;
  while (a < c) {
    const int m = (a + c) >> 1;
    if (!key_less(h, l, hi[m], lo[m])) a = m + 1;
    else c = m;
  }
  return a;
}


__global__ void __launch_bounds__(kTreeThreads, 1)
    best_first_tree_kernel(const int32_t* __restrict__ cand_token, const float* __restrict__ cand_logp,
                           const int32_t* __restrict__ root_token, int Dmax, int K, int N,
                           int32_t* __restrict__ parent, int32_t* __restrict__ draft,
                           int32_t* __restrict__ depth_out, float* __restrict__ score_out,
                           const int32_t* __restrict__ budget, int32_t* dev_err) {
  // The chosen set G (at most N keys, in key order) and its successor, double-buffered;
  // this level's candidates C (at most N * kMaxK slots) and the merge's scratch.
  extern __shared__ uint64_t s_keys[];
  uint64_t* g_hi = s_keys;
  uint64_t* g_lo = g_hi + kMaxTreeN;
  uint64_t* x_hi = g_lo + kMaxTreeN;
  uint64_t* x_lo = x_hi + kMaxTreeN;
  uint64_t* c_hi = x_lo + kMaxTreeN;
  uint64_t* c_lo = c_hi + kCandMax;
  uint64_t* c_bhi = c_lo + kCandMax;
  uint64_t* c_blo = c_bhi + kCandMax;
  __shared__ float s_lp[kMaxDepth * kMaxK];
  __shared__ int s_tok[kMaxDepth * kMaxK];
  __shared__ int s_warp[kMaxTreeN / 32];
  grid_dependency_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This sequence's budget: N, or budget[b] clamped to [1, N] (per-sequence budgets).
  int Nb = N;
  if (budget != nullptr) {
    const int raw = budget[b];
    Nb = max(1, min(raw, N));
    if (raw != Nb && threadIdx.x == 0) report(dev_err, JF_DEVERR_BAD_TREE_LEN);
  }
  for (int e = threadIdx.x; e < Dmax * K; e += blockDim.x) {
    s_lp[e] = cand_logp[static_cast<size_t>(b) * Dmax * K + e];
    s_tok[e] = cand_token[static_cast<size_t>(b) * Dmax * K + e];
  }
  if (threadIdx.x == 0) {                          // G starts as the root
    g_hi[0] = static_cast<uint64_t>(desc_bits(0.f)) << 32;
    g_lo[0] = 0ull;
  }
  int nG = 1;
  __syncthreads();
  for (int d = 1; d <= Dmax; ++d) {
    const int shift = 4 * (kMaxDepth - d);
    // Level-d candidates: children of the chosen level-(d-1) nodes.  Once G holds N nodes
    // a child only matters if it beats G's last; a parent's children fall in score with
    // their rank, so those form a prefix of its K children.  Slot f's count is found by
    // thread f and scanned per warp and across the (at most 8) warps.
    const bool full = nG == Nb;
    const uint64_t thr_hi = full ? g_hi[Nb - 1] : ~0ull, thr_lo = full ? g_lo[Nb - 1] : ~0ull;
    const int f = threadIdx.x;
    int cnt = 0;
    float ps = 0.f;
    if (f < nG && (g_hi[f] & 0xFFFFFFFFull) == static_cast<uint64_t>(d - 1)) {
      ps = from_desc_bits(static_cast<uint32_t>(g_hi[f] >> 32));
      for (int r = 0; r < K; ++r) {
        const float cs = __fadd_rn(ps, s_lp[(d - 1) * K + r]);
        const uint64_t ch = (static_cast<uint64_t>(desc_bits(cs)) << 32) | static_cast<uint64_t>(d);
        const uint64_t cl = g_lo[f] | (static_cast<uint64_t>(r) << shift);
        if (!key_less(ch, cl, thr_hi, thr_lo)) break;
        ++cnt;
      }
    }
    // One scan gives both C's size (the counts) and each parent's index among the slots
    // that have children (the flags, in the upper half).  A parent's children fall in key
    // order with their rank, so each parent writes a sorted run of kMaxK slots, the ranks
    // past its count padded with the largest key.
    int incl = cnt | ((cnt > 0 ? 1 : 0) << 16);
    if (f < kMaxTreeN) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_warp[warp] = incl;
    }
    __syncthreads();
    int tot = 0, base = 0;
#pragma unroll
    for (int w = 0; w < kMaxTreeN / 32; ++w) {
      base += w < warp ? s_warp[w] : 0;
      tot += s_warp[w];
    }
    const int nC = tot & 0xFFFF, npar = tot >> 16;
    if (nC == 0) break;
    const bool few = nC <= kCountMaxC;               // few candidates: C stays unsorted
    int runs = 1;
    while (runs < npar) runs <<= 1;
    const int nS = few ? nC : runs * kMaxK;          // candidate slots
    if (cnt > 0) {
      const int o = few ? ((base + incl) & 0xFFFF) - cnt : (((base + incl) >> 16) - 1) * kMaxK;
      const uint64_t pc = g_lo[f];
      for (int r = 0; r < (few ? cnt : kMaxK); ++r) {
        uint64_t h = ~0ull, l = ~0ull;
        if (r < cnt) {
          const float cs = __fadd_rn(ps, s_lp[(d - 1) * K + r]);
          h = (static_cast<uint64_t>(desc_bits(cs)) << 32) | static_cast<uint64_t>(d);
          l = pc | (static_cast<uint64_t>(r) << shift);
        }
        c_hi[o + r] = h;
        c_lo[o + r] = l;
      }
    }
    for (int e = (few ? nS : npar * kMaxK) + threadIdx.x; e < nS; e += blockDim.x) {   // empty runs
      c_hi[e] = ~0ull;
      c_lo[e] = ~0ull;
    }
    __syncthreads();
    // Merge the runs pairwise until C is one sorted run: a key's place in the merged pair is
    // its index in its own run plus the keys of the other run below it (at or below it, for
    // the second run: the padding keys are equal and keep their order).  Real keys come
    // first; they are distinct.
    int src = 0;                                     // the merge's current buffer
    for (int L = kMaxK; !few && L < nS; L <<= 1, src ^= 1) {
      const uint64_t* sh = src ? c_bhi : c_hi;
      const uint64_t* sl = src ? c_blo : c_lo;
      uint64_t* dh = src ? c_hi : c_bhi;
      uint64_t* dl = src ? c_lo : c_blo;
      for (int i = threadIdx.x; i < nS; i += blockDim.x) {
        const int p0 = i & ~(2 * L - 1);
        const bool in_a = (i & L) == 0;
        const uint64_t h = sh[i], l = sl[i];
        const int at = in_a ? (i - p0) + lower_bound_key(sh + p0 + L, sl + p0 + L, L, h, l)
                            : (i - p0 - L) + upper_bound_key(sh + p0, sl + p0, L, h, l);
        dh[p0 + at] = h;
        dl[p0 + at] = l;
      }
      __syncthreads();
    }
    const uint64_t* sh = src ? c_bhi : c_hi;         // C, sorted unless few
    const uint64_t* sl = src ? c_blo : c_lo;
    // The next G is the first N keys of G + C: a key's place is the number of keys below
    // it, its index in its own sorted set plus the other set's keys below it (counted
    // one by one when C is small and unsorted).
    const int total = nG + nC, keep = min(Nb, total);
    int kept_d = 0;
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
      const bool in_g = e < nG;
      const uint64_t h = in_g ? g_hi[e] : sh[e - nG], l = in_g ? g_lo[e] : sl[e - nG];
      int pos;
      if (few) {                                     // unsorted C: count its keys below
        pos = in_g ? e : lower_bound_key(g_hi, g_lo, nG, h, l);
        for (int j = 0; j < nC; ++j) pos += key_less(sh[j], sl[j], h, l) ? 1 : 0;
      } else {
        pos = in_g ? e + lower_bound_key(sh, sl, nC, h, l)
                   : (e - nG) + lower_bound_key(g_hi, g_lo, nG, h, l);
      }
      if (pos < keep) {
        x_hi[pos] = h;
        x_lo[pos] = l;
        kept_d |= in_g ? 0 : 1;
      }
    }
    kept_d = __syncthreads_or(kept_d);
    uint64_t* t = g_hi; g_hi = x_hi; x_hi = t;
    t = g_lo; g_lo = x_lo; x_lo = t;
    nG = keep;
    // stop once no level-d node made it (deeper ones cannot either)
    if (!kept_d) break;
  }
  // G in key order is the tree in pop order: node id = slot
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const size_t o = static_cast<size_t>(b) * N + i;
    if (i >= nG) {                          // past the sequence's budget: padding
      parent[o] = -1; draft[o] = -1; depth_out[o] = -1;
      if (score_out != nullptr) score_out[o] = -INFINITY;
      continue;
    }
    const int d = static_cast<int>(g_hi[i] & 0xFFFFFFFFull);
    const uint64_t code = g_lo[i];
    int par = -1, tok = root_token != nullptr ? root_token[b] : -1;
    if (d > 0) {
      const int shift = 4 * (kMaxDepth - d);
      const int r = static_cast<int>((code >> shift) & 0xFull);
      tok = s_tok[(d - 1) * K + r];
      const uint64_t pcode = code & ~(0xFull << shift);
      for (int u = 0; u < i; ++u)
        if (g_lo[u] == pcode && static_cast<int>(g_hi[u] & 0xFFFFFFFFull) == d - 1) { par = u; break; }
    }
    parent[o] = par;
    draft[o] = tok;
    depth_out[o] = d;
    if (score_out != nullptr) score_out[o] = from_desc_bits(static_cast<uint32_t>(g_hi[i] >> 32));
  }
  grid_dependents_launch();
}

}  // namespace
}  // namespace jf

namespace {

jf_status build_draft_tree_call(const void* draft_logits, int32_t dtype, const int32_t* root_token,
                                int32_t B, int32_t Dmax, int32_t V, int32_t K, int32_t N,
                                int32_t* cand_token, float* cand_logp, int32_t* parent,
                                int32_t* draft, int32_t* depth, float* score,
                                const int32_t* budget, int32_t* dev_err, jf_stream_t stream) {
  if (draft_logits == nullptr || cand_token == nullptr || cand_logp == nullptr || parent == nullptr ||
      draft == nullptr || depth == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (dtype != JF_DTYPE_BF16 && dtype != JF_DTYPE_F32) return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || Dmax < 1 || K < 1 || N < 1 || V < 1) return JF_ERR_INVALID_ARGUMENT;
  if (K > jf::kMaxK || Dmax > jf::kMaxDepth || N > jf::kMaxTreeN || V < K) return JF_ERR_UNSUPPORTED;
  // the lattice must hold N nodes: 1 + K + K^2 + ... + K^Dmax >= N
  long long lattice = 1, level = 1;
  for (int d = 1; d <= Dmax && lattice < N; ++d) {
    level *= K;
    lattice += level;
  }
  if (lattice < N) return JF_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Dmax > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Rows are split over a cluster of `parts` CTAs only as far as it takes to give the GPU
  // about two CTAs per SM: many rows run one CTA per row (no merge), few rows up to 8.
  const int sms = jf::current_sm_count() > 0 ? jf::current_sm_count() : 148;
  const long long rows = static_cast<long long>(B) * Dmax;
  const int parts = static_cast<int>(std::min<long long>(
      jf::kRowParts, std::max<long long>(1, (2LL * sms + rows - 1) / rows)));
  if (rows * parts > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(rows * parts));
  lc.blockDim = dim3(jf::kTopThreads);
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(parts);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  // A grid that fits in one wave at three CTAs per SM runs the register-capped kernel.
  const bool one_wave = rows * parts <= 3LL * sms;
  const uint16_t* lb = static_cast<const uint16_t*>(draft_logits);
  const float* lf = static_cast<const float*>(draft_logits);
  cudaError_t e;
  if (dtype == JF_DTYPE_BF16)
    e = one_wave ? cudaLaunchKernelEx(&lc, jf::draft_candidates_kernel<uint16_t, 3>, lb, V, K, parts,
                                      cand_token, cand_logp)
                 : cudaLaunchKernelEx(&lc, jf::draft_candidates_kernel<uint16_t, 2>, lb, V, K, parts,
                                      cand_token, cand_logp);
  else
    e = cudaLaunchKernelEx(&lc, jf::draft_candidates_kernel<float, 1>, lf, V, K, parts, cand_token,
                           cand_logp);
  if (e != cudaSuccess) return JF_ERR_CUDA;
  constexpr size_t kTreeSmem = (4 * jf::kMaxTreeN + 4 * jf::kCandMax) * sizeof(uint64_t);
  {
    // Once per device; host threads calling concurrently serialise on the mutex.
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 64 || !attr_set[dev]) {
      if (cudaFuncSetAttribute(jf::best_first_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kTreeSmem)) != cudaSuccess)
        return JF_ERR_CUDA;
      if (dev < 64) attr_set[dev] = true;
    }
  }
  e = jf::launch_pdl(jf::best_first_tree_kernel, dim3(static_cast<unsigned>(B)), dim3(jf::kTreeThreads), kTreeSmem, s,
                     static_cast<const int32_t*>(cand_token), static_cast<const float*>(cand_logp),
                     root_token, Dmax, K, N, parent, draft, depth, score, budget, dev_err);
  return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

}  // namespace

extern "C" jf_status jf_build_draft_tree(const void* draft_logits, int32_t dtype,
                                         const int32_t* root_token, int32_t B, int32_t Dmax,
                                         int32_t V, int32_t K, int32_t N, int32_t* cand_token,
                                         float* cand_logp, int32_t* parent, int32_t* draft,
                                         int32_t* depth, float* score, jf_stream_t stream) {
  return build_draft_tree_call(draft_logits, dtype, root_token, B, Dmax, V, K, N, cand_token,
                               cand_logp, parent, draft, depth, score, nullptr, nullptr, stream);
}

extern "C" jf_status jf_build_draft_tree_ragged(const void* draft_logits, int32_t dtype,
                                                const int32_t* root_token, const int32_t* budget,
                                                int32_t B, int32_t Dmax, int32_t V, int32_t K,
                                                int32_t N, int32_t* cand_token, float* cand_logp,
                                                int32_t* parent, int32_t* draft, int32_t* depth,
                                                float* score, int32_t* dev_err,
                                                jf_stream_t stream) {
  if (budget == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return build_draft_tree_call(draft_logits, dtype, root_token, B, Dmax, V, K, N, cand_token,
                               cand_logp, parent, draft, depth, score, budget, dev_err, stream);
}
