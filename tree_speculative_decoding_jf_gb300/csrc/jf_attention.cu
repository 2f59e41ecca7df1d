// jf_attention.cu -- tree-causal paged attention for sm_103a (TMA + tcgen05/TMEM).
//
// What it computes (JetFlow explainer, technical summary §2 "Tree-Causal Attention Mask"
// and the branch factorisation q(pi(v)|x) = prod_{u in pi(v)} q(y_u | x, h_x, pi_{<u});
// §3 "paged FlashAttention with tree-mask staging" used for tree verification): every
// draft node attends to the whole paged prefix and to its own ancestors only.
//
// Work decomposition.  For sequence b and kv-head g, the G = Hq/Hkv query heads of the N
// nodes form M = N*G rows, node-major (row = node*G + head-in-group), so the G rows of a
// node share one mask row and the contraction has a real M dimension.  Rows come in
// 128-row tiles; one CTA owns NT tiles (NT = 2 when there are at least two) and a range
// of 128-key tiles ("split"), so every K/V tile it loads feeds NT tensor-core tiles.
// Splits and CTA count are chosen on the host from the SM count.  The partial results of
// a unit's splits merge by log-sum-exp either inside a thread-block cluster through
// distributed shared memory or, through a workspace, in a combine kernel launched as a
// programmatic dependent.  With more units than SMs and several row-tile groups per
// kv-head, a stream-K variant runs one CTA per SM over equal ranges of all key tiles.
//
// Roles inside a CTA (128 * (1 + NT) threads):
//   warp 0      TMA producer: page ids travel through registers four tiles ahead (bounds-
//               checked at use); Q is loaded once; per key tile K then V go into a ring
//               (2 K + 3 V stages for D = 128) as one 128-row box per 64-column half when the
//               tile's eight pages are consecutive in the pool, else one box per (page,
//               half) issued by 16 lanes at once.  Pages past the sequence end load as
//               zeros, and V rows past the sequence end in the last tile are zeroed once it
//               has landed (garbage in unused page slots must not meet a zero probability
//               as NaN).  A stage is reloaded once a step record (below) says the MMAs
//               that read it have completed.
//   warp 1      allocates TMEM and issues the MMAs; the whole warp runs the issue loop and
//               one elected lane executes the tcgen05 instructions, a row tile's 8 K-step
//               MMAs from one inline-PTX block:
//                 S_t = Q_t K^T  (128 x 128, fp32 in TMEM),  O_t += P_t V  (P from TMEM).
//               Row tile t's step j (PV of key tile j, then S of key tile j + 1) goes once
//               its softmax and its data voucher have arrived; after the last row tile's
//               step j one commit completes step record j + 1.
//   warps 2..   data vouchers, one per row tile: the last arrival on p_full[t] once the V
//               and K tiles that the step reads have landed.
//   warps 4..   one warpgroup per row tile t: TMEM lane = row, so each thread owns one
//               full score row.  On key tiles reaching positions >= P_b the node's
//               ancestor-mask words are read into registers before the tile's S is waited
//               for and turned into one 32-bit visibility word per 32 keys.  Online softmax
//               in the log2 domain (row max and row sum over independent partial
//               accumulators); the running max is only raised when a tile's max exceeds it
//               by more than 8 (factor 256), which keeps P <= 256 in bf16 and makes the O
//               rescale (TMEM load/scale/store) rare.  P (bf16; hi + lo parts on tree tiles
//               of short prefixes) is written back into the S columns and consumed by the
//               PV MMA from TMEM.
// The control warpgroup hands registers to the softmax warpgroups (setmaxnreg).
// All waits are bounded (see jf_sm100.cuh); on a timeout the CTA records
// JF_DEVERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "jf_common.cuh"
#include "jf_sm100.cuh"

namespace jf {
namespace {

constexpr int kKeyTile = 128;     // keys per pipeline stage
constexpr int kRowTile = 128;     // rows per tensor-core tile (TMEM lanes)
constexpr int kPage = 16;
constexpr int kPagesPerTile = kKeyTile / kPage;
constexpr float kRescaleThreshold = 8.0f;               // log2 units
// Sequences with fewer prefix keys than this store P as hi + lo bf16 parts on the key
// tiles that hold tree keys (see row_probs); longer prefixes give every row at least this
// many visible keys, over which the bf16 rounding of P averages out.
constexpr int kSplitPrefix = 128;
constexpr int kLptMaxB = 256;                           // longest-first dispatch up to this B

// Step records: record i completes once step i - 1 (every row tile's PV of key tile i - 1
// and S of key tile i) has finished on the tensor cores; record 0 marks the first S MMAs.
constexpr int kStepRing = 8;

template <int NT, int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                  // 128-byte swizzle atoms per row
  // V stages are released only when a tile's last PV MMA completes, K stages as soon as
  // the next tile's S MMAs are issued, so V gets the deeper ring.
  static constexpr int kKStages = (D == 64) ? 4 : 2;
  static constexpr int kVStages = (D == 64) ? 6 : 3;
  // K tile j may load after record j - kKStages, V tile j after record j - kVStages + 1;
  // the producer loads both after record j - kStageLag.
  static constexpr int kStageLag = kKStages < kVStages - 1 ? kKStages : kVStages - 1;
  static constexpr int kTileBytes = kRowTile * D * 2;     // one 128-row bf16 tile
  static constexpr int kHalfBytes = kRowTile * 128;       // one 64-column half of a tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NT * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kRingBytes = (kKStages + kVStages) * kTileBytes;
  // After the last MMA the ring holds the epilogue: fp32 rows [NT][128][D], then LSEs.
  static constexpr int kPartLseOff = kKOff + NT * 2 * kTileBytes;
  static_assert(NT * 2 * kTileBytes + NT * kRowTile * 4 <= kRingBytes, "epilogue fits the ring");
  static constexpr int kSmemBytes = kKOff + kRingBytes + 1024;
  static constexpr int kThreads = 128 * (1 + NT);
  static constexpr uint32_t kTmemCols = (NT == 2) ? 512 : 256;
  static constexpr uint32_t kTmemO = 0;                   // O_t at column t*128
  static constexpr uint32_t kTmemS = NT * 128;            // S_t (and P_t) at kTmemS + t*128
};

struct AttnParams {
  const int32_t* block_table;
  const int32_t* prefix_len;
  const uint64_t* mask;
  uint16_t* out;        // bf16 [B][N][Hq][D]      (splits == 1)
  float* lse;           // [B][Hq][N] or null      (splits == 1)
  float* ws_o;          // [B][Hkv][splits][M][D]  (splits > 1), row r = node * G + head
  float* ws_lse;        // [B][Hkv][splits][M]     (log2 domain)
  int* ws_desc;         // stream-K: per range boundary, the pair it splits (8 ints)
  int32_t* dev_err;
  int B, N, Hq, Hkv, G, W, max_pages, num_pages;
  int n_groups, splits, chunk_tiles, M;
  int cluster_merge;    // 1: the splits of a unit form one cluster and merge through DSMEM
  float scale_log2;     // softmax scale * log2(e)
  const int32_t* tree_len;  // ragged calls: nodes per sequence (else null: N everywhere)
  const int32_t* cu;        // packed calls: cumulative node counts [B + 1] (else null)
  long long T;              // packed calls: total nodes (rows of q, out, mask)
};

// Packed calls (cu != null) keep q, out and mask as [T][...] rows, sequence b's nodes at
// rows cu[b] .. cu[b + 1] - 1, and lse as [Hq][T]; the others [B][N][...] and [B][Hq][N].
// row0 is the sequence's first row (b * N when not packed).
__device__ __forceinline__ size_t out_row(long long row0, int i, int Hq, int h) {
  return static_cast<size_t>((row0 + i) * Hq + h);
}
__device__ __forceinline__ size_t lse_index(bool packed, long long row0, long long T, int b,
                                            int h, int i, int Hq, int N) {
  return packed ? static_cast<size_t>(h * T + row0 + i)
                : static_cast<size_t>((static_cast<long long>(b) * Hq + h) * N + i);
}

// Time limit of the kernels' bounded waits on their own pipeline (the waits that drain
// copies and MMAs before a CTA exits always allow kWaitLimitNs).  Lowered only through
// jf_debug_set_wait_limit_ns, to test the timeout path.
__device__ uint64_t g_wait_limit_ns = kWaitLimitNs;
// Test hook: non-zero makes the data-voucher warps withhold their arrivals, so the MMA
// issuer waits for a barrier phase that can never complete (a wait nothing satisfies).
__device__ int g_withhold_vouchers = 0;

// Nodes of sequence b's tree: N, or tree_len[b] clamped to [1, N] for ragged calls.  The
// tree's keys are the n positions after the prefix, so the sequence has P_b + n keys.
__device__ __forceinline__ int tree_nodes(const int32_t* tree_len, int b, int N) {
  return tree_len == nullptr ? N : max(1, min(tree_len[b], N));
}

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t wlim) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, wlim) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

__device__ __forceinline__ void set_abort(volatile int* abort, int32_t* dev_err) {
  if (*abort == 0) {
    *abort = 1;
    report(dev_err, JF_DEVERR_TIMEOUT);
  }
}

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Paired fp32 arithmetic (one instruction for two lanes of data) and a 3-input max.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Bits [rel, rel + 32) of the 192-bit little-endian window w[0..3) (zero outside it).
__device__ __forceinline__ uint32_t window_bits32(const uint64_t (&w)[3], int rel) {
  if (rel <= -32 || rel >= 192) return 0u;
  if (rel < 0) return static_cast<uint32_t>(w[0] << (-rel));
  const int wi = rel >> 6, off = rel & 63;
  const uint64_t lo = wi == 0 ? w[0] : (wi == 1 ? w[1] : w[2]);
  const uint64_t hi = wi == 0 ? w[1] : (wi == 1 ? w[2] : 0ull);
  uint64_t v = lo >> off;
  if (off > 32) v |= hi << (64 - off);
  return static_cast<uint32_t>(v);
}

// Four 32-column TMEM loads followed by one wait that ties all 128 registers.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  tmem_ld32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  tmem_ld32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
  tmem_ld32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&r[64]));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&r[96]));
}

// Probabilities of one 128-score row (log2 domain: p = 2^(s * sl2 - m)), written back to
// the row's TMEM S columns as the bf16 A operand of the PV MMA: P in columns 0..63 (two
// keys per 32-bit column).  With SPLIT, P is also stored as a second bf16 part
// lo = bf16(p - bf16(p)) in columns 64..127 and the MMA issuer adds a PV MMA on it, so the
// probabilities that reach the tensor cores carry a relative error of about 2^-17 instead
// of bf16's 2^-9.  That matters on tiles that hold tree keys: a row with only a few
// visible keys gets no averaging of the rounding errors, and the output of such a row can
// be small where its values cancel.  Returns the fp32 row sum.
template <bool SPLIT>
__device__ __forceinline__ float row_probs(const float* sv, float sl2, float neg, uint32_t tS) {
  const uint64_t sl2x2 = f2(sl2, sl2), negx2 = f2(neg, neg);
  uint64_t ls2[2] = {0ull, 0ull};       // paired partial row sums (0ull == {+0, +0})
  if constexpr (SPLIT) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {        // quarters of 32 keys keep few registers live
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int cc = 16 * h + c;
        float x0, x1;
        f2_split(ffma2(f2(sv[2 * cc], sv[2 * cc + 1]), sl2x2, negx2), x0, x1);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        ls2[c & 1] = fadd2(ls2[c & 1], f2(p0, p1));
        ph[c] = pack_bf16x2(p0, p1);
        pl[c] = pack_bf16x2(p0 - __uint_as_float(ph[c] << 16), p1 - __uint_as_float(ph[c] & 0xFFFF0000u));
      }
      tmem_st16(tS + 16 * h, ph);
      tmem_st16(tS + 64 + 16 * h, pl);
    }
  } else {
    uint32_t pk[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      float x0, x1;
      f2_split(ffma2(f2(sv[2 * c], sv[2 * c + 1]), sl2x2, negx2), x0, x1);
      const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
      ls2[c & 1] = fadd2(ls2[c & 1], f2(p0, p1));
      pk[c] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
    tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
  }
  float la, lb, lc, ld;
  f2_split(ls2[0], la, lb);
  f2_split(ls2[1], lc, ld);
  return (la + lb) + (lc + ld);
}

// One key tile of the online softmax for the calling thread's score row (its TMEM lane):
// waits for the tile's S, applies visibility, raises the running maximum when needed,
// writes P back to TMEM, rescales O when the maximum moved, and arrives on p_full.
// MASKED tiles reach positions >= P (tree keys, possibly keys past the sequence end): the
// node's ancestor words are loaded before the wait.  SPLIT (only on masked tiles of
// sequences with a prefix shorter than kSplitPrefix) stores P as hi + lo parts.  Prefix
// tiles take the MASKED = false instantiation, whose loop carries none of that code.  With
// a non-null lo_flag the writer thread records SPLIT there for the MMA issuer once the
// tile's S has arrived.  Returns false if the wait gave up.
template <bool MASKED, bool SPLIT, int D>
__device__ __forceinline__ bool softmax_tile(uint64_t* s_full_bar, uint32_t parity,
                                             volatile int* abort, uint64_t* p_full_bar,
                                             uint32_t tS, uint32_t tO, const uint64_t* mrow,
                                             bool valid, int W, int key0, int P, int L, float sl2,
                                             bool not_first, volatile int* lo_flag, bool writer,
                                             float& m_run, float& l, uint64_t wlim) {
  uint64_t mw[3] = {0ull, 0ull, 0ull};
  const int w_lo = MASKED ? (max(key0 - P, 0) >> 6) : 0;
  if constexpr (MASKED) {
    if (valid) {
#pragma unroll
      for (int u = 0; u < 3; ++u)
        if (w_lo + u < W) mw[u] = __ldg(reinterpret_cast<const unsigned long long*>(mrow) + w_lo + u);
    }
  }
  if (!wait_warp(s_full_bar, parity, abort, wlim)) return false;
  if (lo_flag != nullptr && writer) *lo_flag = SPLIT ? 1 : 0;
  tc_fence_after();
  uint32_t sr[128];
  tmem_ld128(tS, sr);
  float* sv = reinterpret_cast<float*>(sr);
  if constexpr (MASKED) {
    // Visibility of the tile's 128 keys as four 32-bit words: prefix keys always, tree key
    // j iff bit j of the node's ancestor mask, nothing past the sequence end.
    const int pre = min(max(P - key0, 0), kKeyTile);
    const int end = min(max(L - key0, 0), kKeyTile);
    uint32_t vis[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int c0 = 32 * w;
      uint32_t m = window_bits32(mw, key0 + c0 - P - 64 * w_lo);
      const int np = min(max(pre - c0, 0), 32);
      const int ne = min(max(end - c0, 0), 32);
      m |= np >= 32 ? 0xFFFFFFFFu : ((1u << np) - 1u);
      m &= ne >= 32 ? 0xFFFFFFFFu : ((1u << ne) - 1u);
      vis[w] = m;
    }
#pragma unroll
    for (int c = 0; c < kKeyTile; ++c)
      if (!((vis[c >> 5] >> (c & 31)) & 1u)) sv[c] = -INFINITY;
  }
  float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
  for (int c = 4; c < kKeyTile; c += 2) m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], sv[c], sv[c + 1]);
  const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
  const float mt = mx * sl2;
  const bool raise = mt > m_run + kRescaleThreshold;
  const float m_old = m_run;
  if (raise) m_run = mt;
  const float corr = raise ? fast_exp2(m_old - m_run) : 1.f;   // 0 when m_old = -inf
  const float neg = (m_run == -INFINITY) ? 0.f : -m_run;
  l = l * corr + row_probs<SPLIT>(sv, sl2, neg, tS);
  // O holds PV of the earlier tiles (complete: this tile's S was committed after them).
  const bool need = raise && not_first && m_old != -INFINITY;
  if (__any_sync(0xffffffffu, need)) {
    const float f = need ? corr : 1.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
      tmem_ld_wait(o);
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
      tmem_st32(tO + c * 32, o);
    }
  }
  tmem_st_wait();
  tc_fence_before();
  mbar_arrive(p_full_bar);
  return true;
}

// Split partials of one unit live in the shared memory of the cluster's CTAs: normalised
// fp32 rows in the (idle) K/V ring, row r's 16-byte chunk k at chunk k ^ (r % 8), and the
// log2-domain LSE of each row right after them.  CTA `rank` merges rows
// [rank * R / S, (rank + 1) * R / S) of the unit's R = NT * 128 rows through distributed
// shared memory, batching the remote loads so each phase costs about one round trip.
template <int NT, int D>
__device__ __forceinline__ float* part_row(uint8_t* sm, int t, int row) {
  return reinterpret_cast<float*>(sm + Cfg<NT, D>::kKOff + (t * kRowTile + row) * (D * 4));
}
template <int NT, int D>
__device__ __forceinline__ float* part_lse(uint8_t* sm, int t) {
  return reinterpret_cast<float*>(sm + Cfg<NT, D>::kPartLseOff + t * kRowTile * 4);
}

// Out of line: the merge runs once per CTA and its code stays out of the hot loops' way.
struct MergeArgs {
  uint16_t* out;
  float* lse;
  int N, Hq, G, M, splits;
  long long row0, T;   // the sequence's first row; total rows (packed calls)
  int rows;            // rows the sequence owns: N, or its node count when packed
  bool packed;
};

template <int NT, int D>
__device__ __noinline__ void merge_cluster(uint8_t* sm, const MergeArgs p, int b, int g, int mp, int rank) {
  constexpr int kChunks = D / 4;                         // 16-byte chunks per fp32 row
  constexpr int kMaxSplits = 8;
  cluster_sync();                                        // every split's partial is written
  const int S = p.splits;
  const int R = NT * kRowTile;
  const int per = (R + S - 1) / S;
  const int r_lo = rank * per;
  const int nrows = max(0, min(R, r_lo + per) - r_lo);
  // Scratch in this CTA's (idle) Q area: per merged row, the split weights.
  float* s_w = reinterpret_cast<float*>(sm + Cfg<NT, D>::kQOff);          // [nrows][8]
  // 1) every (row, split) LSE in one batch of remote loads
  for (int e = threadIdx.x; e < nrows * S; e += blockDim.x) {
    const int rr = r_lo + e / S, s2 = e % S;
    s_w[(e / S) * kMaxSplits + s2] =
        dsmem_ld_f32(dsmem_addr(part_lse<NT, D>(sm, rr / kRowTile) + rr % kRowTile, s2));
  }
  __syncthreads();
  // 2) per row: weights 2^(lse_s - max) / sum and the merged LSE
  for (int e = threadIdx.x; e < nrows; e += blockDim.x) {
    float* w = s_w + e * kMaxSplits;
    float mx = -INFINITY;
    for (int s2 = 0; s2 < S; ++s2) mx = fmaxf(mx, w[s2]);
    float sum = 0.f;
    for (int s2 = 0; s2 < S; ++s2) {
      const float x = (w[s2] == -INFINITY) ? 0.f : exp2f(w[s2] - mx);
      w[s2] = x;
      sum += x;
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int s2 = 0; s2 < S; ++s2) w[s2] *= inv;
    const int rr = r_lo + e;
    const int rg = (mp * NT + rr / kRowTile) * kRowTile + rr % kRowTile;
    if (p.lse != nullptr && rg < p.M && rg / p.G < p.rows) {
      const int i = rg / p.G, h = g * p.G + (rg % p.G);
      p.lse[lse_index(p.packed, p.row0, p.T, b, h, i, p.Hq, p.N)] =
          (sum > 0.f ? mx + __log2f(sum) : -INFINITY) * 0.69314718055994531f;
    }
  }
  __syncthreads();
  // 3) (row, 16-byte chunk) items: all splits' chunks are requested before any is used
  for (int e = threadIdx.x; e < nrows * kChunks; e += blockDim.x) {
    const int el = e / kChunks, k = e % kChunks;
    const int rr = r_lo + el;
    const int t = rr / kRowTile, row = rr % kRowTile;
    const int rg = (mp * NT + t) * kRowTile + row;
    if (rg >= p.M || rg / p.G >= p.rows) continue;
    const float* w = s_w + el * kMaxSplits;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(part_row<NT, D>(sm, t, row)) +
                         ((static_cast<uint32_t>(k) ^ static_cast<uint32_t>(row & 7)) << 4);
    float4 v[kMaxSplits];
#pragma unroll
    for (int s2 = 0; s2 < kMaxSplits; ++s2)
      if (s2 < S && w[s2] != 0.f) v[s2] = dsmem_ld_f32x4(dsmem_addr(src, s2));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s2 = 0; s2 < kMaxSplits; ++s2)
      if (s2 < S && w[s2] != 0.f) {
        acc.x += w[s2] * v[s2].x; acc.y += w[s2] * v[s2].y;
        acc.z += w[s2] * v[s2].z; acc.w += w[s2] * v[s2].w;
      }
    const int i = rg / p.G, h = g * p.G + (rg % p.G);
    uint16_t* dst = p.out + out_row(p.row0, i, p.Hq, h) * D + k * 4;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
  cluster_sync();                                        // nobody leaves while others read it
}

// O += P_lo V from the second bf16 part of P (columns 64..127 of a row tile's S region).
// Out of line: the MMA issuer's steady-state loop carries none of this code.
__device__ __noinline__ void issue_pv_lo(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, uint32_t idO) {
  mma_ts_tile(d_tmem, a_tmem + 64, db, idO, true);
}

// Longest sequences first: with one CTA per unit and ragged prefixes, CTAs are handed to
// SMs in block order, so ordering sequences by length (descending, ties by index) keeps
// one long sequence from starting in the last wave.  Every CTA of the grid ranks all B
// lengths itself (the same order everywhere) and grid slot `slot` takes the sequence of
// rank `slot`.  Kept out of line: only longest-first launches call it.
__device__ __noinline__ int lpt_sequence(const int32_t* prefix_len, int B, int capn, int slot) {
  __shared__ int s_len[kLptMaxB];
  __shared__ int s_seq;
  for (int u = threadIdx.x; u < B; u += blockDim.x) s_len[u] = max(0, min(prefix_len[u], capn));
  __syncthreads();
  for (int u = threadIdx.x; u < B; u += blockDim.x) {
    const int lu = s_len[u];
    int rank = 0;
    for (int v = 0; v < B; ++v) {
      const int lv = s_len[v];
      rank += (lv > lu || (lv == lu && v < u)) ? 1 : 0;
    }
    if (rank == slot) s_seq = u;
  }
  __syncthreads();
  return s_seq;
}

// LPT: the grid's sequence slots are length ranks (longest-first dispatch); a separate
// instantiation, so launches without it run exactly the kernel they would otherwise.
template <int NT, int D, bool LPT>
__global__ void __launch_bounds__(Cfg<NT, D>::kThreads, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap kmap_run,
                          const __grid_constant__ CUtensorMap vmap_run,
                          const __grid_constant__ CUtensorMap omap,
                          const __grid_constant__ CUtensorMap wmap, const AttnParams p) {
  using C = Cfg<NT, D>;
  constexpr int SK = C::kKStages;
  constexpr int SV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t q_full, o_full, fin;
  __shared__ uint64_t k_full[SK], v_full[SV], step_done[kStepRing];
  __shared__ uint64_t s_full[NT], p_full[NT], v_tail;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  uint8_t* q_s = sm + C::kQOff;
  uint8_t* k_s = sm + C::kKOff;
  uint8_t* v_s = sm + C::kVOff;

  // ---- which (b, kv-head, row-tile group, split) this CTA owns; split fastest, then the
  // row-tile group, so CTAs that read the same K/V tiles run side by side.
  int bid = blockIdx.x;
  const int split = bid % p.splits;      // == rank in the cluster when merging through DSMEM
  bid /= p.splits;
  const int mp = bid % p.n_groups;
  bid /= p.n_groups;
  const int g = bid % p.Hkv;
  const int slot = bid / p.Hkv;          // a sequence, or its length rank under LPT
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Barriers and descriptor prefetches touch no input, so they overlap the tail of the
  // previous kernel (programmatic dependent launch).
  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&o_full, 1);
    mbar_init(&fin, 1);
    for (int st = 0; st < SK; ++st) mbar_init(&k_full[st], 1);
    for (int st = 0; st < SV; ++st) mbar_init(&v_full[st], 1);
    for (int st = 0; st < kStepRing; ++st) mbar_init(&step_done[st], 1);
    for (int t = 0; t < NT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128 + 1);   // the softmax warpgroup + its data voucher
    }
    mbar_init(&v_tail, 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&kmap_run);
    tma_prefetch_desc(&vmap_run);
  }
  const uint64_t wlim = g_wait_limit_ns;
  grid_dependency_wait();

  int b = slot;
  if constexpr (LPT) b = lpt_sequence(p.prefix_len, p.B, p.max_pages * kPage - p.N, slot);

  // Q does not depend on the sequence length: its load starts before anything is read
  // (packed calls read the sequence's first row first; rows of the next sequence or past
  // the end that a tile reaches are padding rows, their results never stored).
  if (threadIdx.x == 0) {
    int qrow0 = 0, qb = b;
    if (p.cu != nullptr) {
      qrow0 = static_cast<int>(seq_span(p.cu, nullptr, b, p.N, p.T).row0);
      qb = 0;
    }
    mbar_arrive_expect_tx(&q_full, NT * C::kTileBytes);
    for (int t = 0; t < NT; ++t) {
      const int node0 = ((mp * NT + t) * kRowTile) / p.G;
      for (int hh = 0; hh < C::kHalves; ++hh)
        tma_load_4d(q_s + t * C::kTileBytes + hh * C::kHalfBytes, &qmap, &q_full, hh * 64,
                    g * p.G, qrow0 + node0, qb);
    }
  }
  // The first key tiles' page ids are read together with the prefix length (one round
  // trip for both) and parked in shared memory; they are checked against the sequence end
  // once it is known.
  constexpr int kLookahead = 4;
  const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
  __shared__ int s_pid0[kLookahead][kPagesPerTile];
  if (warp == 0 && lane < kPagesPerTile) {
    int raw[kLookahead];
#pragma unroll
    for (int u = 0; u < kLookahead; ++u) {
      const int pl = (split * p.chunk_tiles + u) * kPagesPerTile + lane;
      raw[u] = pl < p.max_pages ? __ldg(bt + pl) : p.num_pages;
    }
#pragma unroll
    for (int u = 0; u < kLookahead; ++u) s_pid0[u][lane] = raw[u];
  }

  const int cap = p.max_pages * kPage;
  const SeqSpan sp = seq_span(p.cu, p.tree_len, b, p.N, p.T);
  const int nt = sp.n;
  if (!sp.ok && threadIdx.x == 0) report(p.dev_err, JF_DEVERR_BAD_TREE_LEN);
  int P = p.prefix_len[b];
  if (P < 0 || P > cap - nt) {
    if (threadIdx.x == 0) report(p.dev_err, JF_DEVERR_BAD_PREFIX);
    P = max(0, min(P, cap - nt));
  }
  const int L = P + nt;
  const int ntiles = (L + kKeyTile - 1) / kKeyTile;
  const int k0 = split * p.chunk_tiles;
  const int k1 = min(ntiles, k0 + p.chunk_tiles);
  const int T = max(0, k1 - k0);

  // Ragged and packed calls: a row-tile group whose rows all belong to padding nodes
  // (node >= n_b) has nothing to compute (those rows carry no meaning; a packed sequence
  // with a bad span has n_b = 0).  The splits of a unit share the group, so the CTAs of a
  // merging cluster leave together.  The Q load is drained first.
  if ((p.tree_len != nullptr || p.cu != nullptr) && (mp * NT * kRowTile) / p.G >= nt) {
    if (threadIdx.x == 0) {
      int zero = 0;
      mbar_wait(&q_full, 0, &zero);
    }
    return;
  }

  if (T == 0) {
    // An empty split still drains its Q load before the shared memory is reused or freed.
    if (threadIdx.x == 0) {
      int zero = 0;
      mbar_wait(&q_full, 0, &zero);
    }
    if (p.cluster_merge) {            // weight 0, but it joins the merge
      __syncthreads();
      for (int t = 0; t < NT; ++t)
        for (int e = threadIdx.x; e < kRowTile; e += blockDim.x) part_lse<NT, D>(sm, t)[e] = -INFINITY;
      merge_cluster<NT, D>(sm, MergeArgs{p.out, p.lse, p.N, p.Hq, p.G, p.M, p.splits, sp.row0, p.T, sp.rows, p.cu != nullptr}, b, g, mp, split);
      return;
    }
    if (warp >= 4) {                  // split past the sequence: an empty partial (weight 0)
      const int t = (warp >> 2) - 1;
      const int r = (mp * NT + t) * kRowTile + ((warp & 3) * 32 + lane);
      if (r < p.M) {
        const size_t prow = ((static_cast<size_t>(b) * p.Hkv + g) * p.splits + split) * p.M + r;
        p.ws_lse[prow] = -INFINITY;
        float4* dst = reinterpret_cast<float4*>(p.ws_o + prow * D);
        for (int d = 0; d < D / 4; ++d) dst[d] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }

  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // 384 threads x 168 registers at launch (NT == 2): the control warpgroup hands
  // registers to the two softmax warpgroups (96 * 128 + 200 * 256 <= 168 * 384).  The
  // adjustment sits inside each role's branch so the compiler budgets each region.
  if (warp < 4) {
  if constexpr (NT == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
  if (warp == 0) {
    // ================================================================ TMA producer
    // Page ids travel through registers: lane q < 8 holds page q of the next kLookahead
    // tiles, loaded kLookahead tiles before use so the block-table latency overlaps the
    // wait for free stages.  Pages past the sequence end (and malformed ids, reported)
    // become the out-of-bounds id num_pages, which TMA fills with zeros.
    auto load_pid = [&](int j) -> int {
      const int pl = (k0 + j) * kPagesPerTile + lane;
      if (lane >= kPagesPerTile || j >= T || pl * kPage >= L) return p.num_pages;
      return __ldg(bt + pl);
    };
    int pid[kLookahead];
#pragma unroll
    for (int u = 0; u < kLookahead; ++u) {
      const int pl = (k0 + u) * kPagesPerTile + lane;
      pid[u] = (lane >= kPagesPerTile || u >= T || pl * kPage >= L) ? p.num_pages : s_pid0[u][lane];
    }
    int bad = 0;
    // When the tile's eight pages are consecutive in the pool (page q == page 0 + q) one
    // 128-row box per 64-column half moves the whole tile; otherwise one box per (page,
    // half), issued by lanes [0, 8 * halves) in parallel.
    auto issue = [&](uint8_t* ring, const CUtensorMap* map, const CUtensorMap* map_run,
                     uint64_t* full, int st, int page, int page0, bool run) {
      if (run) {
        if (lane < C::kHalves)
          tma_load_3d(ring + st * C::kTileBytes + lane * C::kHalfBytes, map_run, full, lane * 64, g,
                      page0 * kPage);
      } else if (lane < kPagesPerTile * C::kHalves) {
        const int q = lane % kPagesPerTile, hh = lane / kPagesPerTile;
        tma_load_3d(ring + st * C::kTileBytes + hh * C::kHalfBytes + q * (kPage * 128), map, full,
                    hh * 64, g, page * kPage);
      }
    };
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      int mine = pid[0];
      if (mine < 0 || mine > p.num_pages) { bad = 1; mine = p.num_pages; }
      else if (mine == p.num_pages && lane < kPagesPerTile &&
               ((k0 + j) * kPagesPerTile + lane) * kPage < L) bad = 1;
      const int page = __shfl_sync(0xffffffffu, mine, lane % kPagesPerTile);
      const int page0 = __shfl_sync(0xffffffffu, mine, 0);
      const bool run = __all_sync(0xffffffffu, page == page0 + lane % kPagesPerTile);
#pragma unroll
      for (int u = 0; u < kLookahead - 1; ++u) pid[u] = pid[u + 1];
      pid[kLookahead - 1] = load_pid(j + kLookahead);
      const int sk = j % SK, sv = j % SV;
      // K tile j reuses the stage of K tile j - SK, last read by the S MMAs of step
      // j - SK - 1; V tile j reuses that of V tile j - SV, read in step j - SV.  One step
      // record covers both (see Cfg::kStageLag).
      const int rec = j - C::kStageLag;
      int okl = 1;
      if (lane == 0) {
        if (rec >= 0 && !mbar_wait(&step_done[rec % kStepRing],
                                   static_cast<uint32_t>(rec / kStepRing) & 1u, abort, wlim)) {
          okl = 0;
        } else {
          mbar_arrive_expect_tx(&k_full[sk], C::kTileBytes);
          mbar_arrive_expect_tx(&v_full[sv], C::kTileBytes);
        }
      }
      if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
      issue(k_s, &kmap, &kmap_run, &k_full[sk], sk, page, page0, run);
      k_issued = j + 1;
      issue(v_s, &vmap, &vmap_run, &v_full[sv], sv, page, page0, run);
      v_issued = j + 1;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.dev_err, JF_DEVERR_BAD_PAGE);
    // V rows past the sequence end in the last key tile hold whatever the unused page
    // slots contain; they meet a zero probability, so they must be finite: zero them once
    // the tile has landed, then let the MMA issuer use it.
    const int last_key0 = (k0 + T - 1) * kKeyTile;
    if (ok && last_key0 + kKeyTile > L) {
      const int jl = T - 1;
      if (!wait_warp(&v_full[jl % SV], static_cast<uint32_t>(jl / SV) & 1u, abort, wlim)) {
        ok = false;
      } else {
        const int r0 = L - last_key0;
        uint8_t* vt = v_s + (jl % SV) * C::kTileBytes;
        const int per_half = (kKeyTile - r0) * 8;                 // 16-byte chunks per half
        for (int c = lane; c < per_half * C::kHalves; c += 32) {
          const int hh = c / per_half, rem = c % per_half;
          *reinterpret_cast<uint4*>(vt + hh * C::kHalfBytes + (r0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&v_tail);
      }
    }
    if (!ok && lane == 0) set_abort(abort, p.dev_err);
    __syncwarp();
    // Drain: make sure no copy is still landing in shared memory when the CTA exits.
    if (lane == 0) {
      int zero_q = 0;
      mbar_wait(&q_full, 0, &zero_q);
      int zero = 0;
      for (int j = max(0, k_issued - SK); j < k_issued; ++j)
        mbar_wait(&k_full[j % SK], static_cast<uint32_t>(j / SK) & 1u, &zero);
      for (int j = max(0, v_issued - SV); j < v_issued; ++j)
        mbar_wait(&v_full[j % SV], static_cast<uint32_t>(j / SV) & 1u, &zero);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t idS = idesc_bf16(kRowTile, kKeyTile, false, false);
    constexpr uint32_t idO = idesc_bf16(kRowTile, D, false, true);
    // Matrix descriptors of the first Q tile / K stage / V stage; a tile, a stage or a
    // K-step only moves the 14-bit start-address field (addresses < 256 KB, no carry).
    const uint64_t dq = desc_sw128(smem_u32(q_s), 16, 1024);
    const uint64_t dk = desc_sw128(smem_u32(k_s), 16, 1024);
    const uint64_t dv = desc_sw128(smem_u32(v_s), C::kHalfBytes, 1024);
    auto issue_s = [&](int t, int st) {
      const uint64_t da = dq + static_cast<uint64_t>((t * C::kTileBytes) >> 4);
      const uint64_t db = dk + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
      const uint32_t d_tmem = tmem + C::kTmemS + t * 128;
      mma_ss_tile<D / 16>(d_tmem, da, db, idS);
    };
    // O_t (+)= P_t V; with `lo`, also O_t += P_lo V from the second bf16 part of P (columns
    // 64..127 of the S region), issued before the next S MMA overwrites those columns.
    auto issue_pv = [&](int t, int st, bool acc, bool lo) {
      const uint64_t db = dv + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
      const uint32_t d_tmem = tmem + C::kTmemO + t * 128;
      const uint32_t a_tmem = tmem + C::kTmemS + t * 128;
      mma_ts_tile(d_tmem, a_tmem, db, idO, acc);
      if (lo) issue_pv_lo(d_tmem, a_tmem, db, idO);
    };
    bool ok = wait_warp(&q_full, 0, abort, wlim) && wait_warp(&k_full[0], 0, abort, wlim);
    if (ok) {
      // The whole warp runs this loop (warp-uniform counters and descriptors); the MMA and
      // commit wrappers issue from one elected lane.
      tc_fence_after();
      for (int t = 0; t < NT; ++t) {
        issue_s(t, 0);
        mma_commit(&s_full[t]);
      }
      mma_commit(&step_done[0]);
      // One warp drives every row tile.  Row tile t's next step is PV of key tile jn[t]
      // followed by S of key tile jn[t] + 1.  It may go once p_full[t] completes: the
      // tile's softmax has arrived and so has its voucher warp, which arrives only after V
      // tile jn[t] and K tile jn[t] + 1 have landed, so a step costs the issuer a single
      // barrier probe.  The warp probes the tiles in turn and issues whichever step is
      // ready, so one tile's softmax never holds back the other tile's MMAs.
      // After the last row tile's step j one commit completes step record j + 1.
      // When P is stored as hi + lo (prefix shorter than kSplitPrefix), steps from j_tree on
      // cover key tiles that hold tree keys: the polling loop stops before them and an
      // ordered tail issues them with the second (lo) PV MMA, so the steady-state loop
      // stays free of that code.
      const int j_tree = P < kSplitPrefix ? min(max(P / kKeyTile - k0, 0), T) : T;
      int jn[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) jn[t] = 0;
      int left = NT * j_tree;
      uint32_t idle = 0;
      uint64_t idle_since = 0;
      while (left > 0) {
        bool progressed = false;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int j = jn[t];
          if (j >= j_tree) continue;
          // lane 0's probe decides for the warp
          if (__shfl_sync(0xffffffffu, mbar_try_wait(&p_full[t], static_cast<uint32_t>(j) & 1u) ? 1 : 0, 0) == 0)
            continue;
          bool last = true;                  // the other row tiles are past key tile j
#pragma unroll
          for (int u = 0; u < NT; ++u)
            if (u != t && jn[u] <= j) last = false;
          tc_fence_after();
          issue_pv(t, j % SV, j > 0, false);
          if (j + 1 < T) {
            issue_s(t, (j + 1) % SK);
            mma_commit(&s_full[t]);
          }
          if (last) mma_commit(&step_done[(j + 1) % kStepRing]);
          jn[t] = j + 1;
          --left;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else {
          if (idle == 0) idle_since = global_timer_ns();
          if ((++idle & 255u) == 0u &&
              __shfl_sync(0xffffffffu, (*abort || global_timer_ns() - idle_since > wlim) ? 1 : 0, 0) != 0) {
            ok = false;
            break;
          }
        }
      }
      for (int j = j_tree; j < T && ok; ++j) {
        for (int t = 0; t < NT && ok; ++t) {
          if (!wait_warp(&p_full[t], static_cast<uint32_t>(j) & 1u, abort, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, j % SV, j > 0, true);
          if (j + 1 < T) {
            issue_s(t, (j + 1) % SK);
            mma_commit(&s_full[t]);
          }
          if (t == NT - 1) mma_commit(&step_done[(j + 1) % kStepRing]);
        }
      }
    }
    if (!ok && lane == 0) set_abort(abort, p.dev_err);
    if (ok) mma_commit(&o_full);
    mma_commit(&fin);   // all MMAs done before TMEM is released
    {
      int zero = 0;
      wait_warp(&fin, 0, &zero, kWaitLimitNs);
    }
  } else if (warp >= 2 && warp < 2 + NT) {
    // ================================================================ data vouchers
    // Warp 2 + t adds the last arrival to p_full[t] for key tile j once V tile j, K tile
    // j + 1 and (for the last tile) the zeroed V tail have landed, so the MMA issuer needs
    // no probe of its own on the K/V barriers.  It waits for phase j - 1 of p_full[t]
    // first, so its arrival cannot count toward an earlier phase.
    const int t = warp - 2;
    const bool tail = (k0 + T) * kKeyTile > L;
    if (lane == 0 && g_withhold_vouchers == 0) {
      for (int j = 0; j < T; ++j) {
        const bool ready =
            (j == 0 || mbar_wait(&p_full[t], static_cast<uint32_t>(j - 1) & 1u, abort, wlim)) &&
            mbar_wait(&v_full[j % SV], static_cast<uint32_t>(j / SV) & 1u, abort, wlim) &&
            (j + 1 >= T ||
             mbar_wait(&k_full[(j + 1) % SK], static_cast<uint32_t>((j + 1) / SK) & 1u, abort, wlim)) &&
            (j + 1 < T || !tail || mbar_wait(&v_tail, 0u, abort, wlim));
        if (!ready) {
          set_abort(abort, p.dev_err);
          break;
        }
        mbar_arrive(&p_full[t]);
      }
    }
    __syncwarp();
  }
  } else {
    if constexpr (NT == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
    // ================================================================ softmax / epilogue
    const int t = (warp >> 2) - 1;
    const int wq = warp & 3;
    const int rl = wq * 32 + lane;                       // row within the tile = TMEM lane
    const int r = (mp * NT + t) * kRowTile + rl;
    const bool valid = r < p.M && r / p.G < sp.rows;    // the row exists in memory
    const int node_base = ((mp * NT + t) * kRowTile) / p.G;
    const int i = r / p.G;
    const int h = g * p.G + (r % p.G);
    const int W = p.W;
    // The node's ancestor-mask words a tile needs (at most three 64-bit words for 128
    // keys) are loaded into registers before the tile's S is waited for.
    const uint64_t* mrow = p.mask + (sp.row0 + (valid ? i : 0)) * W;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + C::kTmemS + t * 128 + lane_off;
    const uint32_t tO = tmem + C::kTmemO + t * 128 + lane_off;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;
    float l = 0.f;
    bool ok = true;
    // Key tiles before jm hold prefix keys only; the rest reach the tree.
    const int jm = min(max(P / kKeyTile - k0, 0), T);
    for (int j = 0; j < jm && ok; ++j)
      ok = softmax_tile<false, false, D>(&s_full[t], static_cast<uint32_t>(j) & 1u, abort, &p_full[t], tS, tO,
                                  mrow, valid, W, (k0 + j) * kKeyTile, P, L, sl2, j > 0, nullptr,
                                  false, m_run, l, wlim);
    if (P < kSplitPrefix) {
      for (int j = jm; j < T && ok; ++j)
        ok = softmax_tile<true, true, D>(&s_full[t], static_cast<uint32_t>(j) & 1u, abort, &p_full[t], tS,
                                         tO, mrow, valid, W, (k0 + j) * kKeyTile, P, L, sl2, j > 0,
                                         nullptr, false, m_run, l, wlim);
    } else {
      for (int j = jm; j < T && ok; ++j)
        ok = softmax_tile<true, false, D>(&s_full[t], static_cast<uint32_t>(j) & 1u, abort, &p_full[t],
                                          tS, tO, mrow, valid, W, (k0 + j) * kKeyTile, P, L, sl2, j > 0,
                                          nullptr, false, m_run, l, wlim);
    }
    // Every thread of the warpgroup reaches this vote (all waits are bounded), so the
    // epilogue's own barriers are entered by all of them or by none.
    const bool done = named_bar_and(1 + t, 128, ok && wait_warp(&o_full, 0, abort, wlim));
    if (p.cluster_merge) {
      // Normalised fp32 row and its LSE stay in this CTA's shared memory for the merge.
      float lse2 = -INFINITY;
      if (done) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        lse2 = l > 0.f ? m_run + __log2f(l) : -INFINITY;
        uint8_t* dstrow = reinterpret_cast<uint8_t*>(part_row<NT, D>(sm, t, rl));
        const uint32_t sw = static_cast<uint32_t>(rl & 7);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint32_t k = static_cast<uint32_t>(c * 8 + v);
            *reinterpret_cast<float4*>(dstrow + ((k ^ sw) << 4)) =
                make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                            __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
          }
        }
      } else {
        set_abort(abort, p.dev_err);
      }
      part_lse<NT, D>(sm, t)[rl] = lse2;
    } else if (done) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_run + __log2f(l) : -INFINITY;
      // Every MMA has completed, so the K/V ring is free: stage this tile's output rows
      // there in the 128-byte-swizzled layout of the TMA box (16-byte chunk k of row r at
      // chunk k ^ (r % 8)), then one thread stores the tile with TMA.
      const int tile_row0 = (mp * NT + t) * kRowTile;
      const uint32_t sw = static_cast<uint32_t>(rl & 7);
      // A packed call's tile that reaches past the sequence's last node is stored row by
      // row (a TMA box would overwrite the next sequence's rows).
      const bool row_store = p.cu != nullptr && node_base + kRowTile / p.G > nt;
      if (p.splits == 1 && row_store) {
        uint16_t* orow = p.out + out_row(sp.row0, valid ? i : 0, p.Hq, h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);                 // every lane: the load is warp-wide
          tmem_ld_wait(o);
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + c * 32 + v * 8) = w;
            }
          }
        }
      } else if (p.splits == 1) {
        uint8_t* stg = sm + C::kKOff + t * C::kTileBytes;          // [half][128 rows][128 B]
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
          uint8_t* half = stg + (c >> 1) * C::kHalfBytes + rl * 128;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            const uint32_t k = static_cast<uint32_t>((c & 1) * 4 + v);
            *reinterpret_cast<uint4*>(half + ((k ^ sw) << 4)) = w;
          }
        }
        fence_proxy_async_smem();
        named_bar(1 + t, 128);
        if (rl == 0) {
          for (int hh = 0; hh < C::kHalves; ++hh)
            tma_store_4d(&omap, stg + hh * C::kHalfBytes, hh * 64, g * p.G,
                         p.cu != nullptr ? static_cast<int>(sp.row0) + node_base : node_base,
                         p.cu != nullptr ? 0 : b);
          bulk_commit();
          bulk_wait_read_all();
        }
      } else {
        uint8_t* stg = sm + C::kKOff + t * 2 * C::kTileBytes;      // [32-col block][128 rows][128 B]
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
          uint8_t* blk = stg + c * C::kHalfBytes + rl * 128;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(blk + ((static_cast<uint32_t>(v) ^ sw) << 4)) =
                make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                            __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
        fence_proxy_async_smem();
        named_bar(1 + t, 128);
        if (rl == 0) {
          const int plane = (b * p.Hkv + g) * p.splits + split;
          for (int c = 0; c < D / 32; ++c)
            tma_store_3d(&wmap, stg + c * C::kHalfBytes, c * 32, tile_row0, plane);
          bulk_commit();
          bulk_wait_read_all();
        }
      }
      if (valid) {
        if (p.splits == 1) {
          if (p.lse != nullptr)
            p.lse[lse_index(p.cu != nullptr, sp.row0, p.T, b, h, i, p.Hq, p.N)] =
                lse2 * 0.69314718055994531f;
        } else {
          p.ws_lse[((static_cast<size_t>(b) * p.Hkv + g) * p.splits + split) * p.M + r] = lse2;
        }
      }
    } else {
      set_abort(abort, p.dev_err);
    }
  }

  if (p.cluster_merge) merge_cluster<NT, D>(sm, MergeArgs{p.out, p.lse, p.N, p.Hq, p.G, p.M, p.splits, sp.row0, p.T, sp.rows, p.cu != nullptr}, b, g, mp, split);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
  grid_dependents_launch();
}

// ============================================================ stream-K variant
// With more (sequence, kv-head, row-tile group) units than SMs, one unit (or split) per
// CTA leaves the last wave partly idle and makes every CTA pay its own prologue and
// epilogue.  The stream-K variant runs one CTA per SM instead.  The key tiles of all
// (sequence, kv-head) pairs are laid end to end (sequence-major; pair (b, g) has
// tiles(b) = ceil((P_b + N) / 128)) and cut into nvirt equal ranges; the n_groups CTAs of
// range v (one per row-tile group) walk the same range, so the row-tile groups of a
// kv-head keep reading each K/V tile at about the same time.  A range is a run of
// segments, each a key-tile range of one pair: a whole pair is written straight to `out`;
// a range's first and last segments may be pieces of a pair, which go to the range's
// partial slots 0 and 1 and are merged by tree_attention_sk_combine_kernel.
//
// The roles are those of tree_attention_kernel with every counter running over the
// range's tiles as one sequence jg = 0 .. Wc-1, and the MMA issuer runs exactly that
// kernel's loop: it knows nothing of segments.  Step jg issues PV of tile jg and S of
// tile jg + 1 even when that tile opens the next segment, so the segment logic sits in the
// other roles: the producer reloads Q once step record e - 1 (S of the segment's last tile
// e - 1 done) completes; the voucher of the last tile waits for that Q and for the tail;
// the softmax warpgroups learn that the segment's last PV is done from the S barrier of
// tile e (committed after it), write the segment's rows, and zero O in tensor memory
// before they release the next segment's first tile, whose PV then accumulates onto zero.
struct SkSched {
  const int* pre;      // pre[b] = tiles of sequences < b (shared memory), pre[B] = S
  int B;
  int S;               // tiles of one kv head over all sequences
  int q, rem;          // W = Hkv * S tiles cut into nvirt ranges: rem of q + 1 tiles, then q
  __device__ SkSched(const int* pre_, int B_, int Hkv, int nvirt) : pre(pre_), B(B_), S(pre_[B_]) {
    const int W = Hkv * S;
    q = W / nvirt;
    rem = W - q * nvirt;
  }
  __device__ int tiles(int b) const { return pre[b + 1] - pre[b]; }
  __device__ int start(int b, int g) const { return g * S + pre[b]; }
  __device__ int range_lo(int v) const { return v * q + min(v, rem); }
  // the range containing x
  __device__ int range_of(int x) const {
    const int big = rem * (q + 1);
    return x < big ? x / (q + 1) : rem + (x - big) / q;
  }
};

// pre[0] = 0, pre[b + 1] = key tiles of sequences 0..b (prefix lengths clamped to the
// pool, tree sizes to [1, N], the clamps reported through `err` when given).  Every thread of the block calls it;
// B <= kLptMaxB <= blockDim.x.  Each warp scans 32 sequences with shuffles, then adds the
// totals of the warps before it.
__device__ __noinline__ void sk_tile_prefix(int* pre, const int32_t* prefix_len,
                                            const int32_t* tree_len, int B, int N, int cap,
                                            int* err) {
  const int u = threadIdx.x, lane = u & 31;
  int x = 0;
  if (u < B) {
    const int n = tree_nodes(tree_len, u, N);
    if (tree_len != nullptr && n != tree_len[u] && err != nullptr) report(err, JF_DEVERR_BAD_TREE_LEN);
    int P = prefix_len[u];
    if (P < 0 || P > cap - n) {
      if (err != nullptr) report(err, JF_DEVERR_BAD_PREFIX);
      P = max(0, min(P, cap - n));
    }
    x = (P + n + kKeyTile - 1) / kKeyTile;
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (u < B) pre[u + 1] = x;
  if (u == 0) pre[0] = 0;
  __syncthreads();
  int add = 0;
  if (u < B)
    for (int w = 0; w < (u >> 5); ++w) add += pre[min(32 * w + 32, B)];
  __syncthreads();
  if (u < B) pre[u + 1] = x + add;
  __syncthreads();
}

struct SkSeg {
  int b, g, k0, k1, slot;   // slot -1: whole pair; 0 / 1: the range's first / last partial
  int x1;                   // end of the segment in the global order
};

// The segment of range [lo, hi) that starts at global position x (32-bit positions keep
// the roles' register budgets free of 64-bit division).
__device__ __forceinline__ SkSeg sk_segment(const SkSched& s, int x, int lo, int hi) {
  SkSeg r;
  r.g = x / s.S;
  const int off = x - r.g * s.S;
  int a = 0, c = s.B;
  while (c - a > 1) {
    const int mid = (a + c) >> 1;
    if (s.pre[mid] <= off) a = mid; else c = mid;
  }
  r.b = a;
  r.k0 = off - s.pre[a];
  r.x1 = min(hi, s.start(r.b, r.g) + s.tiles(r.b));
  r.k1 = r.k0 + (r.x1 - x);
  r.slot = (r.k0 == 0 && r.k1 == s.tiles(r.b)) ? -1 : (x == lo ? 0 : 1);
  return r;
}
// The producer may finish several short segments before a voucher looks at the first, so
// "segment s's V tail is ready" is a count (release on the producer side, acquire here)
// rather than a phase of a reused barrier.
__device__ __forceinline__ void count_release_add(int* c) {
  asm volatile("red.release.cta.shared::cta.add.s32 [%0], 1;" ::"r"(smem_u32(c)) : "memory");
}
__device__ __forceinline__ int count_acquire(int* c) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(c)) : "memory");
  return v;
}
__device__ __forceinline__ bool wait_count_above(int* c, int target, volatile int* abort,
                                                 uint64_t wlim) {
  if (count_acquire(c) > target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (count_acquire(c) > target) return true;
    if ((it & 255u) == 0u && (*abort || global_timer_ns() - t0 > wlim)) return false;
  }
}

template <int NT, int D>
__global__ void __launch_bounds__(Cfg<NT, D>::kThreads, 1)
    tree_attention_sk_kernel(const __grid_constant__ CUtensorMap qmap,
                             const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap,
                             const __grid_constant__ CUtensorMap kmap_run,
                             const __grid_constant__ CUtensorMap vmap_run, const AttnParams p,
                             int nvirt) {
  using C = Cfg<NT, D>;
  constexpr int SK = C::kKStages;
  constexpr int SV = C::kVStages;
  constexpr int R = NT * kRowTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t q_full, o_full, fin;
  __shared__ uint64_t k_full[SK], v_full[SV], step_done[kStepRing];
  __shared__ uint64_t s_full[NT], p_full[NT];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int s_tails;                    // segments whose V tail is ready
  __shared__ int s_lo[NT];                   // current key tile of row tile t holds tree keys
  __shared__ int s_pre[kLptMaxB + 1];
  volatile int* abort = &abort_flag;
  uint8_t* q_s = sm + C::kQOff;
  uint8_t* k_s = sm + C::kKOff;
  uint8_t* v_s = sm + C::kVOff;
  const int v = blockIdx.x / p.n_groups;
  const int mp = blockIdx.x % p.n_groups;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&o_full, 1);
    mbar_init(&fin, 1);
    for (int st = 0; st < SK; ++st) mbar_init(&k_full[st], 1);
    for (int st = 0; st < SV; ++st) mbar_init(&v_full[st], 1);
    for (int st = 0; st < kStepRing; ++st) mbar_init(&step_done[st], 1);
    for (int t = 0; t < NT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128 + 1);   // the softmax warpgroup + its data voucher
    }
    s_tails = 0;
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&kmap_run);
    tma_prefetch_desc(&vmap_run);
  }
  const uint64_t wlim = g_wait_limit_ns;
  grid_dependency_wait();

  // ---- the schedule: tiles per sequence, their running sums, this range's segments
  const int cap = p.max_pages * kPage;
  sk_tile_prefix(s_pre, p.prefix_len, p.tree_len, p.B, p.N, cap, blockIdx.x == 0 ? p.dev_err : nullptr);
  const SkSched sch(s_pre, p.B, p.Hkv, nvirt);
  const int lo = sch.range_lo(v), hi = sch.range_lo(v + 1);
  const int Wc = hi - lo;
  // Boundary v (this range's start) as the combine kernel needs it: the pair whose
  // pieces it merges there, if v is the first boundary inside that pair.  (With fewer
  // tiles than ranges the last ranges are empty and merge nothing.)
  if (mp == 0 && threadIdx.x == 0 && v > 0) {
    int4 d0 = make_int4(-1, 0, 0, 0), d1 = make_int4(0, 0, 0, 0);
    const SkSeg f = Wc > 0 ? sk_segment(sch, lo, lo, hi) : SkSeg{0, 0, 0, 0, 0, 0};
    if (Wc > 0 && f.k0 > 0) {
      const int sw = sch.start(f.b, f.g);
      const int va = sch.range_of(sw);
      if (va == v - 1) {
        d0 = make_int4(f.b, f.g, va, sch.range_of(sw + sch.tiles(f.b) - 1));
        d1.x = sch.range_lo(va) == sw ? 0 : 1;     // slot of the first piece
      }
    }
    reinterpret_cast<int4*>(p.ws_desc)[2 * v] = d0;
    reinterpret_cast<int4*>(p.ws_desc)[2 * v + 1] = d1;
  }
  if (Wc <= 0) return;
  // end (exclusive, in range tiles) of the segment that starts at range tile j
  auto seg_end = [&](int j) -> int { return sk_segment(sch, lo + j, lo, hi).x1 - lo; };

  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp < 4) {
  if constexpr (NT == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
  if (warp == 0) {
    // ================================================================ TMA producer
    constexpr int kLookahead = 4;
    int k_issued = 0, v_issued = 0, q_issued = 0, bad = 0;
    bool ok = true;
    auto issue = [&](uint8_t* ring, const CUtensorMap* map, const CUtensorMap* map_run,
                     uint64_t* full, int st, int page, int page0, int g, bool run) {
      if (run) {
        if (lane < C::kHalves)
          tma_load_3d(ring + st * C::kTileBytes + lane * C::kHalfBytes, map_run, full, lane * 64, g,
                      page0 * kPage);
      } else if (lane < kPagesPerTile * C::kHalves) {
        const int q = lane % kPagesPerTile, hh = lane / kPagesPerTile;
        tma_load_3d(ring + st * C::kTileBytes + hh * C::kHalfBytes + q * (kPage * 128), map, full,
                    hh * 64, g, page * kPage);
      }
    };
    int jg0 = 0;
    for (int s = 0; jg0 < Wc && ok; ++s) {
      const SkSeg sg = sk_segment(sch, lo + jg0, lo, hi);
      const int T = sg.k1 - sg.k0;
      const int nsg = tree_nodes(p.tree_len, sg.b, p.N);
      const int L = max(0, min(p.prefix_len[sg.b], cap - nsg)) + nsg;
      const int32_t* bt = p.block_table + static_cast<size_t>(sg.b) * p.max_pages;
      // this segment's Q, once the previous segment's S MMAs no longer read the buffer
      int okq = 1;
      if (lane == 0) {
        const int rq = jg0 - 1;   // S of the previous segment's last tile: step record rq
        if (s > 0 && !mbar_wait(&step_done[rq % kStepRing], static_cast<uint32_t>(rq / kStepRing) & 1u,
                                abort, wlim)) {
          okq = 0;
        } else {
          mbar_arrive_expect_tx(&q_full, NT * C::kTileBytes);
          for (int t = 0; t < NT; ++t) {
            const int node0 = ((mp * NT + t) * kRowTile) / p.G;
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_4d(q_s + t * C::kTileBytes + hh * C::kHalfBytes, &qmap, &q_full, hh * 64,
                          sg.g * p.G, node0, sg.b);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, okq, 0)) { ok = false; break; }
      q_issued = s + 1;
      auto load_pid = [&](int j) -> int {
        const int pl = (sg.k0 + j) * kPagesPerTile + lane;
        if (lane >= kPagesPerTile || j >= T || pl * kPage >= L) return p.num_pages;
        return __ldg(bt + pl);
      };
      int pid[kLookahead];
#pragma unroll
      for (int u = 0; u < kLookahead; ++u) pid[u] = load_pid(u);
      for (int j = 0; j < T; ++j) {
        const int jg = jg0 + j;
        int mine = pid[0];
        if (mine < 0 || mine > p.num_pages) { bad = 1; mine = p.num_pages; }
        else if (mine == p.num_pages && lane < kPagesPerTile &&
                 ((sg.k0 + j) * kPagesPerTile + lane) * kPage < L) bad = 1;
        const int page = __shfl_sync(0xffffffffu, mine, lane % kPagesPerTile);
        const int page0 = __shfl_sync(0xffffffffu, mine, 0);
        const bool run = __all_sync(0xffffffffu, page == page0 + lane % kPagesPerTile);
#pragma unroll
        for (int u = 0; u < kLookahead - 1; ++u) pid[u] = pid[u + 1];
        pid[kLookahead - 1] = load_pid(j + kLookahead);
        const int sk = jg % SK, sv = jg % SV;
        const int rec = jg - C::kStageLag;
        int okl = 1;
        if (lane == 0) {
          if (rec >= 0 && !mbar_wait(&step_done[rec % kStepRing],
                                     static_cast<uint32_t>(rec / kStepRing) & 1u, abort, wlim)) {
            okl = 0;
          } else {
            mbar_arrive_expect_tx(&k_full[sk], C::kTileBytes);
            mbar_arrive_expect_tx(&v_full[sv], C::kTileBytes);
          }
        }
        if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
        issue(k_s, &kmap, &kmap_run, &k_full[sk], sk, page, page0, sg.g, run);
        k_issued = jg + 1;
        issue(v_s, &vmap, &vmap_run, &v_full[sv], sv, page, page0, sg.g, run);
        v_issued = jg + 1;
      }
      if (!ok) break;
      // V rows past the sequence end in the segment's last tile meet a zero probability:
      // make them zero, then release the tile to the MMA issuer's voucher (every segment).
      const int jl = jg0 + T - 1;
      if ((sg.k1) * kKeyTile > L) {
        if (!wait_warp(&v_full[jl % SV], static_cast<uint32_t>(jl / SV) & 1u, abort, wlim)) { ok = false; break; }
        const int r0 = L - (sg.k1 - 1) * kKeyTile;
        uint8_t* vt = v_s + (jl % SV) * C::kTileBytes;
        const int per_half = (kKeyTile - r0) * 8;
        for (int c = lane; c < per_half * C::kHalves; c += 32) {
          const int hh = c / per_half, rem = c % per_half;
          *reinterpret_cast<uint4*>(vt + hh * C::kHalfBytes + (r0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) count_release_add(&s_tails);
      jg0 += T;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.dev_err, JF_DEVERR_BAD_PAGE);
    if (!ok && lane == 0) set_abort(abort, p.dev_err);
    __syncwarp();
    if (lane == 0) {                   // no copy may still be landing when the CTA exits
      int zero = 0;
      if (q_issued > 0) mbar_wait(&q_full, static_cast<uint32_t>(q_issued - 1) & 1u, &zero);
      for (int j = max(0, k_issued - SK); j < k_issued; ++j)
        mbar_wait(&k_full[j % SK], static_cast<uint32_t>(j / SK) & 1u, &zero);
      for (int j = max(0, v_issued - SV); j < v_issued; ++j)
        mbar_wait(&v_full[j % SV], static_cast<uint32_t>(j / SV) & 1u, &zero);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t idS = idesc_bf16(kRowTile, kKeyTile, false, false);
    constexpr uint32_t idO = idesc_bf16(kRowTile, D, false, true);
    const uint64_t dq = desc_sw128(smem_u32(q_s), 16, 1024);
    const uint64_t dk = desc_sw128(smem_u32(k_s), 16, 1024);
    const uint64_t dv = desc_sw128(smem_u32(v_s), C::kHalfBytes, 1024);
    auto issue_s = [&](int t, int st) {
      const uint64_t da = dq + static_cast<uint64_t>((t * C::kTileBytes) >> 4);
      const uint64_t db = dk + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
      const uint32_t d_tmem = tmem + C::kTmemS + t * 128;
      mma_ss_tile<D / 16>(d_tmem, da, db, idS);
    };
    // O_t (+)= P_t V; with `lo`, also O_t += P_lo V from the second bf16 part of P (columns
    // 64..127 of the S region), issued before the next S MMA overwrites those columns.
    auto issue_pv = [&](int t, int st, bool acc, bool lo) {
      const uint64_t db = dv + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
      const uint32_t d_tmem = tmem + C::kTmemO + t * 128;
      const uint32_t a_tmem = tmem + C::kTmemS + t * 128;
      mma_ts_tile(d_tmem, a_tmem, db, idO, acc);
      if (lo) issue_pv_lo(d_tmem, a_tmem, db, idO);
    };
    bool ok = wait_warp(&q_full, 0, abort, wlim) && wait_warp(&k_full[0], 0, abort, wlim);
    if (ok) {
      // The whole warp runs this loop; the MMA and commit wrappers issue from one elected
      // lane (see tree_attention_kernel).
      tc_fence_after();
      for (int t = 0; t < NT; ++t) {
        issue_s(t, 0);
        mma_commit(&s_full[t]);
      }
      mma_commit(&step_done[0]);
      // The polling loop of tree_attention_kernel over the range's Wc tiles.
      int jn[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) jn[t] = 0;
      int left = NT * Wc;
      uint32_t idle = 0;
      uint64_t idle_since = 0;
      while (left > 0) {
        bool progressed = false;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int j = jn[t];
          if (j >= Wc) continue;
          if (__shfl_sync(0xffffffffu, mbar_try_wait(&p_full[t], static_cast<uint32_t>(j) & 1u) ? 1 : 0, 0) == 0)
            continue;
          bool last = true;
#pragma unroll
          for (int u = 0; u < NT; ++u)
            if (u != t && jn[u] <= j) last = false;
          tc_fence_after();
          // s_lo[t] was written before the softmax's arrival on p_full[t]: lane 0 reads it
          const bool lo = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&s_lo[t]), 0) != 0;
          issue_pv(t, j % SV, j > 0, lo);
          if (j + 1 < Wc) {
            issue_s(t, (j + 1) % SK);
            mma_commit(&s_full[t]);
          }
          if (last) mma_commit(&step_done[(j + 1) % kStepRing]);
          jn[t] = j + 1;
          --left;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else {
          if (idle == 0) idle_since = global_timer_ns();
          if ((++idle & 255u) == 0u &&
              __shfl_sync(0xffffffffu, (*abort || global_timer_ns() - idle_since > wlim) ? 1 : 0, 0) != 0) {
            ok = false;
            break;
          }
        }
      }
    }
    if (!ok && lane == 0) set_abort(abort, p.dev_err);
    if (ok) mma_commit(&o_full);   // the range's last PV
    mma_commit(&fin);   // all MMAs done before TMEM is released
    {
      int zero = 0;
      wait_warp(&fin, 0, &zero, kWaitLimitNs);
    }
  } else if (warp >= 2 && warp < 2 + NT) {
    // ================================================================ data vouchers
    // As in tree_attention_kernel, plus: at a segment's last tile the V tail of that
    // segment, and, when another segment follows, that segment's Q (its first S MMAs are
    // issued in this tile's step).
    const int t = warp - 2;
    if (lane == 0 && g_withhold_vouchers == 0) {
      int s = 0, e = seg_end(0);
      for (int j = 0; j < Wc; ++j) {
        const bool last_of_seg = j + 1 == e;
        const bool ready =
            (j == 0 || mbar_wait(&p_full[t], static_cast<uint32_t>(j - 1) & 1u, abort, wlim)) &&
            mbar_wait(&v_full[j % SV], static_cast<uint32_t>(j / SV) & 1u, abort, wlim) &&
            (j + 1 >= Wc ||
             mbar_wait(&k_full[(j + 1) % SK], static_cast<uint32_t>((j + 1) / SK) & 1u, abort, wlim)) &&
            (!last_of_seg || wait_count_above(&s_tails, s, abort, wlim)) &&
            (!last_of_seg || j + 1 >= Wc ||
             mbar_wait(&q_full, static_cast<uint32_t>(s + 1) & 1u, abort, wlim));
        if (!ready) {
          set_abort(abort, p.dev_err);
          break;
        }
        mbar_arrive(&p_full[t]);
        if (last_of_seg) {
          ++s;
          if (j + 1 < Wc) e = seg_end(j + 1);
        }
      }
    }
    __syncwarp();
  }
  } else {
    if constexpr (NT == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
    // ================================================================ softmax / epilogue
    const int t = (warp >> 2) - 1;
    const int wq = warp & 3;
    const int rl = wq * 32 + lane;                       // row within the tile = TMEM lane
    const int r = (mp * NT + t) * kRowTile + rl;
    const bool valid = r < p.M;
    const int i = r / p.G;
    const int W = p.W;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + C::kTmemS + t * 128 + lane_off;
    const uint32_t tO = tmem + C::kTmemO + t * 128 + lane_off;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int jg0 = 0;
    for (int s = 0; jg0 < Wc && ok; ++s) {
      const SkSeg sgm = sk_segment(sch, lo + jg0, lo, hi);
      const int T = sgm.k1 - sgm.k0;
      const int b = sgm.b, g = sgm.g;
      const int nsg = tree_nodes(p.tree_len, b, p.N);
      const int P = max(0, min(p.prefix_len[b], cap - nsg)), L = P + nsg;
      const int h = g * p.G + (r % p.G);
      const uint64_t* mrow = p.mask + (static_cast<size_t>(b) * p.N + (valid ? i : 0)) * W;
      float m_run = -INFINITY;
      float l = 0.f;
      // Key tiles before jm hold prefix keys only; the rest reach the tree.
      const int jm = min(max(P / kKeyTile - sgm.k0, 0), T);
      volatile int* lo_flag = &s_lo[t];
      for (int j = 0; j < jm && ok; ++j)
        ok = softmax_tile<false, false, D>(&s_full[t], static_cast<uint32_t>(jg0 + j) & 1u, abort, &p_full[t],
                                    tS, tO, mrow, valid, W, (sgm.k0 + j) * kKeyTile, P, L, sl2, j > 0,
                                    lo_flag, rl == 0, m_run, l, wlim);
      if (P < kSplitPrefix) {
        for (int j = jm; j < T && ok; ++j)
          ok = softmax_tile<true, true, D>(&s_full[t], static_cast<uint32_t>(jg0 + j) & 1u, abort,
                                           &p_full[t], tS, tO, mrow, valid, W, (sgm.k0 + j) * kKeyTile, P,
                                           L, sl2, j > 0, lo_flag, rl == 0, m_run, l, wlim);
      } else {
        for (int j = jm; j < T && ok; ++j)
          ok = softmax_tile<true, false, D>(&s_full[t], static_cast<uint32_t>(jg0 + j) & 1u, abort,
                                            &p_full[t], tS, tO, mrow, valid, W, (sgm.k0 + j) * kKeyTile, P,
                                            L, sl2, j > 0, lo_flag, rl == 0, m_run, l, wlim);
      }
      // A failed wait still reaches the warpgroup vote below (every warp must enter it).
      if (!ok && lane == 0) set_abort(abort, p.dev_err);
      // ---- the segment's rows: O / l, straight from TMEM to global memory, once its last
      // PV is done: S of the next tile (committed after it) or, for the range's last
      // segment, o_full.  Every warp of the warpgroup reaches this vote (all waits are
      // bounded), so it is all-or-none.
      const int je = jg0 + T;
      const bool pv_done = ok && (je < Wc ? wait_warp(&s_full[t], static_cast<uint32_t>(je) & 1u, abort, wlim)
                                          : wait_warp(&o_full, 0u, abort, wlim));
      if (!named_bar_and(1 + t, 128, pv_done)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_run + __log2f(l) : -INFINITY;
      const size_t prow = (static_cast<size_t>(v * 2 + max(sgm.slot, 0)) * p.n_groups + mp) * R +
                          t * kRowTile + rl;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        if (!valid) continue;
        if (sgm.slot < 0) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + ((static_cast<size_t>(b) * p.N + i) * p.Hq + h) * D + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
            dst[q] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + prow * D + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                                 __uint_as_float(o[4 * q + 2]) * inv, __uint_as_float(o[4 * q + 3]) * inv);
        }
      }
      if (valid) {
        if (sgm.slot < 0) {
          if (p.lse != nullptr)
            p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.N + i] = lse2 * 0.69314718055994531f;
        } else {
          p.ws_lse[prow] = lse2;
        }
      }
      if (je < Wc) {                   // the next segment's first PV accumulates onto zero
        uint32_t z[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) z[e] = 0u;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_st32(tO + c * 32, z);
      }
      jg0 += T;
    }
    if (!ok) set_abort(abort, p.dev_err);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
  grid_dependents_launch();
}

// Merges the stream-K partials.  A (sequence, kv-head) pair cut by range boundaries left
// one partial per range it touches (slot 0 where the range starts inside or at the pair,
// slot 1 where the range ends in it); the pair is merged at its first inner boundary,
// which the split kernel described in `desc` (b, g, first range, last range; slot of the
// first piece).  Block (v * n_groups + mp, y): boundary v, row-tile group mp, four rows
// of the group per warp; blocks of boundaries that merge nothing exit at once.  A split
// pair has at least two pieces: the first two of all four rows are fetched together, so
// a warp waits about one memory round trip for the common case.
template <int D>
__global__ void __launch_bounds__(256, 4)
    tree_attention_sk_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                                     const int4* __restrict__ desc, int N, int Hq, int Hkv,
                                     int n_groups, int R, uint16_t* __restrict__ out,
                                     float* __restrict__ lse) {
  constexpr int E = D / 32;
  constexpr int kRows = 4;
  using VecE = typename std::conditional<E == 4, float4, float2>::type;
  grid_dependency_wait();
  const int v = blockIdx.x / n_groups, mp = blockIdx.x % n_groups;
  if (v == 0) return;
  const int4 d0 = desc[2 * v];
  if (d0.x < 0) return;
  const int slot_a = desc[2 * v + 1].x;
  const int b = d0.x, g = d0.y, va = d0.z, n = d0.w - d0.z + 1;
  const int G = Hq / Hkv, M = N * G;
  const int lane = threadIdx.x & 31;
  const int rw0 = blockIdx.y * (8 * kRows) + (threadIdx.x >> 5) * kRows;
  auto prow = [&](int rw, int k) -> long long {    // partial row of piece k (range va + k)
    return (static_cast<long long>((va + k) * 2 + (k == 0 ? slot_a : 0)) * n_groups + mp) * R + rw;
  };
  auto ld = [&](int rw, int k) -> VecE {
    return *reinterpret_cast<const VecE*>(ws_o + prow(rw, k) * D + lane * E);
  };
  float lk[kRows];
  VecE x0[kRows], x1[kRows];
#pragma unroll
  for (int q = 0; q < kRows; ++q) {
    const int rw = rw0 + q;
    const bool ok = rw < R && mp * R + rw < M;
    lk[q] = (ok && lane < n) ? ws_lse[prow(rw, lane)] : -INFINITY;
    if (ok) { x0[q] = ld(rw, 0); x1[q] = ld(rw, 1); }
  }
#pragma unroll
  for (int q = 0; q < kRows; ++q) {
    const int rw = rw0 + q;
    const int r = mp * R + rw;
    if (rw >= R || r >= M) break;
    float mx = lk[q];
    for (int k = 32 + lane; k < n; k += 32) mx = fmaxf(mx, ws_lse[prow(rw, k)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[E];
    float wsum = 0.f;
    {
      const float wk = (lk[q] == -INFINITY) ? 0.f : exp2f(lk[q] - mx);
      const float w0 = __shfl_sync(0xffffffffu, wk, 0), w1 = __shfl_sync(0xffffffffu, wk, 1);
      const float* a0 = reinterpret_cast<const float*>(&x0[q]);
      const float* a1 = reinterpret_cast<const float*>(&x1[q]);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = w0 * a0[e] + w1 * a1[e];
      wsum = w0 + w1;
      for (int k = 2; k < n; ++k) {                // pairs spread over more than two ranges
        const float lv = (k < 32) ? lk[q] : ws_lse[prow(rw, k)];
        const float wl = (lv == -INFINITY) ? 0.f : exp2f(lv - mx);
        const float w = k < 32 ? __shfl_sync(0xffffffffu, wl, k) : wl;
        const VecE x = ld(rw, k);
        const float* xs = reinterpret_cast<const float*>(&x);
        wsum += w;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * xs[e];
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int i = r / G, h = g * G + (r % G);
    uint16_t* dst = out + ((static_cast<long long>(b) * N + i) * Hq + h) * D + lane * E;
    uint32_t packed[E / 2];
#pragma unroll
    for (int e = 0; e < E; e += 2) packed[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    if constexpr (E == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    }
    if (lse != nullptr && lane == 0)
      lse[(static_cast<long long>(b) * Hq + h) * N + i] =
          (wsum > 0.f ? mx + __log2f(wsum) : -INFINITY) * 0.69314718055994531f;
  }
}

// Merges split partials: O = sum_s 2^(lse_s - lse) O_s,  lse = log2 sum_s 2^lse_s.
// One warp per output row, rows enumerated in the output's [B][N][Hq] order so that
// consecutive warps write consecutive rows; each lane owns D/32 consecutive columns.
// Splits are taken kBatch at a time: lane q fetches split q's LSE while every lane fetches
// its columns of all kBatch partial rows, so a batch costs one memory round trip.  The
// host picks the smallest batch that covers the splits: wider batches hold more partial
// rows in registers and leave fewer warps per SM for the bandwidth-bound many-row case.
template <int D, int kBatch>
__global__ void __launch_bounds__(256)
    tree_attention_combine_kernel(const float* __restrict__ ws_o,
                                  const float* __restrict__ ws_lse, int splits, int N, int Hq,
                                  int Hkv, long long rows, uint16_t* __restrict__ out,
                                  float* __restrict__ lse, const int32_t* __restrict__ cu,
                                  long long T) {
  constexpr int E = D / 32;
  static_assert(kBatch >= 1 && kBatch <= 16 && (kBatch & (kBatch - 1)) == 0, "batch of splits");
  using VecE = typename std::conditional<E == 4, float4, float2>::type;
  // Launched as a programmatic dependent of the split kernel: wait for its results.
  grid_dependency_wait();
  const long long rr = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rr >= rows) return;
  const int h = static_cast<int>(rr % Hq);
  const long long bi = rr / Hq;
  const int i = static_cast<int>(bi % N);
  const long long b = bi / N;
  const int G = Hq / Hkv;
  const int g = h / G;
  const long long M = static_cast<long long>(N) * G;
  const long long r = static_cast<long long>(i) * G + (h % G);
  const long long base = (b * Hkv + g) * splits;       // partial row of split s: (base + s) * M + r
  // Packed calls: rows of nodes past the sequence's last one do not exist in out and lse.
  long long row0 = b * N;
  if (cu != nullptr) {
    const SeqSpan sp = seq_span(cu, nullptr, static_cast<int>(b), N, T);
    if (i >= sp.rows) return;
    row0 = sp.row0;
  }
  // With more than one batch the running maximum must be known first.
  float mx = -INFINITY;
  if (splits > kBatch) {
    for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, ws_lse[(base + s) * M + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int s0 = 0; s0 < splits; s0 += kBatch) {
    const int sq = s0 + (lane % kBatch);
    const float lq = sq < splits ? ws_lse[(base + sq) * M + r] : -INFINITY;
    VecE v[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
      if (s0 + q < splits)
        v[q] = *reinterpret_cast<const VecE*>(ws_o + ((base + s0 + q) * M + r) * D + lane * E);
    if (splits <= kBatch) {
      mx = lq;
#pragma unroll
      for (int o = kBatch / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float wq = (lq == -INFINITY) ? 0.f : exp2f(lq - mx);
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const float w = __shfl_sync(0xffffffffu, wq, q);
      if (s0 + q < splits) {
        wsum += w;
        const float* vf = reinterpret_cast<const float*>(&v[q]);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * vf[e];
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* dst = out + out_row(row0, i, Hq, h) * D + lane * E;
  uint32_t packed[E / 2];
#pragma unroll
  for (int e = 0; e < E; e += 2) packed[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  }
  if (lse != nullptr && lane == 0)
    lse[lse_index(cu != nullptr, row0, T, static_cast<int>(b), h, i, Hq, N)] =
        (wsum > 0.f ? mx + __log2f(wsum) : -INFINITY) * 0.69314718055994531f;
}

// ------------------------------------------------------------------------ host side

struct AttnPlan {
  int NT, n_groups, splits, chunk_tiles;
  bool cluster;          // splits merged through distributed shared memory (no workspace)
  bool streamk;          // one CTA per SM over equal ranges of all key tiles (stream-K)
  int nvirt;             // stream-K: ranges (each walked by n_groups CTAs)
  size_t ws_bytes;
};

template <int NT, int D, bool LPT>
bool ensure_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(tree_attention_kernel<NT, D, LPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<NT, D>::kSmemBytes) != cudaSuccess)
    return false;
  if (dev < 64) done[dev] = true;
  return true;
}

template <int NT, int D>
bool ensure_smem_attr_sk() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(tree_attention_sk_kernel<NT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<NT, D>::kSmemBytes) != cudaSuccess)
    return false;
  if (dev < 64) done[dev] = true;
  return true;
}

template <int D>
jf_status launch_sk(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                    const CUtensorMap& kr, const CUtensorMap& vr, const AttnParams& prm, int nvirt,
                    long long rows, uint16_t* out, float* lse, cudaStream_t s) {
  using C = Cfg<2, D>;
  if (!ensure_smem_attr_sk<2, D>()) return JF_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(nvirt * prm.n_groups));
  lc.blockDim = dim3(C::kThreads);
  lc.dynamicSmemBytes = C::kSmemBytes;
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, tree_attention_sk_kernel<2, D>, qm, km, vm, kr, vr, prm, nvirt) != cudaSuccess)
    return JF_ERR_CUDA;
  cudaLaunchConfig_t lc2 = {};
  lc2.gridDim = dim3(static_cast<unsigned>(nvirt * prm.n_groups), static_cast<unsigned>(2 * kRowTile / 32));
  lc2.blockDim = dim3(256);
  lc2.stream = s;
  lc2.attrs = attr;
  lc2.numAttrs = 1;
  const float* wso = prm.ws_o;
  const float* wsl = prm.ws_lse;
  const int4* dsc = reinterpret_cast<const int4*>(prm.ws_desc);
  const int R = 2 * kRowTile;
  return cudaLaunchKernelEx(&lc2, tree_attention_sk_combine_kernel<D>, wso, wsl, dsc, prm.N, prm.Hq,
                            prm.Hkv, prm.n_groups, R, out, lse) == cudaSuccess
             ? JF_OK
             : JF_ERR_CUDA;
}

// How many clusters of `s` CTAs of this kernel fit on the current device at once
// (0 if that cluster shape cannot be launched).  Cached per device.
template <int NT, int D>
int cluster_capacity(int s) {
  static std::mutex mu;
  static int cache[64][9];
  static bool init = false;
  int dev = 0;
  if (s < 2 || s > 8 || cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& row : cache)
      for (int& v : row) v = -1;
    init = true;
  }
  if (cache[dev][s] >= 0) return cache[dev][s];
  int n = 0;
  if (ensure_smem_attr<NT, D, false>()) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s) * 64);
    cfg.blockDim = dim3(Cfg<NT, D>::kThreads);
    cfg.dynamicSmemBytes = Cfg<NT, D>::kSmemBytes;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = static_cast<unsigned>(s);
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, tree_attention_kernel<NT, D, false>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  cache[dev][s] = n;
  return n;
}

int cluster_capacity_for(int NT, int D, int s) {
  if (D == 128) return NT == 2 ? cluster_capacity<2, 128>(s) : cluster_capacity<1, 128>(s);
  return NT == 2 ? cluster_capacity<2, 64>(s) : cluster_capacity<1, 64>(s);
}

bool shape_supported(int B, int N, int Hq, int Hkv, int D, int max_pages, int page_size) {
  if (B < 1 || N < 1 || N > JF_MAX_NODES || Hq < 1 || Hkv < 1 || max_pages < 1) return false;
  if (D != 64 && D != 128) return false;
  if (page_size != kPage) return false;
  if (Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  if (G > kRowTile || (G & (G - 1)) != 0) return false;
  if (static_cast<long long>(max_pages) * kPage < N) return false;
  if (static_cast<long long>(max_pages) * kPage > (1ll << 30)) return false;
  return true;
}

// allow_streamk = false for ragged calls: stream-K ranges are walked by every row-tile
// group of a (sequence, kv-head) pair together, so padding groups could not skip their work.
bool plan_attention(int B, int N, int Hq, int Hkv, int D, int max_pages, int sms, AttnPlan* pl,
                    bool allow_streamk = true) {
  const int G = Hq / Hkv;
  const long long M = static_cast<long long>(N) * G;
  const int mtiles = static_cast<int>((M + kRowTile - 1) / kRowTile);
  pl->NT = mtiles >= 2 ? 2 : 1;
  pl->n_groups = (mtiles + pl->NT - 1) / pl->NT;
  const int max_tiles = (max_pages * kPage + kKeyTile - 1) / kKeyTile;
  const long long units = static_cast<long long>(B) * Hkv * pl->n_groups;
  if (sms <= 0) sms = 148;
  // Time model: waves * (tiles per split + prologue/epilogue) * max(tensor time of a key
  // tile, its share of HBM bandwidth), plus, for workspace splits, writing and re-reading
  // the partials (at L2 speed while they fit in a third of it) and one more launch.  Cluster splits (2..8 CTAs merging through DSMEM)
  // pay no merge traffic but pack fewer CTAs per wave.
  const double hbm_per_tile = 2.0 * kKeyTile * D * 2;          // K + V bytes per key tile
  const double flops_per_tile = 4.0 * kRowTile * kKeyTile * D;  // QK^T + PV per row tile
  const double per_sm_flops = 1.9e15 / sms, hbm = 6.5e12, l2bw = 20e12;
  auto t_tile = [&](double active) {
    return std::max(pl->NT * flops_per_tile / per_sm_flops, hbm_per_tile * active / hbm);
  };
  double best = 1e300;
  int best_s = 1;
  bool best_cluster = false;
  for (int s = 1; s <= max_tiles; ++s) {
    const int chunk = (max_tiles + s - 1) / s;
    if (s > 1 && (s - 1) * chunk >= max_tiles) continue;         // last split would be empty
    const long long ctas = units * s;
    const long long waves = (ctas + sms - 1) / sms;
    double est = waves * (chunk + 1.5) * t_tile(static_cast<double>(std::min<long long>(ctas, sms)));
    if (s > 1) {
      // the partials are written and read back once; up to a third of L2 they stay there
      const double part = static_cast<double>(B) * Hq * N * s * (D + 1) * 4.0;
      est += 1.5e-6 + 2.0 * part / (part <= 43e6 ? l2bw : hbm);
    }
    if (est < best * 0.98) { best = est; best_s = s; best_cluster = false; }
    // Clusters only when every cluster of the grid is resident at once: with several
    // waves, a finished cluster must wait for s SMs of one GPC to free up together.
    const int cap = (s >= 2 && s <= 8) ? cluster_capacity_for(pl->NT, D, s) : 0;
    if (cap > 0 && units <= cap) {
      const double est_c = (chunk + 1.5) * t_tile(static_cast<double>(units * s)) + 4e-6;
      if (est_c < best * 0.98) { best = est_c; best_s = s; best_cluster = true; }
    }
  }
  pl->splits = best_s;
  pl->cluster = best_cluster;
  pl->chunk_tiles = (max_tiles + best_s - 1) / best_s;
  pl->ws_bytes = (best_s > 1 && !best_cluster)
                     ? static_cast<size_t>(B) * Hq * N * best_s * (D + 1) * sizeof(float) + 256
                     : 0;
  pl->streamk = false;
  pl->nvirt = 0;
  // Stream-K (one CTA per SM over equal ranges of all key tiles) when one unit per CTA
  // leaves the last wave under 90% full and the work is tensor-bound: several row-tile
  // groups read each K/V tile.  On HBM-bound work (one group) the range walk measured
  // slower than the plain dispatch.  Positions in the range order are 32-bit.
  const long long waves1 = (units + sms - 1) / sms;
  const bool ragged_waves = units < waves1 * sms * 9 / 10;
  const long long max_tiles_all =
      static_cast<long long>(B) * Hkv * (static_cast<long long>(max_pages) * kPage / kKeyTile + 1);
  if (allow_streamk && pl->NT == 2 && pl->n_groups >= 2 && units >= sms && ragged_waves && B <= kLptMaxB &&
      pl->n_groups <= sms && max_tiles_all < (1ll << 30)) {
    pl->streamk = true;
    pl->nvirt = sms / pl->n_groups;
    pl->splits = 1;
    pl->cluster = false;
    pl->chunk_tiles = max_tiles;
    pl->ws_bytes = static_cast<size_t>(pl->nvirt) * 2 * pl->n_groups * pl->NT * kRowTile * (D + 1) *
                       sizeof(float) + static_cast<size_t>(pl->nvirt) * 8 * sizeof(int) + 256;
  }
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box,
            CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, rank, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, int D, bool LPT>
jf_status launch(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                 const CUtensorMap& kr, const CUtensorMap& vr, const CUtensorMap& om,
                 const CUtensorMap& wm, const AttnParams& prm, long long grid, cudaStream_t s) {
  using C = Cfg<NT, D>;
  if (!ensure_smem_attr<NT, D, LPT>()) return JF_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid));
  lc.blockDim = dim3(C::kThreads);
  lc.dynamicSmemBytes = C::kSmemBytes;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (prm.cluster_merge) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(prm.splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.numAttrs = 2;
  }
  const cudaError_t e =
      cudaLaunchKernelEx(&lc, tree_attention_kernel<NT, D, LPT>, qm, km, vm, kr, vr, om, wm, prm);
  return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
}

}  // namespace
}  // namespace jf

extern "C" size_t jf_tree_attention_workspace_size(int32_t B, int32_t N, int32_t Hq, int32_t Hkv,
                                                   int32_t D, int32_t max_pages,
                                                   int32_t page_size) {
  if (!jf::shape_supported(B, N, Hq, Hkv, D, max_pages, page_size)) return static_cast<size_t>(-1);
  const int sms = jf::current_sm_count();
  if (sms <= 0) return static_cast<size_t>(-1);
  jf::AttnPlan pl, pr;
  jf::plan_attention(B, N, Hq, Hkv, D, max_pages, sms, &pl);
  jf::plan_attention(B, N, Hq, Hkv, D, max_pages, sms, &pr, false);   // the ragged call's plan
  return std::max(pl.ws_bytes, pr.ws_bytes);
}

namespace {

// Packed calls pass cu (cumulative node counts, [B + 1]) and T = total nodes; N is then
// the largest tree the call may hold.  The others pass nullptr and 0.
jf_status tree_attention_call(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, const int32_t* prefix_len,
                              const int32_t* tree_len, const uint64_t* mask, int32_t B,
                              int32_t N, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                              int32_t max_pages, int32_t num_pages, float scale, void* out,
                              float* lse, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err, jf_stream_t stream, const int32_t* cu = nullptr,
                              int32_t T = 0) {
  using namespace jf;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      prefix_len == nullptr || mask == nullptr || out == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || D < 1 || page_size < 1 || max_pages < 1 ||
      num_pages < 1 || !(scale > 0.f) || !std::isfinite(scale))
    return JF_ERR_INVALID_ARGUMENT;
  if (!shape_supported(B, N, Hq, Hkv, D, max_pages, page_size)) return JF_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * kPage >= (1ll << 31)) return JF_ERR_UNSUPPORTED;
  if (cu != nullptr && T < 1) return JF_ERR_INVALID_ARGUMENT;
  if (cu != nullptr && static_cast<long long>(T) + N >= (1ll << 31)) return JF_ERR_UNSUPPORTED;
  if (!aligned_to(q, 16) || !aligned_to(k_cache, 16) || !aligned_to(v_cache, 16) ||
      !aligned_to(out, 16) || !aligned_to(mask, 8))
    return JF_ERR_MISALIGNED;
  const int sms = current_sm_count();
  if (sms <= 0) return JF_ERR_CUDA;
  AttnPlan pl;
  plan_attention(B, N, Hq, Hkv, D, max_pages, sms, &pl, tree_len == nullptr && cu == nullptr);
  if (pl.ws_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < pl.ws_bytes) return JF_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned_to(workspace, 16)) return JF_ERR_MISALIGNED;
  }
  const int G = Hq / Hkv;
  CUtensorMap qm, km, vm, kr, vr, om, wm;
  std::memset(&om, 0, sizeof(om));
  std::memset(&wm, 0, sizeof(wm));
  {
    // q and out share one layout: [B][N][Hq][D] ([1][T][Hq][D] packed), 128-row tiles of
    // (node, head-in-group).
    const cuuint64_t rows_n = cu != nullptr ? static_cast<cuuint64_t>(T) : static_cast<cuuint64_t>(N);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), rows_n,
                                cu != nullptr ? 1u : static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hq) * D * 2,
                                   rows_n * Hq * D * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kRowTile / G), 1};
    if (!encode(&qm, q, 4, dims, strides, box)) return JF_ERR_CUDA;
    if (pl.splits == 1 && !encode(&om, out, 4, dims, strides, box)) return JF_ERR_CUDA;
  }
  if (pl.splits > 1 && !pl.cluster) {
    // split partials O_s: fp32 [B * Hkv * splits][M][D], stored in 32-column boxes
    const long long M = static_cast<long long>(N) * G;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(M),
                                static_cast<cuuint64_t>(B) * Hkv * pl.splits};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                                   static_cast<cuuint64_t>(M) * D * 4};
    const cuuint32_t box[3] = {32, kRowTile, 1};
    if (!encode(&wm, workspace, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return JF_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(num_pages) * kPage};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hkv) * D * 2};
    const cuuint32_t box[3] = {64, 1, kPage};
    if (!encode(&km, k_cache, 3, dims, strides, box)) return JF_ERR_CUDA;
    if (!encode(&vm, v_cache, 3, dims, strides, box)) return JF_ERR_CUDA;
    const cuuint32_t box_run[3] = {64, 1, kKeyTile};   // eight consecutive pages at once
    if (!encode(&kr, k_cache, 3, dims, strides, box_run)) return JF_ERR_CUDA;
    if (!encode(&vr, v_cache, 3, dims, strides, box_run)) return JF_ERR_CUDA;
  }
  AttnParams prm;
  prm.block_table = block_table;
  prm.prefix_len = prefix_len;
  prm.tree_len = tree_len;
  prm.cu = cu;
  prm.T = cu != nullptr ? T : 0;
  prm.mask = mask;
  prm.out = static_cast<uint16_t*>(out);
  prm.lse = lse;
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  prm.ws_o = pl.ws_bytes > 0 ? static_cast<float*>(workspace) : nullptr;
  const size_t part_rows = pl.streamk
                               ? static_cast<size_t>(pl.nvirt) * 2 * pl.n_groups * pl.NT * kRowTile
                               : rows * pl.splits;
  prm.ws_lse = pl.ws_bytes > 0 ? static_cast<float*>(workspace) + part_rows * D : nullptr;
  prm.ws_desc = pl.streamk ? reinterpret_cast<int*>(prm.ws_lse + part_rows) : nullptr;
  prm.dev_err = dev_err;
  prm.B = B; prm.N = N; prm.Hq = Hq; prm.Hkv = Hkv; prm.G = G; prm.W = (N + 63) / 64;
  prm.max_pages = max_pages; prm.num_pages = num_pages;
  prm.n_groups = pl.n_groups; prm.splits = pl.splits; prm.chunk_tiles = pl.chunk_tiles;
  prm.M = N * G;
  prm.cluster_merge = pl.cluster ? 1 : 0;
  // Longest-first dispatch when every unit is one CTA and sequence lengths may differ.
  const bool lpt = pl.splits == 1 && B >= 2 && B <= jf::kLptMaxB;
  prm.scale_log2 = scale * 1.4426950408889634f;
  if (pl.streamk) {
    cudaStream_t s0 = reinterpret_cast<cudaStream_t>(stream);
    uint16_t* o16 = static_cast<uint16_t*>(out);
    const long long nrows = static_cast<long long>(rows);
    return D == 128 ? launch_sk<128>(qm, km, vm, kr, vr, prm, pl.nvirt, nrows, o16, lse, s0)
                    : launch_sk<64>(qm, km, vm, kr, vr, prm, pl.nvirt, nrows, o16, lse, s0);
  }
  const long long grid = static_cast<long long>(B) * Hkv * pl.splits * pl.n_groups;
  if (grid > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  jf_status st;
  if (D == 128)
    st = pl.NT == 2 ? (lpt ? launch<2, 128, true>(qm, km, vm, kr, vr, om, wm, prm, grid, s)
                           : launch<2, 128, false>(qm, km, vm, kr, vr, om, wm, prm, grid, s))
                    : (lpt ? launch<1, 128, true>(qm, km, vm, kr, vr, om, wm, prm, grid, s)
                           : launch<1, 128, false>(qm, km, vm, kr, vr, om, wm, prm, grid, s));
  else
    st = pl.NT == 2 ? (lpt ? launch<2, 64, true>(qm, km, vm, kr, vr, om, wm, prm, grid, s)
                           : launch<2, 64, false>(qm, km, vm, kr, vr, om, wm, prm, grid, s))
                    : (lpt ? launch<1, 64, true>(qm, km, vm, kr, vr, om, wm, prm, grid, s)
                           : launch<1, 64, false>(qm, km, vm, kr, vr, om, wm, prm, grid, s));
  if (st != JF_OK) return st;
  if (pl.splits > 1 && !pl.cluster) {
    const long long nb = (static_cast<long long>(rows) + 7) / 8;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(nb));
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const float* wso = prm.ws_o;
    const float* wsl = prm.ws_lse;
    const int nsp = pl.splits;
    const long long nrows = static_cast<long long>(rows);
    uint16_t* o16 = static_cast<uint16_t*>(out);
    auto pick = [&](auto kern4, auto kern8, auto kern16) {
      const long long Tl = prm.T;
      return nsp <= 4   ? cudaLaunchKernelEx(&lc, kern4, wso, wsl, nsp, N, Hq, Hkv, nrows, o16, lse, cu, Tl)
             : nsp <= 8 ? cudaLaunchKernelEx(&lc, kern8, wso, wsl, nsp, N, Hq, Hkv, nrows, o16, lse, cu, Tl)
                        : cudaLaunchKernelEx(&lc, kern16, wso, wsl, nsp, N, Hq, Hkv, nrows, o16, lse, cu, Tl);
    };
    const cudaError_t e =
        D == 128 ? pick(tree_attention_combine_kernel<128, 4>, tree_attention_combine_kernel<128, 8>,
                        tree_attention_combine_kernel<128, 16>)
                 : pick(tree_attention_combine_kernel<64, 4>, tree_attention_combine_kernel<64, 8>,
                        tree_attention_combine_kernel<64, 16>);
    return e == cudaSuccess ? JF_OK : JF_ERR_CUDA;
  }
  return JF_OK;
}

}  // namespace

extern "C" jf_status jf_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       const uint64_t* mask, int32_t B, int32_t N, int32_t Hq,
                                       int32_t Hkv, int32_t D, int32_t page_size,
                                       int32_t max_pages, int32_t num_pages, float scale,
                                       void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_err,
                                       jf_stream_t stream) {
  return tree_attention_call(q, k_cache, v_cache, block_table, prefix_len, nullptr, mask, B, N, Hq,
                             Hkv, D, page_size, max_pages, num_pages, scale, out, lse, workspace,
                             workspace_bytes, dev_err, stream);
}

extern "C" jf_status jf_tree_attention_ragged(const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_table,
                                              const int32_t* prefix_len, const int32_t* tree_len,
                                              const uint64_t* mask, int32_t B, int32_t N,
                                              int32_t Hq, int32_t Hkv, int32_t D,
                                              int32_t page_size, int32_t max_pages,
                                              int32_t num_pages, float scale, void* out,
                                              float* lse, void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, jf_stream_t stream) {
  if (tree_len == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return tree_attention_call(q, k_cache, v_cache, block_table, prefix_len, tree_len, mask, B, N,
                             Hq, Hkv, D, page_size, max_pages, num_pages, scale, out, lse,
                             workspace, workspace_bytes, dev_err, stream);
}

extern "C" jf_status jf_tree_attention_packed(const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_table,
                                              const int32_t* prefix_len, const int32_t* cu_seqlens,
                                              const uint64_t* mask, int32_t B, int32_t N_max,
                                              int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                              int32_t page_size, int32_t max_pages,
                                              int32_t num_pages, float scale, void* out,
                                              float* lse, void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, jf_stream_t stream) {
  if (cu_seqlens == nullptr) return JF_ERR_INVALID_ARGUMENT;
  return tree_attention_call(q, k_cache, v_cache, block_table, prefix_len, nullptr, mask, B, N_max,
                             Hq, Hkv, D, page_size, max_pages, num_pages, scale, out, lse,
                             workspace, workspace_bytes, dev_err, stream, cu_seqlens, T);
}

extern "C" jf_status jf_debug_set_wait_limit_ns(uint64_t limit_ns, int32_t withhold_arrivals) {
  const uint64_t v = limit_ns == 0 ? jf::kWaitLimitNs : limit_ns;
  const int w = withhold_arrivals != 0 ? 1 : 0;
  if (cudaMemcpyToSymbol(jf::g_wait_limit_ns, &v, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(jf::g_withhold_vouchers, &w, sizeof(w)) != cudaSuccess) {
    cudaGetLastError();
    return JF_ERR_CUDA;
  }
  return JF_OK;
}
