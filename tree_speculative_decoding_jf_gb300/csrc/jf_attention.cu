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
// Splits and CTA count are chosen on the host from the SM count; partial results of a
// split go to a workspace and a second kernel merges them by log-sum-exp.
//
// Roles inside a CTA (128 * (1 + NT) threads):
//   warp 0      TMA producer: stages the split's page ids from the block table in shared
//               memory (bounds-checked), loads the Q tiles once, then per key tile eight
//               16-key pages of K and of V (one TMA box each per 64-column half) into a
//               STAGES-deep ring.  Pages past the sequence end load as zeros.
//   warp 1      allocates TMEM and issues tcgen05.mma from one lane:
//                 S_t = Q_t K^T  (128 x 128, fp32 in TMEM),  O_t += P_t V  (P from TMEM).
//               It zeroes V rows past the sequence end in the last tile (garbage in unused
//               page slots must not meet a zero probability as NaN).
//   warps 4..   one warpgroup per row tile t: TMEM lane = row, so each thread owns one
//               full score row.  Ancestor bitmasks of the tile's nodes are staged in
//               shared memory and applied to keys at positions >= P_b.  Online softmax in
//               the log2 domain; the running max is only raised when a tile's max
//               exceeds it by more than 8 (factor 256), which keeps P <= 256 in bf16 and
//               makes the O rescale (TMEM load/scale/store) rare.  P (bf16) is written
//               back into the S columns and consumed by the PV MMA from TMEM.
// All waits are bounded (see jf_sm100.cuh); on a timeout the CTA records
// JF_DEVERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "jf_common.cuh"
#include "jf_sm100.cuh"

namespace jf {
namespace {

constexpr int kKeyTile = 128;     // keys per pipeline stage
constexpr int kRowTile = 128;     // rows per tensor-core tile (TMEM lanes)
constexpr int kPage = 16;
constexpr int kPagesPerTile = kKeyTile / kPage;
constexpr int kPageWindowTiles = 256;                   // page ids staged at a time
constexpr int kMaskBytesPerTile = 8192;                 // staged mask words per row tile
constexpr float kRescaleThreshold = 8.0f;               // log2 units

template <int NT, int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                  // 128-byte swizzle atoms per row
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kTileBytes = kRowTile * D * 2;     // one 128-row bf16 tile
  static constexpr int kHalfBytes = kRowTile * 128;       // one 64-column half of a tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NT * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kPageOff = kVOff + kStages * kTileBytes;
  static constexpr int kMaskOff = kPageOff + kPageWindowTiles * kPagesPerTile * 4;
  static constexpr int kSmemBytes = kMaskOff + NT * kMaskBytesPerTile + 1024;
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
  float* ws_o;          // [B][Hq][N][splits][D]   (splits > 1)
  float* ws_lse;        // [B][Hq][N][splits]      (log2 domain)
  int32_t* dev_err;
  int B, N, Hq, Hkv, G, W, max_pages, num_pages;
  int n_groups, splits, chunk_tiles, M;
  float scale_log2;     // softmax scale * log2(e)
};

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
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

template <int NT, int D>
__global__ void __launch_bounds__(Cfg<NT, D>::kThreads, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  using C = Cfg<NT, D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t q_full, o_full, fin;
  __shared__ uint64_t k_full[S], v_full[S], k_empty[S], v_empty[S];
  __shared__ uint64_t s_full[NT], p_full[NT];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;

  // ---- which (b, kv-head, row-tile group, split) this CTA owns; group index fastest so
  // CTAs that read the same K/V tiles run side by side.
  int bid = blockIdx.x;
  const int mp = bid % p.n_groups;
  bid /= p.n_groups;
  const int split = bid % p.splits;
  bid /= p.splits;
  const int g = bid % p.Hkv;
  const int b = bid / p.Hkv;

  const int cap = p.max_pages * kPage;
  int P = p.prefix_len[b];
  if (P < 0 || P > cap - p.N) {
    if (threadIdx.x == 0) report(p.dev_err, JF_DEVERR_BAD_PREFIX);
    P = max(0, min(P, cap - p.N));
  }
  const int L = P + p.N;
  const int ntiles = (L + kKeyTile - 1) / kKeyTile;
  const int k0 = split * p.chunk_tiles;
  const int k1 = min(ntiles, k0 + p.chunk_tiles);
  const int T = max(0, k1 - k0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (T == 0) {   // this split lies past the sequence: an empty partial (weight 0)
    if (warp >= 4) {
      const int t = (warp >> 2) - 1;
      const int r = (mp * NT + t) * kRowTile + ((warp & 3) * 32 + lane);
      if (r < p.M) {
        const int i = r / p.G, h = g * p.G + (r % p.G);
        const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.N + i;
        p.ws_lse[row * p.splits + split] = -INFINITY;
        float4* dst = reinterpret_cast<float4*>(p.ws_o + (row * p.splits + split) * D);
        for (int d = 0; d < D / 4; ++d) dst[d] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&o_full, 1);
    mbar_init(&fin, 1);
    for (int st = 0; st < S; ++st) {
      mbar_init(&k_full[st], 1);
      mbar_init(&v_full[st], 1);
      mbar_init(&k_empty[st], 1);
      mbar_init(&v_empty[st], 1);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  uint8_t* q_s = sm + C::kQOff;
  uint8_t* k_s = sm + C::kKOff;
  uint8_t* v_s = sm + C::kVOff;

  if (warp == 0) {
    // ================================================================ TMA producer
    int32_t* s_pages = reinterpret_cast<int32_t*>(sm + C::kPageOff);
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_pages;
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(&q_full, NT * C::kTileBytes);
      for (int t = 0; t < NT; ++t) {
        const int node0 = ((mp * NT + t) * kRowTile) / p.G;
        for (int hh = 0; hh < C::kHalves; ++hh)
          tma_load_4d(q_s + t * C::kTileBytes + hh * C::kHalfBytes, &qmap, &q_full, hh * 64,
                      g * p.G, node0, b);
      }
    }
    int issued = 0;
    bool ok = true;
    for (int j = 0; j < T && ok; ++j) {
      if (j % kPageWindowTiles == 0) {
        // Page ids of tiles [k0 + j, k0 + j + window): OOB id (zero fill) past the end.
        int bad = 0;
        for (int e = lane; e < kPageWindowTiles * kPagesPerTile; e += 32) {
          const int tile = k0 + j + e / kPagesPerTile;
          const int pl = tile * kPagesPerTile + (e % kPagesPerTile);
          int pid = p.num_pages;
          if (tile < k1 && pl * kPage < L) {
            const int v = bt[pl];
            if (v < 0 || v >= p.num_pages) bad = 1;
            else pid = v;
          }
          s_pages[e] = pid;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.dev_err, JF_DEVERR_BAD_PAGE);
        __syncwarp();
      }
      int okl = 1;
      if (lane == 0) {
        const int st = j % S;
        const uint32_t reuse_parity = static_cast<uint32_t>((j / S) - 1) & 1u;
        const int* pg = s_pages + (j % kPageWindowTiles) * kPagesPerTile;
        if (j >= S && !mbar_wait(&k_empty[st], reuse_parity, abort)) okl = 0;
        if (okl) {
          mbar_arrive_expect_tx(&k_full[st], C::kTileBytes);
          uint8_t* dst = k_s + st * C::kTileBytes;
          for (int q = 0; q < kPagesPerTile; ++q)
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_3d(dst + hh * C::kHalfBytes + q * (kPage * 128), &kmap, &k_full[st],
                          hh * 64, g, pg[q] * kPage);
        }
        if (okl && j >= S && !mbar_wait(&v_empty[st], reuse_parity, abort)) okl = 0;
        if (okl) {
          mbar_arrive_expect_tx(&v_full[st], C::kTileBytes);
          uint8_t* dst = v_s + st * C::kTileBytes;
          for (int q = 0; q < kPagesPerTile; ++q)
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_3d(dst + hh * C::kHalfBytes + q * (kPage * 128), &vmap, &v_full[st],
                          hh * 64, g, pg[q] * kPage);
          issued = j + 1;
        } else {
          set_abort(abort, p.dev_err);
        }
      }
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
    }
    // Drain: make sure no copy is still landing in shared memory when the CTA exits.
    if (lane == 0) {
      int zero_q = 0;
      mbar_wait(&q_full, 0, &zero_q);
      for (int j = max(0, issued - S); j < issued; ++j) {
        const uint32_t par = static_cast<uint32_t>(j / S) & 1u;
        int zero = 0;
        mbar_wait(&k_full[j % S], par, &zero);
        mbar_wait(&v_full[j % S], par, &zero);
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t idS = idesc_bf16(kRowTile, kKeyTile, false, false);
    constexpr uint32_t idO = idesc_bf16(kRowTile, D, false, true);
    auto issue_s = [&](int t, int st) {
      const uint32_t qa = smem_u32(q_s + t * C::kTileBytes);
      const uint32_t ka = smem_u32(k_s + st * C::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * C::kHalfBytes + (kk % 4) * 32;
        mma_ss(tmem + C::kTmemS + t * 128, desc_sw128(qa + off, 16, 1024),
               desc_sw128(ka + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int st, bool acc) {
      const uint32_t va = smem_u32(v_s + st * C::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < kKeyTile / 16; ++kk)
        mma_ts(tmem + C::kTmemO + t * 128, tmem + C::kTmemS + t * 128 + kk * 8,
               desc_sw128(va + kk * 16 * 128, C::kHalfBytes, 1024), idO,
               (acc || kk > 0) ? 1u : 0u);
    };
    bool ok = wait_warp(&q_full, 0, abort) && wait_warp(&k_full[0], 0, abort);
    if (ok && lane == 0) {
      tc_fence_after();
      for (int t = 0; t < NT; ++t) {
        issue_s(t, 0);
        mma_commit(&s_full[t]);
      }
      mma_commit(&k_empty[0]);
    }
    for (int j = 0; j < T && ok; ++j) {
      const int st = j % S;
      const uint32_t par = static_cast<uint32_t>(j / S) & 1u;
      if (!wait_warp(&v_full[st], par, abort)) { ok = false; break; }
      const int key0 = (k0 + j) * kKeyTile;
      if (key0 + kKeyTile > L) {
        // Zero V rows past the sequence end (all 64-column halves).
        const int r0 = L - key0;
        uint8_t* vt = v_s + st * C::kTileBytes;
        const int nchunks = (kKeyTile - r0) * 8 * C::kHalves;   // 16-byte chunks
        for (int c = lane; c < nchunks; c += 32) {
          const int hh = c / ((kKeyTile - r0) * 8);
          const int rem = c % ((kKeyTile - r0) * 8);
          const int row = r0 + rem / 8;
          *reinterpret_cast<uint4*>(vt + hh * C::kHalfBytes + row * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      for (int t = 0; t < NT && ok; ++t) {
        if (!wait_warp(&p_full[t], static_cast<uint32_t>(j) & 1u, abort)) { ok = false; break; }
        if (lane == 0) {
          tc_fence_after();
          issue_pv(t, st, j > 0);
        }
        if (j + 1 < T) {
          const int st1 = (j + 1) % S;
          if (t == 0 && !wait_warp(&k_full[st1], static_cast<uint32_t>((j + 1) / S) & 1u, abort)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            issue_s(t, st1);
            mma_commit(&s_full[t]);
          }
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(&v_empty[st]);
        if (j + 1 < T) mma_commit(&k_empty[(j + 1) % S]);
      }
      __syncwarp();
    }
    if (!ok) set_abort(abort, p.dev_err);
    if (lane == 0) {
      if (ok) mma_commit(&o_full);
      mma_commit(&fin);   // all MMAs done before TMEM is released
      int zero = 0;
      mbar_wait(&fin, 0, &zero);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ================================================================ softmax / epilogue
    const int t = (warp >> 2) - 1;
    const int wq = warp & 3;
    const int rl = wq * 32 + lane;                       // row within the tile = TMEM lane
    const int r = (mp * NT + t) * kRowTile + rl;
    const bool valid = r < p.M;
    const int node_base = ((mp * NT + t) * kRowTile) / p.G;
    const int i = r / p.G;
    const int h = g * p.G + (r % p.G);
    const int W = p.W;
    uint64_t* s_mask = reinterpret_cast<uint64_t*>(sm + C::kMaskOff + t * kMaskBytesPerTile);
    if (k1 * kKeyTile > P) {                             // this split reaches tree keys
      const int nodes = kRowTile / p.G;
      const uint64_t* src = p.mask + (static_cast<size_t>(b) * p.N + node_base) * W;
      for (int e = rl; e < nodes * W; e += 128)
        s_mask[e] = (node_base + e / W) < p.N ? src[e] : 0ull;
      named_bar(1 + t, 128);
    }
    const uint64_t* my_mask = s_mask + (rl / p.G) * W;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + C::kTmemS + t * 128 + lane_off;
    const uint32_t tO = tmem + C::kTmemO + t * 128 + lane_off;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      if (!wait_warp(&s_full[t], static_cast<uint32_t>(j) & 1u, abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld128(tS, sr);
      float* sv = reinterpret_cast<float*>(sr);
      const int key0 = (k0 + j) * kKeyTile;
      if (key0 + kKeyTile > P) {
#pragma unroll
        for (int c = 0; c < kKeyTile; ++c) {
          const int tk = key0 + c;
          const int jt = tk - P;
          bool vis = tk < P;
          if (!vis && tk < L) vis = (my_mask[jt >> 6] >> (jt & 63)) & 1ull;
          if (!vis) sv[c] = -INFINITY;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeyTile; ++c) mx = fmaxf(mx, sv[c]);
      const float mt = mx * sl2;
      const bool raise = mt > m_run + kRescaleThreshold;
      const float m_old = m_run;
      if (raise) m_run = mt;
      const float corr = raise ? fast_exp2(m_old - m_run) : 1.f;   // 0 when m_old = -inf
      const float neg = (m_run == -INFINITY) ? 0.f : -m_run;
      uint32_t pk[64];
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = fast_exp2(fmaf(sv[2 * c], sl2, neg));
        const float p1 = fast_exp2(fmaf(sv[2 * c + 1], sl2, neg));
        ls += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * corr + ls;
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      // O holds PV of tiles < j (complete: s_full of tile j was committed after them).
      const bool need = raise && j > 0 && m_old != -INFINITY;
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
      mbar_arrive(&p_full[t]);
    }
    if (ok && wait_warp(&o_full, 0, abort)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_run + __log2f(l) : -INFINITY;
      const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.N + i;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        if (valid) {
          if (p.splits == 1) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.out + ((static_cast<size_t>(b) * p.N + i) * p.Hq + h) * D + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
              dst[v] = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + (row * p.splits + split) * D + c * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                   __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
          }
        }
      }
      if (valid) {
        if (p.splits == 1) {
          if (p.lse != nullptr) p.lse[row] = lse2 * 0.69314718055994531f;
        } else {
          p.ws_lse[row * p.splits + split] = lse2;
        }
      }
    } else if (!ok) {
      set_abort(abort, p.dev_err);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// Merges split partials: O = sum_s 2^(lse_s - lse) O_s,  lse = log2 sum_s 2^lse_s.
// One warp per output row (b, h, i); each lane owns D/32 consecutive columns.
template <int D>
__global__ void __launch_bounds__(256)
    tree_attention_combine_kernel(const float* __restrict__ ws_o,
                                  const float* __restrict__ ws_lse, int splits, int N, int Hq,
                                  long long rows, uint16_t* __restrict__ out,
                                  float* __restrict__ lse) {
  constexpr int E = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* ls = ws_lse + row * splits;
  float mx = -INFINITY;
  for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, ls[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float l = ls[s];
    const float w = (l == -INFINITY) ? 0.f : exp2f(l - mx);
    wsum += w;
    const float* o = ws_o + (row * splits + s) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(o + e);
      acc[e] += w * v.x;
      acc[e + 1] += w * v.y;
      acc[e + 2] += w * v.z;
      acc[e + 3] += w * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int i = static_cast<int>(row % N);
  const long long bh = row / N;
  const int h = static_cast<int>(bh % Hq);
  const long long b = bh / Hq;
  uint16_t* dst = out + ((b * N + i) * Hq + h) * D + lane * E;
  uint32_t packed[E / 2];
#pragma unroll
  for (int e = 0; e < E; e += 2) packed[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  }
  if (lse != nullptr && lane == 0)
    lse[row] = (wsum > 0.f ? mx + __log2f(wsum) : -INFINITY) * 0.69314718055994531f;
}

// ------------------------------------------------------------------------ host side

struct AttnPlan {
  int NT, n_groups, splits, chunk_tiles;
  size_t ws_bytes;
};

bool shape_supported(int B, int N, int Hq, int Hkv, int D, int max_pages, int page_size) {
  if (B < 1 || N < 1 || N > JF_MAX_NODES || Hq < 1 || Hkv < 1 || max_pages < 1) return false;
  if (D != 64 && D != 128) return false;
  if (page_size != kPage) return false;
  if (Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  if (G > kRowTile || (G & (G - 1)) != 0) return false;
  const int W = (N + 63) / 64;
  if ((kRowTile / G) * W * 8 > kMaskBytesPerTile) return false;   // staged mask limit
  if (static_cast<long long>(max_pages) * kPage < N) return false;
  if (static_cast<long long>(max_pages) * kPage > (1ll << 30)) return false;
  return true;
}

bool plan_attention(int B, int N, int Hq, int Hkv, int D, int max_pages, int sms, AttnPlan* pl) {
  const int G = Hq / Hkv;
  const long long M = static_cast<long long>(N) * G;
  const int mtiles = static_cast<int>((M + kRowTile - 1) / kRowTile);
  pl->NT = mtiles >= 2 ? 2 : 1;
  pl->n_groups = (mtiles + pl->NT - 1) / pl->NT;
  const int max_tiles = (max_pages * kPage + kKeyTile - 1) / kKeyTile;
  const long long units = static_cast<long long>(B) * Hkv * pl->n_groups;
  if (sms <= 0) sms = 148;
  // Time model (arbitrary units of one key tile of one row tile at full tensor speed):
  // waves * (tiles per split + prologue) * max(compute, HBM share), plus the merge.
  const double hbm_per_tile = 2.0 * kKeyTile * D * 2;          // K + V bytes per key tile
  const double flops_per_tile = 4.0 * kRowTile * kKeyTile * D;  // QK^T + PV per row tile
  const double per_sm_flops = 1.9e15 / sms, hbm = 6.5e12;
  double best = 1e300;
  int best_s = 1;
  for (int s = 1; s <= max_tiles; ++s) {
    const int chunk = (max_tiles + s - 1) / s;
    if (s > 1 && (s - 1) * chunk >= max_tiles) continue;         // last split would be empty
    const long long ctas = units * s;
    const long long waves = (ctas + sms - 1) / sms;
    const double active = static_cast<double>(std::min<long long>(ctas, sms));
    const double t_tile = std::max(pl->NT * flops_per_tile / per_sm_flops, hbm_per_tile * active / hbm);
    double est = waves * (chunk + 1.5) * t_tile;
    if (s > 1) {
      const double part = static_cast<double>(B) * Hq * N * s * (D + 1) * 4.0;
      est += 3e-6 + 2.0 * part / hbm;
    }
    if (est < best * 0.98) { best = est; best_s = s; }
  }
  pl->splits = best_s;
  pl->chunk_tiles = (max_tiles + best_s - 1) / best_s;
  pl->ws_bytes = best_s > 1 ? static_cast<size_t>(B) * Hq * N * best_s * (D + 1) * sizeof(float) + 256 : 0;
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
            const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, int D>
jf_status launch(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                 const AttnParams& prm, long long grid, cudaStream_t s) {
  using C = Cfg<NT, D>;
  static std::mutex mu;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 64 || !attr_set[dev]) {
      if (cudaFuncSetAttribute(tree_attention_kernel<NT, D>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
          cudaSuccess)
        return JF_ERR_CUDA;
      if (dev < 64) attr_set[dev] = true;
    }
  }
  tree_attention_kernel<NT, D><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, s>>>(
      qm, km, vm, prm);
  return launch_status();
}

}  // namespace
}  // namespace jf

extern "C" size_t jf_tree_attention_workspace_size(int32_t B, int32_t N, int32_t Hq, int32_t Hkv,
                                                   int32_t D, int32_t max_pages,
                                                   int32_t page_size) {
  if (!jf::shape_supported(B, N, Hq, Hkv, D, max_pages, page_size)) return static_cast<size_t>(-1);
  const int sms = jf::current_sm_count();
  if (sms <= 0) return static_cast<size_t>(-1);
  jf::AttnPlan pl;
  jf::plan_attention(B, N, Hq, Hkv, D, max_pages, sms, &pl);
  return pl.ws_bytes;
}

extern "C" jf_status jf_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       const uint64_t* mask, int32_t B, int32_t N, int32_t Hq,
                                       int32_t Hkv, int32_t D, int32_t page_size,
                                       int32_t max_pages, int32_t num_pages, float scale,
                                       void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_err,
                                       jf_stream_t stream) {
  using namespace jf;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      prefix_len == nullptr || mask == nullptr || out == nullptr)
    return JF_ERR_INVALID_ARGUMENT;
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || D < 1 || page_size < 1 || max_pages < 1 ||
      num_pages < 1 || !(scale > 0.f) || !std::isfinite(scale))
    return JF_ERR_INVALID_ARGUMENT;
  if (!shape_supported(B, N, Hq, Hkv, D, max_pages, page_size)) return JF_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * kPage >= (1ll << 31)) return JF_ERR_UNSUPPORTED;
  if (!aligned_to(q, 16) || !aligned_to(k_cache, 16) || !aligned_to(v_cache, 16) ||
      !aligned_to(out, 16) || !aligned_to(mask, 8))
    return JF_ERR_MISALIGNED;
  const int sms = current_sm_count();
  if (sms <= 0) return JF_ERR_CUDA;
  AttnPlan pl;
  plan_attention(B, N, Hq, Hkv, D, max_pages, sms, &pl);
  if (pl.ws_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < pl.ws_bytes) return JF_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned_to(workspace, 16)) return JF_ERR_MISALIGNED;
  }
  const int G = Hq / Hkv;
  CUtensorMap qm, km, vm;
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                                static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hq) * D * 2,
                                   static_cast<cuuint64_t>(N) * Hq * D * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kRowTile / G), 1};
    if (!encode(&qm, q, 4, dims, strides, box)) return JF_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(num_pages) * kPage};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hkv) * D * 2};
    const cuuint32_t box[3] = {64, 1, kPage};
    if (!encode(&km, k_cache, 3, dims, strides, box)) return JF_ERR_CUDA;
    if (!encode(&vm, v_cache, 3, dims, strides, box)) return JF_ERR_CUDA;
  }
  AttnParams prm;
  prm.block_table = block_table;
  prm.prefix_len = prefix_len;
  prm.mask = mask;
  prm.out = static_cast<uint16_t*>(out);
  prm.lse = lse;
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  prm.ws_o = pl.ws_bytes > 0 ? static_cast<float*>(workspace) : nullptr;
  prm.ws_lse = pl.ws_bytes > 0 ? static_cast<float*>(workspace) + rows * pl.splits * D : nullptr;
  prm.dev_err = dev_err;
  prm.B = B; prm.N = N; prm.Hq = Hq; prm.Hkv = Hkv; prm.G = G; prm.W = (N + 63) / 64;
  prm.max_pages = max_pages; prm.num_pages = num_pages;
  prm.n_groups = pl.n_groups; prm.splits = pl.splits; prm.chunk_tiles = pl.chunk_tiles;
  prm.M = N * G;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const long long grid = static_cast<long long>(B) * Hkv * pl.splits * pl.n_groups;
  if (grid > 0x7FFFFFFFll) return JF_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  jf_status st;
  if (D == 128)
    st = pl.NT == 2 ? launch<2, 128>(qm, km, vm, prm, grid, s) : launch<1, 128>(qm, km, vm, prm, grid, s);
  else
    st = pl.NT == 2 ? launch<2, 64>(qm, km, vm, prm, grid, s) : launch<1, 64>(qm, km, vm, prm, grid, s);
  if (st != JF_OK) return st;
  if (pl.splits > 1) {
    const long long nb = (static_cast<long long>(rows) + 7) / 8;
    if (D == 128)
      tree_attention_combine_kernel<128><<<static_cast<unsigned>(nb), 256, 0, s>>>(
          prm.ws_o, prm.ws_lse, pl.splits, N, Hq, static_cast<long long>(rows),
          static_cast<uint16_t*>(out), lse);
    else
      tree_attention_combine_kernel<64><<<static_cast<unsigned>(nb), 256, 0, s>>>(
          prm.ws_o, prm.ws_lse, pl.splits, N, Hq, static_cast<long long>(rows),
          static_cast<uint16_t*>(out), lse);
    return launch_status();
  }
  return JF_OK;
}
