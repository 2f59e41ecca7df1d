// jf_sm100.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family, built for
// sm_103a) features the kernels use: mbarriers, TMA tensor loads, TMEM allocation,
// tcgen05 MMA / commit / load / store, and the shared-memory matrix descriptors.
//
// Every wait here is bounded: a wait that runs past its time limit returns false so the
// caller can record an error and unwind instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace jf {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Time limit of one bounded wait.  Legitimate waits in these kernels last microseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;   // 1 s

// Waits for the phase with the given parity to complete.  Gives up (returns false) when
// *abort becomes non-zero (another role of the CTA gave up) or after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// ------------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// Tiled TMA stores from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every bulk store this thread committed has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Waits until every committed bulk store has finished reading its shared-memory source
// (the global writes may still be in flight; they complete before the grid does).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 dsmem_ld_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float2 dsmem_ld_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads
// (tensor-core operand fetches).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------ TMEM / tcgen05

// Whole warp: allocates ncols (power of two >= 32) TMEM columns; the base address is
// written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// MMA issue from a whole warp.  Every lane of the warp runs the issuing code (so loop
// counters and descriptors stay warp-uniform) and elect.sync picks the one lane that
// executes the tcgen05 instructions: always the same lane while the warp is converged, so
// the commits below track that lane's MMAs.  Issuing from lane 0 inside a divergent branch
// instead measured ~110-120 cycles per 128x128x16 MMA next to busy softmax warps on the
// same scheduler, against ~75-80 in this form (64 when the scheduler is otherwise idle).

// The mbarrier gets one arrival when every tcgen05 op the elected lane issued so far is
// done (whole warp calls).
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// The K-step MMAs of one 128 x N tile (kind::f16: bf16 in, fp32 accumulate) from a whole
// warp in one block: one elect.sync, constant accumulate predicates and 32-bit adds on the
// descriptors' start-address word (the word above it stays fixed; addresses stay below
// 256 KB, so the 14-bit field never carries into the next one).
// SS form: D[tmem] = sum_k A_k * B_k^T over KSTEPS steps of 16 (8 for a 128-wide K, 4 for
// 64), A_k / B_k at start-address offsets (16-byte units) from adesc / bdesc.
#define JF_MMA_SS_STEP(OFF, P) \
  "add.u32 al, %1, " #OFF ";\n\tadd.u32 bl, %3, " #OFF ";\n\t" \
  "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, " #P ";\n\t"
template <int KSTEPS>
__device__ __forceinline__ void mma_ss_tile(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  static_assert(KSTEPS == 8 || KSTEPS == 4, "D = 128 or 64");
  const uint32_t alo = static_cast<uint32_t>(adesc), ahi = static_cast<uint32_t>(adesc >> 32);
  const uint32_t blo = static_cast<uint32_t>(bdesc), bhi = static_cast<uint32_t>(bdesc >> 32);
  if constexpr (KSTEPS == 8) {
    // K steps of 16 bf16 (32 bytes) inside a 128-byte swizzle row, then the second 64-column
    // half 16 KB further on (1024 units of 16 bytes).
    asm volatile(
        "{\n\t.reg .pred e, pz, pa;\n\t.reg .b32 r, al, bl;\n\t.reg .b64 ad, bd;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 pz, 0, 0;\n\tsetp.eq.b32 pa, 0, 0;\n\t"
        JF_MMA_SS_STEP(0, pz) JF_MMA_SS_STEP(2, pa) JF_MMA_SS_STEP(4, pa) JF_MMA_SS_STEP(6, pa)
        JF_MMA_SS_STEP(1024, pa) JF_MMA_SS_STEP(1026, pa) JF_MMA_SS_STEP(1028, pa) JF_MMA_SS_STEP(1030, pa)
        "}" ::"r"(d_tmem), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, pz, pa;\n\t.reg .b32 r, al, bl;\n\t.reg .b64 ad, bd;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 pz, 0, 0;\n\tsetp.eq.b32 pa, 0, 0;\n\t"
        JF_MMA_SS_STEP(0, pz) JF_MMA_SS_STEP(2, pa) JF_MMA_SS_STEP(4, pa) JF_MMA_SS_STEP(6, pa)
        "}" ::"r"(d_tmem), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc)
        : "memory");
  }
}
#undef JF_MMA_SS_STEP

// TS form over 128 keys: D[tmem] (+)= sum_k A[tmem cols a + 8k] * B_k, B_k 16 rows of 128
// bytes (128 units of 16 bytes) apart; the first MMA accumulates onto D only if acc0.
#define JF_MMA_TS_STEP(ACOL, BOFF, P) \
  "add.u32 at, %1, " #ACOL ";\n\tadd.u32 bl, %2, " #BOFF ";\n\t" \
  "mov.b64 bd, {bl, %3};\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %4, " #P ";\n\t"
__device__ __forceinline__ void mma_ts_tile(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            bool acc0) {
  const uint32_t blo = static_cast<uint32_t>(bdesc), bhi = static_cast<uint32_t>(bdesc >> 32);
  asm volatile(
      "{\n\t.reg .pred e, p0, pa;\n\t.reg .b32 r, at, bl;\n\t.reg .b64 bd;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.b32 pa, 0, 0;\n\t"
      JF_MMA_TS_STEP(0, 0, p0) JF_MMA_TS_STEP(8, 128, pa) JF_MMA_TS_STEP(16, 256, pa) JF_MMA_TS_STEP(24, 384, pa)
      JF_MMA_TS_STEP(32, 512, pa) JF_MMA_TS_STEP(40, 640, pa) JF_MMA_TS_STEP(48, 768, pa) JF_MMA_TS_STEP(56, 896, pa)
      "}" ::"r"(d_tmem), "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc0 ? 1u : 0u)
      : "memory");
}
#undef JF_MMA_TS_STEP

// Shared-memory matrix descriptor, 128-byte swizzle.  Addresses and offsets in bytes.
//   K-major operand: rows of 128 B (64 bf16 along K), 8-row groups SBO bytes apart; LBO
//   unused.  MN-major operand: 64-element MN blocks LBO bytes apart, 8-row K groups SBO
//   bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;   // descriptor version for the sm_100 family
  d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 32 columns of 32-bit words: thread t of the warp gets lane (base + t),
// columns [col, col + 32).  Call tmem_ld_wait before reading the registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// Waits for this thread's outstanding tcgen05.ld; the register operands tie the wait to
// the loaded values so the compiler cannot read them before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                 "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                 "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 columns: thread t writes r[0..16) to lane (base + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in the low 16 bits.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace jf
