// Device-side helpers for the sm_103a kernels: inline PTX for mbarriers, TMA bulk copies,
// tcgen05 (tensor memory, block-scaled MMA) and bounded waits.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------------------
// Small utilities
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void report_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// Debug builds (-DNVFP4_DEBUG): NVFP4_INDEX_OK(cond) guards a store (or load) of the
// epilogues and the quantizers; a false condition skips the access and is counted in this
// translation unit's device counter (each .cu file is its own device module), which
// nvfp4_debug_index_failures reads. Nothing traps. Release builds compile the checks out: the
// macro is `true` and its condition is not evaluated.
#ifdef NVFP4_DEBUG
static __device__ unsigned int g_index_failures;
__device__ __forceinline__ bool index_check(bool ok) {
  if (!ok) atomicAdd(&g_index_failures, 1u);
  return ok;
}
#define NVFP4_INDEX_OK(cond) (::nvfp4::index_check(cond))
#else
#define NVFP4_INDEX_OK(cond) true
#endif

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with parity `parity` of barrier `bar` has completed, for at most
// `limit_ns` nanoseconds. On time-out records NVFP4_ERR_TIMEOUT in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      report_error(err, NVFP4_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------------------
// TMA (bulk tensor / bulk copies), global -> shared, completing on an mbarrier
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(cache_hint)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Tile load for a CTA pair: lands in this CTA's shared memory at `dst` and completes its bytes
// on the mbarrier at shared::cluster address `bar` (the pair leader's barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                                 uint32_t bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(cache_hint)
      : "memory");
}

// shared::cluster address of the variable at local shared address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in another CTA).
// Arrive on a barrier of any CTA of the cluster, with CTA-scope release semantics: it orders
// nothing but this thread's own prior work, so it does not wait for this thread's earlier
// global stores to become visible cluster-wide (a cluster-scope release would). Callers that
// hand TMEM back to the MMA thread order their tcgen05.ld first with tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}

// 1-D bulk copy: dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Tile store shared -> global through a tensor map (bulk-group completion); the box starts at
// (x, y) with x * element size a multiple of 16 bytes and x, y >= 0.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until this thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy with an L2 cache policy: dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(cache_hint)
      : "memory");
}

// Fire-and-forget global reductions at GPU scope.
__device__ __forceinline__ void red_max_relaxed_gpu(unsigned* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_or_relaxed_gpu(unsigned* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.or.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Release: this thread's earlier writes and reductions are visible before the add.
__device__ __forceinline__ void red_add_release_gpu(unsigned* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Per-thread register budget of the calling warp's warpgroup (every warp of the warpgroup
// executes the same call): give registers back to the block's pool / take them from it.
template <uint32_t kRegs>
__device__ __forceinline__ void warpgroup_reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegs) : "memory");
}
template <uint32_t kRegs>
__device__ __forceinline__ void warpgroup_reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegs) : "memory");
}

// Acquire load of a global word at GPU scope.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Prefetch one tile of a tensor map into L2 (no shared memory involved).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x),
               "r"(y)
               : "memory");
}

// Named barrier `id` over `count` threads (count a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// L2 eviction-priority policies for the cache_hint operand (createpolicy).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core
// ---------------------------------------------------------------------------------------

// Allocates `ncols` TMEM columns (power of two >= 32); the base address is written to the
// shared word at `dst`. Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading / stride byte
// offsets (16-byte units), fixed version bits 46-47 = 0b01, swizzle mode in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle & 7u) << 61;
  return d;
}
constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;

// Block-scaled MMA, NVFP4 (E2M1 x E2M1, UE4M3 scale per 16 K), D (fp32, TMEM) += A * B.
// One thread issues it.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.block16 [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copies a 32-row x 16-byte shared-memory block into TMEM, replicated into all four
// 32-lane quarters (the layout block-scale factors are read from). One thread issues it.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// ---- CTA-pair (cta_group::2) forms: a kernel uses either these or the cta_group::1 ones ----
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// M=256 block-scaled MMA over a CTA pair (issued by the pair leader): A rows 0-127 and
// 128-255 come from the two CTAs' shared memory, B's two 128-row halves likewise, each
// CTA's TMEM receives its 128 rows of D; scales are read from each CTA's own TMEM.
__device__ __forceinline__ void mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.block16 [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// D (+)= A B^T over K = 32 for E4M3 A and B (kind::f8f6f4, no block scales), as a CTA pair:
// M = 256 across the pair, operands in each CTA's shared memory.
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Copies the same shared-memory block of each CTA of the pair into that CTA's TMEM.
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(cta_mask)
      : "memory");
}

// Arrives on `bar` once every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Loads 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// Number-format conversions (hardware cvt instructions)
// ---------------------------------------------------------------------------------------

// Two fp32 -> packed E2M1 pair, round to nearest even, saturating; `lo` lands in bits 0-3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// fp32 (>= 0) -> E4M3 code, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return static_cast<uint32_t>(r & 0xFFu);
}

// Two fp32 -> two signed E4M3 codes (round to nearest even, saturating at +-448), lo in bits
// 0-7, hi in bits 8-15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

// E4M3 code -> fp32 value (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.u16.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(code & 0xFFu));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


// ---------------------------------------------------------------------------------------
// NVFP4 block quantization (shared by the activation quantizer and the GEMM epilogue's NVFP4
// output): per block of 16, s = E4M3(fp32(bamax / fp32(6 ts))); d = fp32(dec(s) ts); a block
// with d < 2^-126 stores scale 0 and codes +0; otherwise code = E2M1(fp32(x * fp32(1 / d))).
// ---------------------------------------------------------------------------------------

constexpr float kFltMin = 1.17549435082e-38f;  // 2^-126

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values as one packed pair (lo in the low half) and the packed product of two pairs:
// each half rounded to nearest even exactly as a scalar fp32 multiply.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t p;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(lo), "f"(hi));
  return p;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// a * b + c on each half, one rounding (as fmaf), and a pair back to its two halves.
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Four packed pairs -> four bytes of E2M1 codes (nearest even, saturating), byte j from pair
// j, its low nibble from the pair's low half.
__device__ __forceinline__ uint32_t e2m1x8(uint64_t p0, uint64_t p1, uint64_t p2, uint64_t p3) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .f32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      "mov.b64 {l0, h0}, %1;\n\tmov.b64 {l1, h1}, %2;\n\tmov.b64 {l2, h2}, %3;\n\tmov.b64 {l3, h3}, %4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, h0, l0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, h1, l1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, h2, l2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, h3, l3;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "l"(p0), "l"(p1), "l"(p2), "l"(p3));
  return r;
}

// 8 bf16 values (in memory order) -> 4 bytes of E2M1 codes, element 2j in the low nibble:
// code = E2M1(fp32(x * inv)), the four products of each pair of words in packed multiplies.
__device__ __forceinline__ uint32_t encode8(const uint4& v, float inv) {
  const uint64_t iv = f32x2(inv, inv);
  return e2m1x8(mul_f32x2(f32x2(bf16_lo(v.x), bf16_hi(v.x)), iv), mul_f32x2(f32x2(bf16_lo(v.y), bf16_hi(v.y)), iv),
                mul_f32x2(f32x2(bf16_lo(v.z), bf16_hi(v.z)), iv), mul_f32x2(f32x2(bf16_lo(v.w), bf16_hi(v.w)), iv));
}

// max(|a|, |b|) per bf16 lane (the sign of the result is discarded by the caller).
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// |bf16| maximum of the 16 values in lo, hi, as the fp32 value (exact).
__device__ __forceinline__ float absmax16(const uint4& lo, const uint4& hi) {
  const uint32_t m = bf16x2_max_abs(bf16x2_max_abs(bf16x2_max_abs(lo.x, lo.y), bf16x2_max_abs(lo.z, lo.w)),
                                    bf16x2_max_abs(bf16x2_max_abs(hi.x, hi.y), bf16x2_max_abs(hi.z, hi.w)));
  const uint32_t h = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
  return __uint_as_float(h << 16);
}

// Entry c (0..127) of the tables of one tensor scale: fp32(1 / d) and the stored code for the
// E4M3 code c, d = fp32(dec(c) ts); zero entries for a zero block. Code 127 is E4M3 NaN (never
// produced by the saturating conversion). Callers fill all 128 entries, then synchronise.
__device__ __forceinline__ void build_scale_table_entry(uint32_t c, float ts, float* inv_tab, uint32_t* code_tab) {
  const float d = __fmul_rn(e4m3_to_f32(c), ts);
  const bool live = ts > 0.0f && c < 127u && d >= kFltMin;
  inv_tab[c] = live ? __fdiv_rn(1.0f, d) : 0.0f;
  code_tab[c] = live ? c : 0u;
}

struct ScaleRoute {
  float six_ts;
  float rcp_six_ts;
  bool fast;  // 1 / (6 ts) finite and normal: the reciprocal route applies
};

__device__ __forceinline__ ScaleRoute scale_route(float ts) {
  ScaleRoute r;
  r.six_ts = __fmul_rn(6.0f, ts);
  r.fast = r.six_ts >= 0x1p-125f && r.six_ts <= 0x1p125f;
  r.rcp_six_ts = r.fast ? __frcp_rn(r.six_ts) : 0.0f;
  return r;
}

// One 16-element block (lo: elements 0-7, hi: 8-15): its 8 code bytes; returns the stored
// scale code (0 for a zero block, whose codes are +0).
__device__ __forceinline__ uint32_t quantize_block(const uint4& lo, const uint4& hi, const ScaleRoute& sr,
                                                   const float* inv_tab, const uint32_t* code_tab, uint2& out) {
  const float bamax = absmax16(lo, hi);
  uint32_t s;
  if (sr.fast) {
    // both ends of the window in one packed multiply and one paired conversion (codes of
    // non-negative values: bits 0-7 from the low end, 8-15 from the high end)
    const float qa = __fmul_rn(bamax, sr.rcp_six_ts);
    uint32_t ends;
    {
      float e_lo, e_hi;
      const uint64_t e = mul_f32x2(f32x2(qa, qa), f32x2(1.0f - 0x1p-20f, 1.0f + 0x1p-20f));
      asm("mov.b64 {%0, %1}, %2;" : "=f"(e_lo), "=f"(e_hi) : "l"(e));
      ends = cvt_e4m3x2(e_lo, e_hi);
    }
    s = (ends & 0xFFu) == (ends >> 8) ? (ends & 0xFFu) : cvt_e4m3(__fdiv_rn(bamax, sr.six_ts));
  } else {
    s = cvt_e4m3(__fdiv_rn(bamax, sr.six_ts));
  }
  s &= 127u;
  const uint32_t stored = code_tab[s];
  out = make_uint2(0u, 0u);
  if (stored != 0u) {
    const float inv = inv_tab[s];
    out = make_uint2(encode8(lo, inv), encode8(hi, inv));
  }
  return stored;
}

// Byte offset of the scale of (row r, 16-element block kb) in the tiled scale layout.
__device__ __forceinline__ uint32_t scale_offset(uint32_t r, uint32_t kb, uint32_t gpr) {
  return ((r >> 7) * gpr + (kb >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u + (kb & 3u);
}


}  // namespace nvfp4
