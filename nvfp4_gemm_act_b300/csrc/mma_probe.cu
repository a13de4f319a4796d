// Tensor-core instruction-rate probe (a diagnostic of the library, declared in nvfp4.h as
// nvfp4_debug_mma_rate): one thread of each CTA (of each CTA pair's leader, for the 2-SM form)
// issues `iters` back-to-back tcgen05.mma of one kind and shape on operands resident in
// shared memory, accumulating into TMEM, and records the SM cycles and nanoseconds the batch
// took (issue of the first to completion of the last). Operands and block scales are zero:
// nothing useful is computed, the figure is the rate at which the tensor pipe retires that
// instruction on this device, which bounds every GEMM built from it.
//
// Kinds: NVFP4 (kind::mxf4nvf4.block_scale.block16, K = 64, block scales in TMEM), FP8 E4M3
// (kind::f8f6f4, K = 32), BF16 (kind::f16, K = 16). Every kind reads 32 bytes of each operand
// row per instruction from 128-byte swizzled K-major tiles, as the GEMM's mainloop does.

#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kOffA = 0;                    // 128 rows x 128 B
constexpr int kOffB = 16 * 1024;            // up to 256 rows x 128 B
constexpr int kOffSf = 48 * 1024;           // 6 KB of block scales (4 k-steps: A, B bands 0-1)
constexpr int kOffBar = 56 * 1024;
constexpr int kProbeSmemUsed = kOffBar + 64;
// requesting this much dynamic shared memory keeps one CTA per SM, so each CTA has the SM's
// tensor pipe and all of its TMEM to itself
constexpr int kProbeSmem = 120 * 1024;
static_assert(kProbeSmemUsed + 1024 <= kProbeSmem, "probe shared memory");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;            // scales after a 256-column accumulator

__host__ __device__ constexpr uint32_t idesc_for(int kind, int m, int n) {
  // D fp32 (bits 4-5 = 1) for kind::f16 and kind::f8f6f4; A/B format at bits 7-9 and 10-12
  // (E2M1 = 1 for mxf4nvf4 with UE4M3 scales, E4M3 = 0 for f8f6f4, BF16 = 1 for f16);
  // N >> 3 at bits 17-22, M >> 4 at bits 24-28; K-major, dense.
  const uint32_t shape = (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
  if (kind == NVFP4_PROBE_NVFP4) return (1u << 7) | (1u << 10) | shape;
  if (kind == NVFP4_PROBE_FP8) return (1u << 4) | shape;
  return (1u << 4) | (1u << 7) | (1u << 10) | shape;
}

// The kind and the CTA-group form are template parameters, so the issue loop holds nothing but
// the descriptor arithmetic and the MMAs themselves (as a GEMM's mainloop does).
template <int kKind, bool pair>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t acc) {
  if constexpr (kKind == NVFP4_PROBE_NVFP4) {
    if constexpr (pair)
      mma_nvf4_pair(d, a, b, idesc, sfa, sfb, acc);
    else
      mma_nvf4(d, a, b, idesc, sfa, sfb, acc);
  } else if constexpr (kKind == NVFP4_PROBE_FP8) {
    if constexpr (pair) {
      mma_f8_pair(d, a, b, idesc, acc);
    } else {
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
          "l"(a), "l"(b), "r"(idesc), "r"(acc)
          : "memory");
    }
  } else {
    if constexpr (pair) {
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
          "l"(a), "l"(b), "r"(idesc), "r"(acc)
          : "memory");
    } else {
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
          "l"(a), "l"(b), "r"(idesc), "r"(acc)
          : "memory");
    }
  }
}

__device__ __forceinline__ uint64_t clock64_now() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
  return t;
}

// out[2 c] = SM cycles, out[2 c + 1] = ns of the batch of CTA (pair) c; written by the issuing
// CTA only.
template <bool kPair, int kind>
__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_probe_kernel(int n, int iters, long long* out, int* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const uint32_t bar_sf = smem_u32(bars + 0);
  const uint32_t bar_done = smem_u32(bars + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool leader = !kPair || cluster_ctarank() == 0;

  // zero the operands and scales (the tensor core reads them through the async proxy)
  for (int i = threadIdx.x; i < kOffBar / 16; i += kProbeThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar_sf, 1);
    mbar_init(bar_done, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const int m = kPair ? 256 : 128;
  const uint32_t idesc = idesc_for(kind, m, n);

  if (warp == 0 && lane == 0 && leader) {
    bool ok = true;
    if (kind == NVFP4_PROBE_NVFP4) {
      // block scales of 4 k-steps into TMEM (A: 4 columns a k-step, B: two 128-row bands)
      for (int j = 0; j < 4; ++j) {
        const uint64_t da = smem_desc(sbase + kOffSf + j * 512, 128, 128, kSwizzleNone);
        const uint64_t db0 = smem_desc(sbase + kOffSf + 2048 + j * 512, 128, 128, kSwizzleNone);
        const uint64_t db1 = smem_desc(sbase + kOffSf + 4096 + j * 512, 128, 128, kSwizzleNone);
        if (kPair) {
          tmem_cp_32x128b_x4_pair(tmem + kSfCol + j * 4, da);
          tmem_cp_32x128b_x4_pair(tmem + kSfCol + 16 + j * 8, db0);
          tmem_cp_32x128b_x4_pair(tmem + kSfCol + 16 + j * 8 + 4, db1);
        } else {
          tmem_cp_32x128b_x4(tmem + kSfCol + j * 4, da);
          tmem_cp_32x128b_x4(tmem + kSfCol + 16 + j * 8, db0);
          tmem_cp_32x128b_x4(tmem + kSfCol + 16 + j * 8 + 4, db1);
        }
      }
      if (kPair)
        tc_commit_pair(bar_sf);
      else
        tc_commit(bar_sf);
      ok = mbar_wait(bar_sf, 0u, timeout_ns, err);
      tc_fence_after();
    }
    if (ok) {
      const uint64_t c0 = clock64_now();
      const uint64_t g0 = global_timer_ns();
      for (int i = 0; i < iters; ++i) {
        const int j = i & 3;
        const uint64_t a = smem_desc(sbase + kOffA + j * 32, 16, 1024, kSwizzle128B);
        const uint64_t b = smem_desc(sbase + kOffB + j * 32, 16, 1024, kSwizzle128B);
        mma_issue<kind, kPair>(tmem, a, b, idesc, tmem + kSfCol + j * 4, tmem + kSfCol + 16 + j * 8,
                               i > 0 ? 1u : 0u);
      }
      if (kPair)
        tc_commit_pair_mc(bar_done, 0x3);
      else
        tc_commit(bar_done);
      ok = mbar_wait(bar_done, 0u, timeout_ns, err);
      const uint64_t c1 = clock64_now();
      const uint64_t g1 = global_timer_ns();
      const int c = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
      out[2 * c] = ok ? static_cast<long long>(c1 - c0) : -1;
      out[2 * c + 1] = ok ? static_cast<long long>(g1 - g0) : -1;
    }
  } else if (kPair && !leader && warp == 0 && lane == 0) {
    // the follower's TMEM and shared memory are in use until the leader's batch completes
    (void)mbar_wait(bar_done, 0u, timeout_ns, err);
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kPair, int kKind>
nvfp4_status launch_probe_form(int n, int iters, int ctas, long long* out, int* err, cudaStream_t s) {
  static const cudaError_t ready =
      cudaFuncSetAttribute(mma_probe_kernel<kPair, kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (ready != cudaSuccess) return NVFP4_ERR_LAUNCH;
  const uint64_t limit = wait_timeout_ns();
  cudaError_t e;
  if constexpr (!kPair) {
    mma_probe_kernel<false, kKind><<<ctas, kProbeThreads, kProbeSmem, s>>>(n, iters, out, err, limit);
    e = cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * ctas), 1, 1);
    cfg.blockDim = dim3(kProbeThreads, 1, 1);
    cfg.dynamicSmemBytes = kProbeSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mma_probe_kernel<true, kKind>, n, iters, out, err, limit);
  }
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_LAUNCH;
}

}  // namespace

nvfp4_status launch_mma_probe(int kind, int cta_group, int n, int iters, int ctas, long long* out, int* err,
                              cudaStream_t s) {
  const bool pair = cta_group == 2;
  switch (kind) {
    case NVFP4_PROBE_NVFP4:
      return pair ? launch_probe_form<true, NVFP4_PROBE_NVFP4>(n, iters, ctas, out, err, s)
                  : launch_probe_form<false, NVFP4_PROBE_NVFP4>(n, iters, ctas, out, err, s);
    case NVFP4_PROBE_FP8:
      return pair ? launch_probe_form<true, NVFP4_PROBE_FP8>(n, iters, ctas, out, err, s)
                  : launch_probe_form<false, NVFP4_PROBE_FP8>(n, iters, ctas, out, err, s);
    default:
      return pair ? launch_probe_form<true, NVFP4_PROBE_BF16>(n, iters, ctas, out, err, s)
                  : launch_probe_form<false, NVFP4_PROBE_BF16>(n, iters, ctas, out, err, s);
  }
}

}  // namespace nvfp4
