// Block-scaled NVFP4 GEMM with a fused epilogue for sm_103a (B300).
//
//   acc[m, n] = sum_kb sA[m, kb] sB[n, kb] sum_{k in kb} qA[m, k] qB[n, k]     (tensor cores)
//   z = alpha * acc + bias[n];  y = epilogue(z)  -> HBM once                  (epilogue warps)
//
// Method: page "How fal made Ideogram V4 6x faster" (news.ditty.ir) -- NVFP4 GEMMs with the
// trailing small op fused into the epilogue (bias; per-head RMSNorm with head_dim 256;
// gated-SiLU "SiLU(C[:, :N//2]) * C[:, N//2:]" over weight columns paired at packing time).
//
// Design: a persistent kernel, one CTA per SM, each CTA walking 128 x 256 output tiles
// (static round-robin over tiles, row tiles fastest so concurrent CTAs share weight tiles).
//   warp 0     TMA producer: A/B code tiles (128-byte swizzle) and the scale tiles (1-D bulk
//              copies) into a 4-stage shared-memory ring; it also prefetches the k-blocks
//              8 ahead into L2, so the ring is fed from L2 rather than DRAM latency;
//   warp 1     allocates TMEM; one thread copies each stage's scales shared -> TMEM
//              (tcgen05.cp) and issues tcgen05.mma kind::mxf4nvf4 (M128 N256 K64, UE4M3
//              scale per 16) into the fp32 accumulator, then frees the stage (tcgen05.commit);
//   warps 2-9  epilogue: TMEM lane = output row; two warps per 32-lane quarter, one per
//              128-column half. Each thread pulls its 128 accumulator columns into registers
//              and releases TMEM at once, so the next tile's MMAs run while it applies the
//              epilogue and stores. Per-head RMSNorm sums are thread-local, combined across
//              the two halves through shared memory when a head spans the whole tile.
// Every wait is bounded (NVFP4_ERR_TIMEOUT in *err on expiry; the CTA then drains what it
// issued, frees TMEM and exits).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;                 // rows of A per tile (TMEM lanes)
constexpr int kBN = 256;                 // columns of the tile (TMEM accumulator columns)
constexpr int kBK = 256;                 // K elements per pipeline stage
constexpr int kBKBytes = kBK / 2;        // 128: one 128-byte swizzle row of packed E2M1
constexpr int kStages = 4;
constexpr int kMmaK = 64;                // K per tcgen05.mma (kind::mxf4nvf4)
constexpr int kKStepsPerStage = kBK / kMmaK;
constexpr int kPrefetchDist = 8;         // k-blocks prefetched into L2 ahead of the ring

constexpr int kABytes = kBM * kBKBytes;                       // 16 KB
constexpr int kBBytes = kBN * kBKBytes;                       // 32 KB
constexpr int kSfAtom = 512;                                  // 128 rows x 4 scales
constexpr int kSfaBytes = (kBM / 128) * kKStepsPerStage * kSfAtom;  // 2 KB
constexpr int kSfbBytes = (kBN / 128) * kKStepsPerStage * kSfAtom;  // 4 KB

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kHalf = kBN / 2;           // columns per epilogue warp

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSfa = kOffB + kStages * kBBytes;
constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr int kOffParam = kOffSfb + kStages * kSfbBytes;      // bias / gamma, double-buffered
constexpr int kParamBytes = 2 * 2 * kBN * 4;
constexpr int kOffXch = kOffParam + kParamBytes;              // RMSNorm half-row sums
constexpr int kXchBytes = 2 * kBM * 4;
constexpr int kOffFlags = kOffXch + kXchBytes;                // epilogue wait results
constexpr int kOffBar = kOffFlags + 64;
constexpr int kBarBytes = 256;
constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;        // + slack to align to 1 KB

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;
constexpr uint32_t kSfCol0 = kBN;                             // scales after the accumulator
constexpr uint32_t kSfaColsPerStage = kKStepsPerStage * 4;    // 4 columns per 128-row atom
constexpr uint32_t kSfColsPerStage = kSfaColsPerStage + kKStepsPerStage * 4 * (kBN / 128);
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

constexpr uint32_t kBarEpiParams = 1;    // named barriers among the epilogue warps
constexpr uint32_t kBarEpiXch = 2;

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1 (format 1), K-major, dense,
// UE4M3 scales (bit 23 = 0), scale-factor ids 0, N >> 3 at bits 17-22, M >> 4 at 24-28.
constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
constexpr uint32_t kIdesc = make_idesc(kBM, kBN);

struct EpiParams {
  const float* a_ts;
  const float* b_ts;
  const float* bias;
  const float* gamma;
  void* out;
  int64_t ldo;
  int M;
  int N;
  int epi;
  int head_dim;
  int norm_cols;
  float eps;
  int out_fp32;
};

// Stores NV consecutive values of one output row (col multiple of 8, 16-byte aligned rows).
template <int NV>
__device__ __forceinline__ void store_row(const EpiParams& p, int row, int col, const float* y) {
  if (p.out_fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + (int64_t)row * p.ldo + col);
#pragma unroll
    for (int i = 0; i < NV / 4; ++i) dst[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo + col);
#pragma unroll
    for (int i = 0; i < NV / 8; ++i)
      dst[i] = make_uint4(pack_bf16x2(y[8 * i], y[8 * i + 1]), pack_bf16x2(y[8 * i + 2], y[8 * i + 3]),
                          pack_bf16x2(y[8 * i + 4], y[8 * i + 5]), pack_bf16x2(y[8 * i + 6], y[8 * i + 7]));
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g * __frcp_rn(1.0f + __expf(-g)) * u;
}

// Epilogue of one thread: its row's 128 columns [c0, c0 + 128) of the tile, already in z
// (z = alpha * acc + bias). `xch` is the shared half-row exchange (RMSNorm, head 256).
__device__ __forceinline__ void epilogue_row(const EpiParams& p, float (&z)[kHalf], int row, int c0,
                                             int half, int row_local, const float* gamma_s,
                                             float* xch) {
  const bool live = row < p.M;
  if (p.epi == NVFP4_EPI_GATED_SILU) {
    float y[kHalf / 2];
#pragma unroll
    for (int j = 0; j < kHalf / 2; ++j) y[j] = silu_mul(z[2 * j], z[2 * j + 1]);
    if (live) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c0 + c * 32 < p.N) store_row<16>(p, row, (c0 + c * 32) >> 1, y + c * 16);
    }
    return;
  }
  if (p.epi == NVFP4_EPI_HEAD_RMSNORM) {
    float cs[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) s = fmaf(z[c * 32 + i], z[c * 32 + i], s);
      cs[c] = s;
    }
    const int hd = p.head_dim;
    float hs[4];
    if (hd == 32) {
#pragma unroll
      for (int c = 0; c < 4; ++c) hs[c] = cs[c];
    } else if (hd == 64) {
      hs[0] = hs[1] = cs[0] + cs[1];
      hs[2] = hs[3] = cs[2] + cs[3];
    } else {
      float s = (cs[0] + cs[1]) + (cs[2] + cs[3]);
      if (hd == 256) {  // the head spans both halves of the tile row
        xch[half * kBM + row_local] = s;
        named_bar_sync(kBarEpiXch, kEpiThreads);
        const float o = xch[(half ^ 1) * kBM + row_local];
        s = half == 0 ? s + o : o + s;  // same summation order in both halves
      }
      hs[0] = hs[1] = hs[2] = hs[3] = s;
    }
    const float inv_hd = 1.0f / static_cast<float>(hd);  // power of two: exact
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c0 + c * 32 < p.norm_cols) {
        const float scale = rsqrtf(fmaf(hs[c], inv_hd, p.eps));
#pragma unroll
        for (int i = 0; i < 32; ++i) z[c * 32 + i] = z[c * 32 + i] * scale * gamma_s[c * 32 + i];
      }
    }
  }
  if (live) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c0 + c * 32 < p.N) store_row<32>(p, row, c0 + c * 32, z + c * 32);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb, int K,
                      int num_m_blocks, int num_tiles, EpiParams ep, int* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  // bars[0..S): full, [S..2S): empty, [2S]: accumulator full, [2S+1]: accumulator empty,
  // [2S+2]: MMA drain
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
  const uint32_t acc_full_bar = smem_u32(bars + 2 * kStages);
  const uint32_t acc_empty_bar = smem_u32(bars + 2 * kStages + 1);
  const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 3);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_k_blocks = (K + kBK - 1) / kBK;
  const int k_atoms = K / 64;                       // scale tiles per 128-row band
  const int sfb_bands = (ep.N + 127) / 128;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full_bar, 1);
    mbar_init(acc_empty_bar, kEpiWarps);
    mbar_init(drain_bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pol = policy_evict_normal();
      uint32_t kc = 0;  // k-blocks issued so far (ring position)
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m_blk = tile % num_m_blocks;
        const int n_blk = tile / num_m_blocks;
        const int halves = (n_blk * 2 + 1 < sfb_bands) ? 2 : 1;
        for (int kb = 0; kb < min(num_k_blocks, kPrefetchDist); ++kb) {
          tma_prefetch_2d(&tm_a, kb * kBKBytes, m_blk * kBM);
          tma_prefetch_2d(&tm_b, kb * kBKBytes, n_blk * kBN);
        }
        for (int kb = 0; kb < num_k_blocks; ++kb) {
          if (kb + kPrefetchDist < num_k_blocks) {
            tma_prefetch_2d(&tm_a, (kb + kPrefetchDist) * kBKBytes, m_blk * kBM);
            tma_prefetch_2d(&tm_b, (kb + kPrefetchDist) * kBKBytes, n_blk * kBN);
          }
          const int s = kc % kStages;
          if (!mbar_wait(empty_bar(s), ((kc / kStages) & 1u) ^ 1u, timeout_ns, err)) {
            ok = false;
            break;
          }
          const int nk = min(kKStepsPerStage, k_atoms - kb * kKStepsPerStage);
          const uint32_t sf_bytes = static_cast<uint32_t>(nk * kSfAtom);
          mbar_arrive_expect_tx(full_bar(s), kABytes + kBBytes + sf_bytes * (1 + halves));
          tma_load_2d(sbase + kOffA + s * kABytes, &tm_a, kb * kBKBytes, m_blk * kBM, full_bar(s), pol);
          tma_load_2d(sbase + kOffB + s * kBBytes, &tm_b, kb * kBKBytes, n_blk * kBN, full_bar(s), pol);
          bulk_load(sbase + kOffSfa + s * kSfaBytes,
                    sfa + ((size_t)m_blk * k_atoms + (size_t)kb * kKStepsPerStage) * kSfAtom, sf_bytes,
                    full_bar(s));
          for (int h = 0; h < halves; ++h)
            bulk_load(sbase + kOffSfb + s * kSfbBytes + h * (kSfbBytes / 2),
                      sfb + ((size_t)(n_blk * 2 + h) * k_atoms + (size_t)kb * kKStepsPerStage) * kSfAtom,
                      sf_bytes, full_bar(s));
          ++kc;
        }
      }
      // Make sure no copy into this CTA's shared memory is still in flight at exit.
      for (uint32_t i = kc > (uint32_t)kStages ? kc - kStages : 0u; i < kc; ++i)
        (void)mbar_wait(full_bar(i % kStages), (i / kStages) & 1u, timeout_ns, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t kc = 0;
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
        const int n_blk = tile / num_m_blocks;
        const int halves = (n_blk * 2 + 1 < sfb_bands) ? 2 : 1;
        // the epilogue has pulled the previous tile's accumulator out of TMEM
        if (!mbar_wait(acc_empty_bar, (it & 1u) ^ 1u, timeout_ns, err)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_k_blocks; ++kb) {
          const int s = kc % kStages;
          if (!mbar_wait(full_bar(s), (kc / kStages) & 1u, timeout_ns, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = min(kKStepsPerStage, k_atoms - kb * kKStepsPerStage);
          const uint32_t sf_col = tmem_base + kSfCol0 + s * kSfColsPerStage;
          const uint32_t sfa_s = sbase + kOffSfa + s * kSfaBytes;
          const uint32_t sfb_s = sbase + kOffSfb + s * kSfbBytes;
          for (int j = 0; j < nk; ++j) {
            tmem_cp_32x128b_x4(sf_col + j * 4, smem_desc(sfa_s + j * kSfAtom, 128, 128, kSwizzleNone));
            for (int h = 0; h < halves; ++h)
              tmem_cp_32x128b_x4(sf_col + kSfaColsPerStage + j * 8 + h * 4,
                                 smem_desc(sfb_s + h * (kSfbBytes / 2) + j * kSfAtom, 128, 128, kSwizzleNone));
          }
          const uint32_t a_s = sbase + kOffA + s * kABytes;
          const uint32_t b_s = sbase + kOffB + s * kBBytes;
          for (int j = 0; j < nk; ++j) {
            const uint64_t adesc = smem_desc(a_s + j * (kMmaK / 2), 16, 1024, kSwizzle128B);
            const uint64_t bdesc = smem_desc(b_s + j * (kMmaK / 2), 16, 1024, kSwizzle128B);
            mma_nvf4(tmem_base + kAccCol, adesc, bdesc, kIdesc, sf_col + j * 4,
                     sf_col + kSfaColsPerStage + j * 8, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(s));
          ++kc;
        }
        if (ok) tc_commit(acc_full_bar);
      }
      // Drain: every MMA this thread issued has finished before TMEM is released.
      tc_commit(drain_bar);
      (void)mbar_wait(drain_bar, 0u, timeout_ns, err);
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int ew = warp - 2;               // 0..7
    const int q = warp & 3;                // TMEM lane quarter this warp may access
    const int half = ew >> 2;              // which 128-column half of the tile
    const int et = ew * 32 + lane;         // 0..255
    const int row_local = q * 32 + lane;
    float* param = reinterpret_cast<float*>(smem + kOffParam);
    float* xch = reinterpret_cast<float*>(smem + kOffXch);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
    const float alpha = __fmul_rn(__ldg(ep.a_ts), __ldg(ep.b_ts));
    const bool gated = ep.epi == NVFP4_EPI_GATED_SILU;
    const int nhalf = ep.N >> 1;
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int m_blk = tile % num_m_blocks;
      const int n_blk = tile / num_m_blocks;
      const int n_base = n_blk * kBN;
      // per-column parameters of this tile -> shared memory (buffer it & 1)
      float* bias_s = param + (it & 1u) * (2 * kBN);
      float* gamma_s = bias_s + kBN;
      {
        const int col = n_base + et;
        float b = 0.0f, g = 1.0f;
        if (ep.bias != nullptr && col < ep.N) {
          // gated: packed column 2j is gate column j, 2j+1 is up column N/2 + j
          const int orig = gated ? ((col & 1) ? nhalf + (col >> 1) : (col >> 1)) : col;
          b = __ldg(ep.bias + orig);
        }
        if (ep.epi == NVFP4_EPI_HEAD_RMSNORM && col < ep.norm_cols) g = __ldg(ep.gamma + col);
        bias_s[et] = b;
        gamma_s[et] = g;
      }
      const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait(acc_full_bar, it & 1u, timeout_ns, err));
      if (lane == 0) flags[ew] = ready ? 1 : 0;
      named_bar_sync(kBarEpiParams, kEpiThreads);
      bool all_ready = true;
#pragma unroll
      for (int w = 0; w < kEpiWarps; ++w) all_ready = all_ready && flags[w] != 0;
      if (!all_ready) break;  // uniform across the epilogue warps
      tc_fence_after();
      float z[kHalf];
      {
        uint32_t (&r)[kHalf] = reinterpret_cast<uint32_t (&)[kHalf]>(z);
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + half * kHalf;
        tmem_ld_32cols(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(r + 0));
        tmem_ld_32cols(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_ld_32cols(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(r + 64));
        tmem_ld_32cols(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(r + 96));
        tmem_ld_wait();
      }
      // accumulator is in registers: hand TMEM back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty_bar);
      const float* bh = bias_s + half * kHalf;
#pragma unroll
      for (int i = 0; i < kHalf; ++i) z[i] = fmaf(alpha, z[i], bh[i]);
      const int row = m_blk * kBM + row_local;
      epilogue_row(ep, z, row, n_base + half * kHalf, half, row_local, gamma_s + half * kHalf, xch);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

nvfp4_status launch_gemm(const GemmArgs& a, cudaStream_t s) {
  CUtensorMap tm_a, tm_b;
  if (!encode_codes_map(&tm_a, a.a_codes, a.M, a.K, kBM)) return NVFP4_ERR_LAUNCH;
  if (!encode_codes_map(&tm_b, a.b_codes, a.N, a.K, kBN)) return NVFP4_ERR_LAUNCH;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return NVFP4_ERR_LAUNCH;
  EpiParams ep;
  ep.a_ts = a.a_ts;
  ep.b_ts = a.b_ts;
  ep.bias = a.bias;
  ep.gamma = a.gamma;
  ep.out = a.out;
  ep.ldo = a.ldo;
  ep.M = static_cast<int>(a.M);
  ep.N = static_cast<int>(a.N);
  ep.epi = a.epi;
  ep.head_dim = a.head_dim;
  ep.norm_cols = static_cast<int>(a.norm_cols);
  ep.eps = a.eps;
  ep.out_fp32 = a.out_fp32;
  const int num_m = static_cast<int>((a.M + kBM - 1) / kBM);
  const int num_n = static_cast<int>((a.N + kBN - 1) / kBN);
  const int num_tiles = num_m * num_n;
  const int grid = std::min(num_tiles, sm_count());
  gemm_nvfp4_kernel<<<grid, kThreads, kSmemBytes, s>>>(tm_a, tm_b, a.a_scales, a.b_scales,
                                                       static_cast<int>(a.K), num_m, num_tiles, ep, a.err,
                                                       wait_timeout_ns());
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_LAUNCH;
}

}  // namespace nvfp4
