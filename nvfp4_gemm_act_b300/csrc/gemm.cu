// Block-scaled NVFP4 GEMM with a fused epilogue for sm_103a (B300).
//
//   acc[m, n] = sum_kb sA[m, kb] sB[n, kb] sum_{k in kb} qA[m, k] qB[n, k]     (tensor cores)
//   z = alpha * acc + bias[n];  y = epilogue(z)  -> HBM once                  (epilogue warps)
//
// Method: page "How fal made Ideogram V4 6x faster" (news.ditty.ir) -- NVFP4 GEMMs with the
// trailing small op fused into the epilogue (bias; per-head RMSNorm with head_dim 256;
// gated-SiLU "SiLU(C[:, :N//2]) * C[:, N//2:]" over weight columns paired at packing time).
//
// Design: a persistent kernel launched as CTA pairs (clusters of 2, one CTA per SM). A pair
// computes 256 x 256 output tiles with the 2-SM MMA (tcgen05.mma.cta_group::2, M256 N256
// K64): CTA r owns rows [128 r, 128 r + 128) of the tile and holds only half of the weight
// tile, so a 256-deep pipeline stage is 38 KB per SM (5 stages in flight). Pairs walk
// (row-tile pair, weight tile) tiles round-robin, row pairs fastest, so concurrent pairs
// share weight tiles in L2.
//   warp 0     (both CTAs) TMA producer of the codes: this CTA's A tile and its half of
//              the B tile;
//   warp 6     (both CTAs) TMA producer of the scales: this CTA's A scale tile and both B
//              scale bands (every CTA needs the scales of all 256 columns in its own TMEM).
//              Both producers' loads complete on the leader CTA's full barrier, where each of
//              the leader's two producers announces its bytes for both CTAs. Every load is a
//              plain (non-multicast) TMA load into the issuing CTA's own shared memory;
//   warp 1     (both CTAs) TMEM allocation (pair-collective); in the leader, the single
//              MMA-issuing thread, whose commits release the stage and publish the
//              accumulator in both CTAs;
//   warps 2-5  (leader) block-scale copies shared -> TMEM (tcgen05.cp.cta_group::2 copies
//              each CTA's own shared block into its own TMEM), warp 2 + j taking 64-deep
//              k-step j of every stage and running ahead of the MMA warp. A copy occupies its
//              issuing thread for about 120 cycles while copies from other warps do not slow
//              the MMAs, so the 12 copies of a 256-deep stage are spread over four warps;
//   warp 7     no role;
//   warps 8-15 (both CTAs) epilogue: TMEM lane = output row; two warps per 32-lane quarter,
//              one per 128-column half. Each thread pulls its 128 accumulator columns into
//              registers, then reports TMEM free to the leader, so the next tile's MMAs run
//              while it applies the epilogue and stores. Per-head RMSNorm sums are
//              thread-local, combined across the two halves through shared memory when a
//              head spans the whole tile.
// Registers: warpgroups 0-1 drop to 72 per thread (setmaxnreg) so that warpgroups 2-3 can
// hold a 128-column accumulator slice (176 per thread); 4 x 32 x (2 x 72 + 2 x 176) = 63488
// of the 512 x 128 the block is launched with.
// Every wait is bounded (NVFP4_ERR_TIMEOUT in *err on expiry; the CTA then drains what it
// issued, frees TMEM and exits).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;                 // rows of A per CTA (TMEM lanes)
constexpr int kBN = 256;                 // columns of the tile (TMEM accumulator columns)
constexpr int kBK = 256;                 // K elements per pipeline stage
constexpr int kBKBytes = kBK / 2;        // 128: one 128-byte swizzle row of packed E2M1
constexpr int kStages = 5;
constexpr int kMmaK = 64;                // K per tcgen05.mma (kind::mxf4nvf4)
constexpr int kKStepsPerStage = kBK / kMmaK;
constexpr int kCluster = 2;              // the CTA pair of the 2-SM MMA
constexpr int kBRowsPerCta = kBN / kCluster;

constexpr int kABytes = kBM * kBKBytes;                       // 16 KB
constexpr int kBBytes = kBRowsPerCta * kBKBytes;              // 16 KB (this CTA's half)
constexpr int kSfAtom = 512;                                  // 128 rows x 4 scales
constexpr int kSfaBytes = kKStepsPerStage * kSfAtom;          // 2 KB
constexpr int kSfbBytes = (kBN / 128) * kKStepsPerStage * kSfAtom;  // 4 KB: both bands

constexpr int kSfWarps = 4;              // warps issuing the scale copies (shared -> TMEM)
constexpr int kSfWarp0 = 2;
constexpr int kEpiWarp0 = 8;             // first epilogue warp (warpgroups 2 and 3)
constexpr int kEpiWarps = 8;
// register split (setmaxnreg on entering each role): warpgroups 0-1 lean, 2-3 epilogue
constexpr uint32_t kRegsLean = 72;
constexpr uint32_t kRegsEpilogue = 176;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = kEpiWarp0 * 32 + kEpiThreads;
constexpr int kHalf = kBN / 2;           // columns per epilogue warp
static_assert(kEpiWarp0 % 4 == 0, "epilogue warps must start on a warpgroup (TMEM lane quarters)");
static_assert(kThreads == 512 && kEpiWarp0 == 8, "two lean and two epilogue warpgroups");
// the split must fit in what the block is launched with (512 threads x 128 registers)
static_assert(128u * (2 * kRegsLean + 2 * kRegsEpilogue) <= 512u * 128u, "register split");

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSfa = kOffB + kStages * kBBytes;
constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr int kOffParam = kOffSfb + kStages * kSfbBytes;      // bias / gamma, double-buffered
constexpr int kParamBytes = 2 * 2 * kBN * 4;
constexpr int kOffXch = kOffParam + kParamBytes;              // RMSNorm half-row sums
constexpr int kXchBytes = 2 * kBM * 4;
constexpr int kOffEpiBuf = kOffXch + kXchBytes;               // per-warp store staging
constexpr int kEpiBufBytes = 32 * 64;                         // 32 rows x 64 bytes per warp
constexpr int kOffFlags = kOffEpiBuf + kEpiWarps * kEpiBufBytes;  // epilogue wait results
static_assert(2 * kEpiWarps * 4 <= 64, "two tiles' epilogue flags");
constexpr int kOffQTab = kOffFlags + 64;                     // NVFP4 output: 1/d and code tables
constexpr int kQTabBytes = 128 * 4 * 2;
constexpr int kOffBar = kOffQTab + kQTabBytes;
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
constexpr uint32_t kBarEpiXch0 = 2;      // + lane quarter: the two warps sharing a quarter (ids 2-5)

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1 (format 1), K-major, dense,
// UE4M3 scales (bit 23 = 0), scale-factor ids 0, N >> 3 at bits 17-22, M >> 4 at 24-28.
constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
constexpr uint32_t kIdesc = make_idesc(kCluster * kBM, kBN);

// Instruction descriptor for kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B E4M3 (format 0 at
// bits 7-9 and 10-12), both K-major, dense, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t make_idesc_f8(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
constexpr uint32_t kIdescF8 = make_idesc_f8(kCluster * kBM, kBN);

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
  // NVFP4 output (codes [M, width/2] + tiled scales, static output tensor scale) instead of
  // `out`: the bf16-rounded epilogue values are quantized exactly as nvfp4_quantize would
  int out_nvfp4;
  uint8_t* out_codes;
  uint8_t* out_scales;
  const float* out_ts;
};

// Shared tables and route of the output tensor scale (NVFP4 output only).
struct QuantOut {
  const float* inv_tab;
  const uint32_t* code_tab;
  ScaleRoute sr;
};

// Stores this warp's 32 rows x NV values (thread = row, y[] = its values, columns
// [col0, col0 + NV) of the output) through the warp's 2 KB shared buffer: each lane writes
// its row's next 64 bytes (16-byte pieces XOR-swizzled by row pair -- the TMA's 64-byte
// swizzle -- so the row-per-lane writes hit distinct banks), then one lane hands the 32 x 64
// byte box to the TMA. The warp issues no global stores of its own, and the memory
// instructions it does issue are a third of a read-back-and-store scheme's.
template <int NV>
__device__ __forceinline__ void store_rows(const EpiParams& p, const void* tm_out, const float* y, int row0,
                                           int col0, int width, uint32_t buf, int lane) {
  if (row0 >= p.M) return;  // the warp's 32 rows all lie past M (uniform across the warp)
  const bool bf16 = !p.out_fp32;
  const int swz_w = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < NV; c += 16) {
    if (bf16 && (c & 31) != 0) continue;  // bf16 chunks are 32 values; handled at c % 32 == 0
    if (col0 + c >= width) break;         // past a ragged last tile's columns
    // the TMA has finished reading the buffer's previous box
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
    // write: 64 bytes of this lane's row (bf16: 32 values; fp32: 16 values)
    if (bf16) {
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        const float* v = y + c + piece * 8;
        const uint4 w = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                   pack_bf16x2(v[6], v[7]));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 64 + ((piece ^ swz_w) * 16)),
                     "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                     : "memory");
      }
    } else {
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        const float* v = y + c + piece * 4;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 64 + ((piece ^ swz_w) * 16)),
                     "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                     "r"(__float_as_uint(v[3]))
                     : "memory");
      }
    }
    fence_proxy_async_smem();  // this lane's writes, visible to the TMA
    __syncwarp();
    if (lane == 0) {
      // rows past M and columns past the width are clipped by the tensor map
      if (NVFP4_INDEX_OK(row0 >= 0 && row0 < p.M && (row0 & 31) == 0 && col0 + c >= 0 && col0 + c < width &&
                         ((col0 + c) * (bf16 ? 2 : 4)) % 16 == 0))
        tma_store_2d(tm_out, buf, col0 + c, row0);
      bulk_commit_group();
    }
  }
}

// NVFP4 output of this thread's row (row0 + lane): its NV values y[] are output columns
// [col0, col0 + NV) (col0 and NV multiples of 64). Each 16-value block is rounded to bf16 and
// quantized; rows past M (padding of the 128-row scale tiles) get zero scales. Codes leave in
// 16-byte stores, a group's four scale bytes in one 32-bit store.
template <int NV>
__device__ __forceinline__ void store_rows_nvfp4(const EpiParams& p, const QuantOut& qo, const float* y, int row0,
                                                 int col0, int width, int lane) {
  static_assert(NV % 64 == 0, "whole 64-column groups");
  // rows past the scale tiles' padding (the second CTA of the last row pair when M spans an
  // odd number of 128-row blocks) have neither codes nor scales (uniform across the warp)
  if (row0 >= ((p.M + 127) / 128) * 128) return;
  const int row = row0 + lane;
  const uint32_t gpr = static_cast<uint32_t>(width) >> 6;  // 64-column scale atoms per row band
  const bool real = row < p.M;
  // a group of 4 blocks (64 columns, col a multiple of 64 and width % 64 == 0, so a group lies
  // wholly inside or wholly past the width): 32 code bytes contiguous in the row, 4 scale
  // bytes contiguous in the tiled layout (blocks 4g..4g+3 of one row)
#pragma unroll
  for (int g = 0; g < NV / 64; ++g) {
    const int col = col0 + g * 64;
    if (col >= width) break;
    uint32_t w[8];
    uint32_t sc = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float* v = y + g * 64 + b * 16;
      const uint4 lo = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                  pack_bf16x2(v[6], v[7]));
      const uint4 hi = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                                  pack_bf16x2(v[14], v[15]));
      uint2 c = make_uint2(0u, 0u);
      const uint32_t stored = real ? quantize_block(lo, hi, qo.sr, qo.inv_tab, qo.code_tab, c) : 0u;
      w[2 * b] = c.x;
      w[2 * b + 1] = c.y;
      sc |= stored << (8 * b);
    }
    if (real && NVFP4_INDEX_OK(row >= 0 && col >= 0 && (col & 63) == 0 && col + 64 <= width)) {
      uint4* dst = reinterpret_cast<uint4*>(p.out_codes + (int64_t)row * (width >> 1) + (col >> 1));
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    const uint32_t soff = scale_offset(static_cast<uint32_t>(row), static_cast<uint32_t>(col >> 4), gpr);
    if (NVFP4_INDEX_OK(row >= 0 && (soff & 3u) == 0u &&
                       static_cast<int64_t>(soff) + 4 <= static_cast<int64_t>((p.M + 127) / 128) * gpr * 512))
      *reinterpret_cast<uint32_t*>(p.out_scales + soff) = sc;
  }
}

template <int NV>
__device__ __forceinline__ void store_out(const EpiParams& p, const QuantOut& qo, const void* tm_out, const float* y,
                                          int row0, int col0, int width, uint32_t buf, int lane) {
  if (p.out_nvfp4)
    store_rows_nvfp4<NV>(p, qo, y, row0, col0, width, lane);
  else
    store_rows<NV>(p, tm_out, y, row0, col0, width, buf, lane);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  // sigma(g) = 1 / (1 + e^-g); __fdividef returns 0 once the denominator exceeds 2^126
  return g * __fdividef(1.0f, 1.0f + __expf(-g)) * u;
}

// Epilogue of one thread: its row's 128 columns [c0, c0 + 128) of the tile, already in z
// (z = alpha * acc + bias). `xch` is the shared half-row exchange (RMSNorm, head 256).
__device__ __forceinline__ void epilogue_row(const EpiParams& p, const QuantOut& qo, const void* tm_out,
                                             float (&z)[kHalf], int row0, int c0, int half, int row_local,
                                             const float* gamma_s, float* xch, uint32_t buf, int lane) {
  if (p.epi == NVFP4_EPI_GATED_SILU) {
    float y[kHalf / 2];
#pragma unroll
    for (int j = 0; j < kHalf / 2; ++j) y[j] = silu_mul(z[2 * j], z[2 * j + 1]);
    store_out<kHalf / 2>(p, qo, tm_out, y, row0, c0 >> 1, p.N >> 1, buf, lane);
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
        // only the two warps of this lane quarter (one per half) exchange their row sums; the
        // slots are free again by the next tile: every epilogue warp passes the per-tile
        // parameter barrier after reading its partner's sum
        xch[half * kBM + row_local] = s;
        named_bar_sync(kBarEpiXch0 + static_cast<uint32_t>(row_local >> 5), 64);
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
        // (z * scale) * gamma, two columns per packed multiply: the same roundings as scalar
        const uint64_t sc2 = f32x2(scale, scale);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 g = *reinterpret_cast<const float2*>(gamma_s + c * 32 + i);
          const uint64_t t = mul_f32x2(f32x2(z[c * 32 + i], z[c * 32 + i + 1]), sc2);
          unpack_f32x2(mul_f32x2(t, f32x2(g.x, g.y)), z[c * 32 + i], z[c * 32 + i + 1]);
        }
      }
    }
  }
  store_out<kHalf>(p, qo, tm_out, z, row0, c0, p.N, buf, lane);
}

// The kernel for both operand formats. kFp8: E4M3 codes, K bytes a row, one scale per tensor
// (kind::f8f6f4, K = 32 per MMA; a 128-byte stage row holds 128 K-elements); the scale
// producer and the scale-copy warps have no work and the MMA thread waits on the full
// barriers itself. Otherwise packed E2M1 codes with UE4M3 block scales (kind::mxf4nvf4,
// K = 64 per MMA). A stage is 128 bytes of each row either way, so the ring, the shared
// memory descriptors and the epilogue are the same.
template <bool kFp8>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_sfa,
                                          const CUtensorMap& tm_sfb, const CUtensorMap& tm_out, int K,
                                          int num_m_blocks, int num_tiles, const EpiParams& ep, int* err,
                                          uint64_t timeout_ns) {
  // num_tiles counts pair tiles: (row-tile pair, weight tile); row pairs fastest.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  // bars[0..S): full (used in the leader), [S..2S): empty, [2S..3S): scales in TMEM (leader),
  // [3S]: accumulator full, [3S+1]: accumulator empty (leader), [3S+2]: MMA drain,
  // [3S+3]: scale-copy drain
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
  auto sf_bar = [&](int s) { return smem_u32(bars + 2 * kStages + s); };
  const uint32_t acc_full_bar = smem_u32(bars + 3 * kStages);
  const uint32_t acc_empty_bar = smem_u32(bars + 3 * kStages + 1);
  const uint32_t drain_bar = smem_u32(bars + 3 * kStages + 2);
  const uint32_t sf_drain_bar = smem_u32(bars + 3 * kStages + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kStages + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row_bytes = kFp8 ? K : K / 2;           // codes per row of A and of B
  const int num_k_blocks = (row_bytes + kBKBytes - 1) / kBKBytes;
  const int k_steps = row_bytes / 32;               // 32-byte MMA k-steps (K % 64 == 0)
  const int k_atoms = K / 64;                       // NVFP4 scale tiles per 128-row band
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x / kCluster;
  const int num_clusters = gridDim.x / kCluster;
  const int num_pairs_m = (num_m_blocks + kCluster - 1) / kCluster;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    if (!kFp8) {
      prefetch_tmap(&tm_sfa);
      prefetch_tmap(&tm_sfb);
    }
    if (!ep.out_nvfp4) prefetch_tmap(&tm_out);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), kFp8 ? 1 : 2);  // the leader's producers' arrivals (+ both CTAs' bytes)
      mbar_init(empty_bar(s), 1);           // the leader's MMA commit
      mbar_init(sf_bar(s), kSfWarps);       // one commit from each scale-copy warp
    }
    mbar_init(acc_full_bar, 1);
    mbar_init(acc_empty_bar, kCluster * kEpiWarps);  // every epilogue warp of both CTAs
    mbar_init(drain_bar, 1);
    mbar_init(sf_drain_bar, kSfWarps);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated, before any signal
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  // ---------------- TMA producers (both CTAs) ----------------
  // warp 0: this CTA's A tile and its half of the B tile; warp 6: its A scale tile and both
  // B scale bands (every CTA needs the scales of all 256 columns). Both complete on the
  // leader CTA's full barrier, on which each producer of the leader announces its bytes for
  // both CTAs.
  auto producer = [&](const bool codes_part) {
    const uint64_t pol = policy_evict_normal();
    uint32_t kc = 0;  // k-blocks issued so far (ring position)
    bool ok = true;
    for (int pt = cluster_id; pt < num_tiles && ok; pt += num_clusters) {
      const int m_blk = (pt % num_pairs_m) * kCluster + rank;  // rows past M load as zeros
      const int n_blk = pt / num_pairs_m;
      const int b_row = n_blk * kBN + rank * kBRowsPerCta;
      for (int kb = 0; kb < num_k_blocks; ++kb) {
        const int s = kc % kStages;
        if (!mbar_wait(empty_bar(s), ((kc / kStages) & 1u) ^ 1u, timeout_ns, err)) {
          ok = false;
          break;
        }
        const uint32_t bar = mapa_shared(full_bar(s), 0);  // the leader's full barrier
        if (codes_part) {
          if (leader) mbar_arrive_expect_tx(full_bar(s), kCluster * (kABytes + kBBytes));
          tma_load_2d_pair(sbase + kOffA + s * kABytes, &tm_a, kb * kBKBytes, m_blk * kBM, bar, pol);
          tma_load_2d_pair(sbase + kOffB + s * kBBytes, &tm_b, kb * kBKBytes, b_row, bar, pol);
        } else {
          if (leader) mbar_arrive_expect_tx(full_bar(s), kCluster * (kSfaBytes + kSfbBytes));
          // scale tiles: row = band * k_atoms + first k-atom of the stage (4 atoms of 512 B)
          tma_load_2d_pair(sbase + kOffSfa + s * kSfaBytes, &tm_sfa, 0,
                           m_blk * k_atoms + kb * kKStepsPerStage, bar, pol);
          // both 128-column B scale bands into this CTA's own shared memory (every CTA needs
          // the scales of all 256 columns in its TMEM); plain loads, no multicast
#pragma unroll
          for (int h = 0; h < kBN / 128; ++h)
            tma_load_2d_pair(sbase + kOffSfb + s * kSfbBytes + h * (kSfbBytes / 2), &tm_sfb, 0,
                             (n_blk * 2 + h) * k_atoms + kb * kKStepsPerStage, bar, pol);
        }
        ++kc;
      }
    }
    // Before exit, no copy may still be in flight into either CTA's shared memory, and no
    // arrival of the leader may still be on its way to this CTA's barriers. The copies of both
    // CTAs complete on the leader's full barriers: the leader waits for the stages it issued
    // last (the follower stays until the leader reaches the closing cluster barrier); every
    // CTA waits for the leader's release of its stages (the MMA commits arrive on them).
    // On the normal path all of these have completed already; after a timed-out wait they
    // are waited for again, each within the time limit.
    const uint32_t first = kc > (uint32_t)kStages ? kc - kStages : 0u;
    if (leader)
      for (uint32_t i = first; i < kc; ++i)
        (void)mbar_wait(full_bar(i % kStages), (i / kStages) & 1u, timeout_ns, err);
    for (uint32_t i = first; i < kc; ++i)
      (void)mbar_wait(empty_bar(i % kStages), (i / kStages) & 1u, timeout_ns, err);
  };

  if (warp == 0) {
    warpgroup_reg_dealloc<kRegsLean>();
    if (lane == 0) producer(true);
  } else if (warp == 1) {
    warpgroup_reg_dealloc<kRegsLean>();
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader) ----------------
      uint32_t kc = 0;
      uint32_t it = 0;
      bool ok = true;
      for (int pt = cluster_id; pt < num_tiles && ok; pt += num_clusters, ++it) {
        // both CTAs' epilogues have pulled the previous accumulator out of TMEM
        if (!mbar_wait(acc_empty_bar, (it & 1u) ^ 1u, timeout_ns, err)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_k_blocks; ++kb) {
          const int s = kc % kStages;
          // NVFP4: the scales are in both TMEMs: the scale warps commit sf_bar only after they
          // saw the stage's full barrier, so the operands of both CTAs have landed too.
          // FP8: the operands of both CTAs have landed (the full barrier)
          if (!mbar_wait(kFp8 ? full_bar(s) : sf_bar(s), (kc / kStages) & 1u, timeout_ns, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = min(kKStepsPerStage, k_steps - kb * kKStepsPerStage);
          const uint32_t sf_col = tmem_base + kSfCol0 + s * kSfColsPerStage;
          const uint32_t a_s = sbase + kOffA + s * kABytes;
          const uint32_t b_s = sbase + kOffB + s * kBBytes;
          for (int j = 0; j < nk; ++j) {
            const uint64_t adesc = smem_desc(a_s + j * (kMmaK / 2), 16, 1024, kSwizzle128B);
            const uint64_t bdesc = smem_desc(b_s + j * (kMmaK / 2), 16, 1024, kSwizzle128B);
            if constexpr (kFp8)
              mma_f8_pair(tmem_base + kAccCol, adesc, bdesc, kIdescF8, (kb | j) != 0 ? 1u : 0u);
            else
              mma_nvf4_pair(tmem_base + kAccCol, adesc, bdesc, kIdesc, sf_col + j * 4,
                            sf_col + kSfaColsPerStage + j * 8, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(empty_bar(s), 0x3);  // release the stage in both CTAs
          ++kc;
        }
        if (ok) tc_commit_pair_mc(acc_full_bar, 0x3);
      }
      // Drain: every MMA issued has finished before TMEM is released.
      tc_commit_pair(drain_bar);
      (void)mbar_wait(drain_bar, 0u, timeout_ns, err);
    }
  } else if (warp < kSfWarp0 + kSfWarps) {
    warpgroup_reg_dealloc<kRegsLean>();
    if (!kFp8 && lane == 0 && leader) {
      // ---------------- block-scale copies, shared -> TMEM (leader, for both CTAs) --------
      // scale warp w copies the scales of 64-deep k-step w of each stage: A, B band 0, B
      // band 1; the TMEM slot of stage s is free again once stage s has been refilled (the
      // refill waited for the MMAs that read the previous scales).
      const int w = warp - kSfWarp0;
      uint32_t kc = 0;
      bool ok = true;
      for (int pt = cluster_id; pt < num_tiles && ok; pt += num_clusters) {
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
          for (int j = w; j < nk; j += kSfWarps) {
            tmem_cp_32x128b_x4_pair(sf_col + j * 4, smem_desc(sfa_s + j * kSfAtom, 128, 128, kSwizzleNone));
#pragma unroll
            for (int h = 0; h < kBN / 128; ++h)
              tmem_cp_32x128b_x4_pair(sf_col + kSfaColsPerStage + j * 8 + h * 4,
                                      smem_desc(sfb_s + h * (kSfbBytes / 2) + j * kSfAtom, 128, 128, kSwizzleNone));
          }
          tc_commit_pair(sf_bar(s));
          ++kc;
        }
      }
      tc_commit_pair(sf_drain_bar);
      (void)mbar_wait(sf_drain_bar, 0u, timeout_ns, err);
    }
  } else if (warp < kEpiWarp0) {
    // warp 6: scale-tile producer; warp 7: no role (it fills warpgroup 1)
    warpgroup_reg_dealloc<kRegsLean>();
    if (!kFp8 && warp == kEpiWarp0 - 2 && lane == 0) producer(false);
  } else {
    // ---------------- epilogue warps (both CTAs) ----------------
    warpgroup_reg_alloc<kRegsEpilogue>();
    const int ew = warp - kEpiWarp0;       // 0..7
    const int q = warp & 3;                // TMEM lane quarter this warp may access
    const int half = ew >> 2;              // which 128-column half of the tile
    const int et = ew * 32 + lane;         // 0..255
    const int row_local = q * 32 + lane;
    const uint32_t leader_acc_empty = mapa_shared(acc_empty_bar, 0);
    float* param = reinterpret_cast<float*>(smem + kOffParam);
    float* xch = reinterpret_cast<float*>(smem + kOffXch);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
    const float alpha = __fmul_rn(__ldg(ep.a_ts), __ldg(ep.b_ts));
    QuantOut qo;
    {
      float* inv_tab = reinterpret_cast<float*>(smem + kOffQTab);
      uint32_t* code_tab = reinterpret_cast<uint32_t*>(smem + kOffQTab + 512);
      qo.inv_tab = inv_tab;
      qo.code_tab = code_tab;
      const float ts_o = ep.out_nvfp4 ? __ldg(ep.out_ts) : 0.0f;
      qo.sr = scale_route(ts_o);
      if (ep.out_nvfp4 && et < 128) build_scale_table_entry(static_cast<uint32_t>(et), ts_o, inv_tab, code_tab);
      // (the first tile's epilogue-wide barrier orders the tables before any use)
    }
    const bool gated = ep.epi == NVFP4_EPI_GATED_SILU;
    const int nhalf = ep.N >> 1;
    uint32_t it = 0;
    for (int pt = cluster_id; pt < num_tiles; pt += num_clusters, ++it) {
      const int m_blk = (pt % num_pairs_m) * kCluster + rank;  // rows past M are not stored
      const int n_blk = pt / num_pairs_m;
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
          if (NVFP4_INDEX_OK(orig >= 0 && orig < ep.N)) b = __ldg(ep.bias + orig);
        }
        if (ep.epi == NVFP4_EPI_HEAD_RMSNORM && col < ep.norm_cols) g = __ldg(ep.gamma + col);
        bias_s[et] = b;
        gamma_s[et] = g;
      }
      // Each warp pulls its columns as soon as it sees the accumulator and hands TMEM back
      // to the leader's MMA warp; the epilogue-wide barrier (parameters staged, every warp's
      // wait result known) comes after, off the MMA warp's critical path.
      // (After a timed-out wait the pull reads stale TMEM, which is harmless: nothing is
      // stored and TMEM is not handed back.)
      const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait(acc_full_bar, it & 1u, timeout_ns, err));
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
      tc_fence_before();
      __syncwarp();
      if (ready && lane == 0) mbar_arrive_cluster(leader_acc_empty);
      // flags double-buffered by tile parity: a warp that is already on the next tile never
      // overwrites a flag another warp has still to read for this one
      volatile int* tile_flags = flags + (it & 1u) * kEpiWarps;
      if (lane == 0) tile_flags[ew] = ready ? 1 : 0;
      named_bar_sync(kBarEpiParams, kEpiThreads);
      bool all_ready = true;
#pragma unroll
      for (int w = 0; w < kEpiWarps; ++w) all_ready = all_ready && tile_flags[w] != 0;
      if (!all_ready) break;  // uniform across the epilogue warps
      const float* bh = bias_s + half * kHalf;
      {  // z = alpha * acc + bias, two columns per packed FMA (each half rounded as fmaf)
        const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < kHalf; i += 2) {
          const float2 b = *reinterpret_cast<const float2*>(bh + i);
          unpack_f32x2(fma_f32x2(a2, f32x2(z[i], z[i + 1]), f32x2(b.x, b.y)), z[i], z[i + 1]);
        }
      }
      epilogue_row(ep, qo, &tm_out, z, m_blk * kBM + q * 32, n_base + half * kHalf, half, row_local,
                   gamma_s + half * kHalf, xch, sbase + kOffEpiBuf + ew * kEpiBufBytes, lane);
    }
    // the warp's tile stores have completed (their sources are this CTA's shared memory)
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA of the pair leaves while the other may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                      const __grid_constant__ CUtensorMap tm_out, int K, int num_m_blocks, int num_tiles,
                      const __grid_constant__ EpiParams ep, int* err, uint64_t timeout_ns) {
  gemm_body<false>(tm_a, tm_b, tm_sfa, tm_sfb, tm_out, K, num_m_blocks, num_tiles, ep, err, timeout_ns);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_out, int K, int num_m_blocks, int num_tiles,
                    const __grid_constant__ EpiParams ep, int* err, uint64_t timeout_ns) {
  gemm_body<true>(tm_a, tm_b, tm_a, tm_a, tm_out, K, num_m_blocks, num_tiles, ep, err, timeout_ns);
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

// Codes [rows, row_bytes] (K/2 bytes a row for NVFP4, K for FP8) in boxes of box_rows rows x
// one 128-byte stage row, 128-byte swizzle.
bool encode_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tiled scale buffer seen as 32-bit words [atoms, 128]: one 512-byte atom per row,
// atoms ordered (128-row band, k-atom) with k-atoms fastest. A stage loads 4 atoms.
bool encode_scales_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t atoms = static_cast<cuuint64_t>((rows + 127) / 128) * static_cast<cuuint64_t>(K / 64);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kSfAtom / 4), atoms};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kSfAtom)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kSfAtom / 4), static_cast<cuuint32_t>(kKStepsPerStage)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The output [M, width] (row stride ldo elements) in boxes of 32 rows x 64 bytes with the
// 64-byte swizzle of the epilogue's staging buffers.
bool encode_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t width, int64_t ldo, bool fp32) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  const int64_t elem = fp32 ? 4 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldo * elem)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / elem), 32u};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Shared-memory opt-in and the register check, once per kernel: the setmaxnreg split assumes
// the block is launched with 128 registers per thread (with fewer, the epilogue warpgroups'
// increase could never be granted).
template <typename Kernel>
cudaError_t prepare_kernel(Kernel kernel) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
  if (e == cudaSuccess && fa.numRegs != 128) e = cudaErrorInvalidConfiguration;
  return e;
}

// As many clusters as can be resident at once (pairs are placed within a GPC).
template <typename Kernel>
int resident_clusters(Kernel kernel, const cudaLaunchConfig_t& cfg) {
  int n = 0;
  cudaLaunchConfig_t q = cfg;
  q.gridDim = dim3(sm_count(), 1, 1);
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &q) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = sm_count() / kCluster;
  }
  return n;
}

}  // namespace

nvfp4_status launch_gemm(const GemmArgs& a, cudaStream_t s) {
  CUtensorMap tm_a, tm_b, tm_sfa, tm_sfb, tm_out;
  const int64_t row_bytes = a.fp8 ? a.K : a.K / 2;
  if (!encode_codes_map(&tm_a, a.a_codes, a.M, row_bytes, kBM)) return NVFP4_ERR_LAUNCH;
  if (!encode_codes_map(&tm_b, a.b_codes, a.N, row_bytes, kBRowsPerCta)) return NVFP4_ERR_LAUNCH;
  if (!a.fp8) {
    if (!encode_scales_map(&tm_sfa, a.a_scales, a.M, a.K)) return NVFP4_ERR_LAUNCH;
    if (!encode_scales_map(&tm_sfb, a.b_scales, a.N, a.K)) return NVFP4_ERR_LAUNCH;
  }
  const int64_t width = a.epi == NVFP4_EPI_GATED_SILU ? a.N / 2 : a.N;
  if (a.out_nvfp4)
    std::memset(&tm_out, 0, sizeof(tm_out));  // unused: the NVFP4 output is stored directly
  else if (!encode_out_map(&tm_out, a.out, a.M, width, a.ldo, a.out_fp32 != 0))
    return NVFP4_ERR_LAUNCH;
  static const cudaError_t nvfp4_ready = prepare_kernel(gemm_nvfp4_kernel);
  static const cudaError_t fp8_ready = prepare_kernel(gemm_fp8_kernel);
  if ((a.fp8 ? fp8_ready : nvfp4_ready) != cudaSuccess) return NVFP4_ERR_LAUNCH;
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
  ep.out_nvfp4 = a.out_nvfp4;
  ep.out_codes = a.out_codes;
  ep.out_scales = a.out_scales;
  ep.out_ts = a.out_ts;
  const int num_m = static_cast<int>((a.M + kBM - 1) / kBM);
  const int num_n = static_cast<int>((a.N + kBN - 1) / kBN);
  const int num_pair_tiles = ((num_m + kCluster - 1) / kCluster) * num_n;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static const int nvfp4_clusters = resident_clusters(gemm_nvfp4_kernel, cfg);
  static const int fp8_clusters = resident_clusters(gemm_fp8_kernel, cfg);
  const int clusters = std::max(1, std::min(num_pair_tiles, a.fp8 ? fp8_clusters : nvfp4_clusters));
  cfg.gridDim = dim3(clusters * kCluster, 1, 1);
  const int K = static_cast<int>(a.K);
  const uint64_t limit = wait_timeout_ns();
  const cudaError_t e =
      a.fp8 ? cudaLaunchKernelEx(&cfg, gemm_fp8_kernel, tm_a, tm_b, tm_out, K, num_m, num_pair_tiles, ep, a.err, limit)
            : cudaLaunchKernelEx(&cfg, gemm_nvfp4_kernel, tm_a, tm_b, tm_sfa, tm_sfb, tm_out, K, num_m,
                                 num_pair_tiles, ep, a.err, limit);
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_LAUNCH;
}


// Failed index checks counted by this file's kernels since the last call (debug builds; always
// 0 otherwise); reading clears the counter. Call with the device idle.
cudaError_t take_index_failures_gemm(unsigned* n) {
#ifdef NVFP4_DEBUG
  unsigned v = 0u;
  const unsigned zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_index_failures, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_index_failures, &zero, sizeof(zero));
  *n = v;
  return e;
#else
  *n = 0u;
  return cudaSuccess;
#endif
}

}  // namespace nvfp4
