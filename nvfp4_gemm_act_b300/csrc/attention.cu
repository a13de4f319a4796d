// Scaled dot-product attention (forward, no mask, bf16 in and out, fp32 softmax and
// accumulation) for sm_103a, head_dim 256: the DiT block's other large op, between the QKV
// projection (which writes Q | K | V side by side, heads contiguous in each) and the output
// projection. Page "How fal made Ideogram V4 6x faster": a pass costs the sum of its layers;
// page "WaveSpeedAI x DataCrunch: FLUX real-time image inference on B200" names a Blackwell
// attention kernel among its optimizations.
//
//   out[m, h*256 + d] = sum_j softmax_j(q_m . k_j / 16) v_j[d]      (per head h)
//
// Design: one CTA per (128-query tile, head), one CTA per SM (224 KB of shared memory).
//   warp 0     TMA producer of Q (once: 4 boxes of 128 rows x 64 columns) and of the K tiles
//              (4 boxes of 64 keys x 64) into a 3-stage ring; a K stage is free again as soon
//              as the S MMAs that read it have completed, so a K tile is requested two tiles
//              ahead of its use (K and V^T tiles take 2,600-4,400 cycles to arrive, measured:
//              each SM takes them in at ~33 bytes a cycle);
//   warp 2     TMA producer of the V^T tiles (256 x 64 keys) into their own 2-stage ring; a V
//              stage is free again when the PV MMAs that read it have completed;
//   warp 1     TMEM allocation (512 columns: two 64-column S buffers, two 32-column P buffers,
//              a 256-column O) and the MMA-issuing thread: S_j = Q K_j^T (M128 N64, 16 x K16,
//              both operands in shared memory), then O += P_{j-1} V_{j-1} (M128 N256, 4 x K16,
//              P read from TMEM), so that the softmax of tile j runs while PV_{j-1} does;
//   warps 4-7  softmax, one query row per thread (TMEM lane = row): S from TMEM, running max
//              in log2 units, p = 2^(s log2(e) / 16 - m) rounded to bf16 and stored into the
//              row's P buffer in TMEM (two bf16 per column), running sum l in fp32. O is
//              rescaled (TMEM load, scale, store) only when a row's max grows by more than 8
//              (a factor 256): until then p <= 256 and the stale max cancels in O / l.
//              At the end O / l is written as bf16.
// Every shared-memory operand is K-major with the 128-byte swizzle: V is handed over
// transposed (V^T, keys contiguous), written by a transpose kernel from the QKV output.
// Every wait is bounded (NVFP4_ERR_TIMEOUT in *err on expiry); a CTA that gives up drains
// what it issued and frees TMEM before it exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kHd = 256;            // head_dim
constexpr int kBQ = 128;            // queries per CTA (TMEM lanes)
constexpr int kBKV = 64;            // keys per tile
constexpr int kKStages = 3;         // K ring
constexpr int kVStages = 2;         // V^T ring
constexpr int kChunk = 64;          // bf16 elements in one 128-byte swizzle row
constexpr int kQChunkBytes = kBQ * 128;        // 16 KB
constexpr int kQBytes = (kHd / kChunk) * kQChunkBytes;   // 64 KB
constexpr int kKChunkBytes = kBKV * 128;       // 8 KB
constexpr int kKBytes = (kHd / kChunk) * kKChunkBytes;   // 32 KB
constexpr int kVBytes = kHd * 128;             // 32 KB: 256 rows (d) x 64 keys
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kKStages * kKBytes;
constexpr int kOffBar = kOffV + kVStages * kVBytes;
constexpr int kBarBytes = 256;                   // 18 barriers and the TMEM slot
constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;   // + 1 KB alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
constexpr int kThreads = 256;
constexpr int kSoftWarp0 = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;       // S buffer b at columns [64 b, 64 b + 64)
constexpr uint32_t kColP = 128;     // P buffer b at columns [128 + 32 b, 160 + 32 b): 64 bf16 a row
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B bf16 (format 1 at bits 7-9
// and 10-12), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_bf16(kBQ, kBKV);
constexpr uint32_t kIdescO = idesc_bf16(kBQ, kHd);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (fp32, TMEM) (+)= A B^T with A (bf16, M = 128 rows = TMEM lanes, two K-elements per
// column) in TMEM and B in shared memory (kind::f16, K = 16 per instruction).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr) { return smem_desc(addr, 16, 1024, kSwizzle128B); }

// 2^x with the MUFU approximation (ex2.approx.ftz.f32: about 2 ulp; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_vt, int M, int hidden, __nv_bfloat16* __restrict__ out,
                     int64_t ldo, int* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  // bars: [0] Q full; [1, 4) K stage full; [4, 7) K stage free (MMA commit after S);
  // [7, 9) S buffer full (MMA commit); [9, 11) S buffer read (4 softmax warps); [11, 13) P
  // buffer written (4 softmax warps); [13, 15) PV done with P buffer b (MMA commit: P buffer
  // and V stage free, O updated); [15, 17) V stage full; [17] drain
  const uint32_t q_full = smem_u32(bars);
  auto k_full = [&](int b) { return smem_u32(bars + 1 + b); };
  auto k_free = [&](int b) { return smem_u32(bars + 4 + b); };
  auto s_full = [&](int b) { return smem_u32(bars + 7 + b); };
  auto s_free = [&](int b) { return smem_u32(bars + 9 + b); };
  auto p_full = [&](int b) { return smem_u32(bars + 11 + b); };
  auto pv_done = [&](int b) { return smem_u32(bars + 13 + b); };
  auto v_full = [&](int b) { return smem_u32(bars + 15 + b); };
  const uint32_t drain_bar = smem_u32(bars + 17);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  static_assert(19 * 8 <= kBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kBQ;
  const int head = blockIdx.y;
  const int nt = (M + kBKV - 1) / kBKV;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_vt);
    mbar_init(q_full, 1);
    for (int b = 0; b < kKStages; ++b) {
      mbar_init(k_full(b), 1);
      mbar_init(k_free(b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(v_full(b), 1);
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), 4);
      mbar_init(p_full(b), 4);
      mbar_init(pv_done(b), 1);
    }
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

  if (warp == 0 || warp == 2) {
    if (lane == 0) {
      // ---------------- TMA producers: Q and K (warp 0), V^T (warp 2) ----------------
      const bool kpart = warp == 0;
      const uint64_t pol = policy_evict_normal();
      if (kpart) {
        mbar_arrive_expect_tx(q_full, kQBytes);
        for (int c = 0; c < kHd / kChunk; ++c)
          tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_q, head * kHd + c * kChunk, q0, q_full, pol);
      }
      const int kcol = hidden + head * kHd;
      const int stages = kpart ? kKStages : kVStages;
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int b = j % stages;
        const uint32_t use = static_cast<uint32_t>(j / stages);  // this stage's use count
        // the stage's previous tile has been read: by its S MMAs (K) or its PV MMAs (V)
        if (j >= stages &&
            !mbar_wait(kpart ? k_free(b) : pv_done(b), (use - 1u) & 1u, timeout_ns, err))
          break;
        if (kpart) {
          const uint32_t stage = sbase + kOffK + b * kKBytes;
          mbar_arrive_expect_tx(k_full(b), kKBytes);
          for (int c = 0; c < kHd / kChunk; ++c)
            tma_load_2d(stage + c * kKChunkBytes, &tm_k, kcol + c * kChunk, j * kBKV, k_full(b), pol);
        } else {
          mbar_arrive_expect_tx(v_full(b), kVBytes);
          tma_load_2d(sbase + kOffV + b * kVBytes, &tm_vt, j * kBKV, head * kHd, v_full(b), pol);
        }
        issued = j + 1;
      }
      // No copy may still be in flight when the CTA exits: the last loads of every stage (the
      // earlier ones were waited for before their stage was reused) and the Q tile.
      if (kpart) (void)mbar_wait(q_full, 0u, timeout_ns, err);
      for (int j = issued >= stages ? issued - stages : 0; j < issued; ++j)
        (void)mbar_wait(kpart ? k_full(j % stages) : v_full(j % stages), static_cast<uint32_t>(j / stages) & 1u,
                        timeout_ns, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      bool ok = mbar_wait(q_full, 0u, timeout_ns, err);
      auto issue_pv = [&](int i) {
        const int b = i & 1;
        if (!mbar_wait(v_full(b), (i >> 1) & 1u, timeout_ns, err) ||
            !mbar_wait(p_full(b), (i >> 1) & 1u, timeout_ns, err))
          return false;
        tc_fence_after();
        const uint32_t v_s = sbase + kOffV + b * kVBytes;
#pragma unroll
        for (int k = 0; k < kBKV / 16; ++k)
          mma_bf16_tmem_a(tmem_base + kColO, tmem_base + kColP + b * (kBKV / 2) + k * 8, kmajor_desc(v_s + k * 32),
                          kIdescO, (i | k) != 0 ? 1u : 0u);
        tc_commit(pv_done(b));
        return true;
      };
      for (int j = 0; j < nt && ok; ++j) {
        const int b = j & 1;
        const int kb = j % kKStages;
        ok = mbar_wait(k_full(kb), static_cast<uint32_t>(j / kKStages) & 1u, timeout_ns, err) &&
             (j < 2 || mbar_wait(s_free(b), ((j - 2) >> 1) & 1u, timeout_ns, err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t k_s = sbase + kOffK + kb * kKBytes;
#pragma unroll
        for (int c = 0; c < kHd / kChunk; ++c)
#pragma unroll
          for (int k = 0; k < kChunk / 16; ++k)
            mma_bf16(tmem_base + kColS + b * kBKV, kmajor_desc(sbase + kOffQ + c * kQChunkBytes + k * 32),
                     kmajor_desc(k_s + c * kKChunkBytes + k * 32), kIdescS, (c | k) != 0 ? 1u : 0u);
        tc_commit(s_full(b));
        tc_commit(k_free(kb));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) (void)issue_pv(nt - 1);
      // every MMA issued has completed before TMEM is released
      tc_commit(drain_bar);
      (void)mbar_wait(drain_bar, 0u, timeout_ns, err);
    }
  } else if (warp >= kSoftWarp0) {
    // ---------------- softmax (one query row per thread) ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const float scale_log2 = 1.4426950408889634f / 16.0f;  // log2(e) / sqrt(head_dim)
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nt && ok; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full(b), (j >> 1) & 1u, timeout_ns, err));
      if (!ok) break;
      tc_fence_after();
      float s[kBKV];
      {
        uint32_t (&r)[kBKV] = reinterpret_cast<uint32_t (&)[kBKV]>(s);
        tmem_ld_32cols(lane_addr + kColS + b * kBKV, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld_32cols(lane_addr + kColS + b * kBKV + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(b));
      const int kbase = j * kBKV;
      if (kbase + kBKV > M) {  // the last tile may run past the keys
#pragma unroll
        for (int c = 0; c < kBKV; ++c)
          if (kbase + c >= M) s[c] = -INFINITY;
      }
      // row max as a tree (8 independent chains)
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
      for (int c = 8; c < kBKV; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
#pragma unroll
      for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) mx8[i] = fmaxf(mx8[i], mx8[i + w]);
      const float m_tile = mx8[0] * scale_log2;
      // rescale O when some row of the warp has a new max more than 2^8 above its old one
      const bool grow = m_tile > m + kRescaleThreshold;
      if (j == 0) {
        m = m_tile;
      } else if (__any_sync(0xFFFFFFFFu, grow)) {
        const float m_new = fmaxf(m, m_tile);
        const float alpha = fast_exp2(m - m_new);
        m = m_new;
        l *= alpha;
        // PV_{j-1} (written with the old max) must have landed in O first
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1u, timeout_ns, err));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < kHd / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_32cols(lane_addr + kColO + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32cols(lane_addr + kColO + cc * 32, o);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      // p = 2^(s * scale_log2 - m), bf16 into P buffer b (128-byte swizzled row `row`)
      float sum8[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
      uint32_t packed[kBKV / 2];
#pragma unroll
      for (int c = 0; c < kBKV; c += 2) {
        const float p0 = fast_exp2(fmaf(s[c], scale_log2, -m));
        const float p1 = fast_exp2(fmaf(s[c + 1], scale_log2, -m));
        sum8[(c >> 1) & 7] += p0 + p1;
        packed[c / 2] = pack_bf16x2(p0, p1);
      }
#pragma unroll
      for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) sum8[i] += sum8[i + w];
      l += sum8[0];
      // the MMAs that read P buffer b last (PV_{j-2}) have completed
      if (j >= 2) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(pv_done(b), ((j - 2) >> 1) & 1u, timeout_ns, err));
        if (!ok) break;
      }
      tmem_st_32cols(lane_addr + kColP + b * (kBKV / 2), packed);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(b));
    }
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(pv_done((nt - 1) & 1), ((nt - 1) >> 1) & 1u, timeout_ns, err));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const int qrow = q0 + row;
      __nv_bfloat16* orow = out + static_cast<int64_t>(qrow) * ldo + head * kHd;
#pragma unroll 1
      for (int cc = 0; cc < kHd / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_32cols(lane_addr + kColO + cc * 32, o);
        tmem_ld_wait();
        if (qrow < M) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// V^T of every head: vt[h * 256 + d, m] = qkv[m, 2 * hidden + h * 256 + d], through a 64 x 64
// shared-memory tile (rows of 128 bytes read and written).
__global__ void __launch_bounds__(256)
    transpose_v_kernel(const __nv_bfloat16* __restrict__ qkv, int64_t ld_qkv, int M, int hidden,
                       __nv_bfloat16* __restrict__ vt, int64_t ld_vt) {
  __shared__ uint32_t tile[64][33];  // [m][d / 2] bf16 pairs
  const int m0 = blockIdx.x * 64, d0 = blockIdx.y * 64;
  const int t = threadIdx.x;
  {
    const int r = t >> 2, c = (t & 3) * 16;  // row m0 + r, columns d0 + c .. + 16
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (m0 + r < M) {
      const __nv_bfloat16* src = qkv + static_cast<int64_t>(m0 + r) * ld_qkv + 2 * hidden + d0 + c;
      v0 = *reinterpret_cast<const uint4*>(src);
      v1 = *reinterpret_cast<const uint4*>(src + 8);
    }
    uint32_t* dst = &tile[r][c >> 1];
    dst[0] = v0.x; dst[1] = v0.y; dst[2] = v0.z; dst[3] = v0.w;
    dst[4] = v1.x; dst[5] = v1.y; dst[6] = v1.z; dst[7] = v1.w;
  }
  __syncthreads();
  {
    const int dr = t >> 2, c = (t & 3) * 16;  // output row d0 + dr, columns m0 + c .. + 16
    if (m0 + c >= M) return;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t a = tile[c + 2 * i][dr >> 1], b = tile[c + 2 * i + 1][dr >> 1];
      const uint32_t lo = (dr & 1) ? (a >> 16) : (a & 0xFFFFu);
      const uint32_t hi = (dr & 1) ? (b >> 16) : (b & 0xFFFFu);
      w[i] = lo | (hi << 16);
    }
    __nv_bfloat16* dst = vt + static_cast<int64_t>(d0 + dr) * ld_vt + m0 + c;
    if (m0 + c + 16 <= M) {
      reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      for (int i = 0; i < 16 && m0 + c + i < M; ++i)
        reinterpret_cast<uint16_t*>(dst)[i] = static_cast<uint16_t>((w[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu);
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// bf16 matrix [rows, cols] (row stride ld elements) in boxes of box_rows x 64, 128-byte swizzle.
bool encode_bf16_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t ld, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunk), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int64_t attention_vt_ld(int64_t M) { return (M + 7) / 8 * 8; }

nvfp4_status launch_attention(const void* qkv, int64_t M, int64_t ld_qkv, int heads, void* vt, void* out, int64_t ldo,
                              int* err, cudaStream_t s) {
  const int hidden = heads * kHd;
  const int64_t ld_vt = attention_vt_ld(M);
  {
    const dim3 grid(static_cast<unsigned>((M + 63) / 64), static_cast<unsigned>(hidden / 64));
    transpose_v_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(qkv), ld_qkv, static_cast<int>(M),
                                             hidden, static_cast<__nv_bfloat16*>(vt), ld_vt);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_LAUNCH;
  }
  CUtensorMap tm_q, tm_k, tm_vt;
  if (!encode_bf16_map(&tm_q, qkv, 3 * static_cast<int64_t>(hidden), M, ld_qkv, kBQ)) return NVFP4_ERR_LAUNCH;
  if (!encode_bf16_map(&tm_k, qkv, 3 * static_cast<int64_t>(hidden), M, ld_qkv, kBKV)) return NVFP4_ERR_LAUNCH;
  if (!encode_bf16_map(&tm_vt, vt, M, hidden, ld_vt, kHd)) return NVFP4_ERR_LAUNCH;
  static const cudaError_t ready =
      cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (ready != cudaSuccess) return NVFP4_ERR_LAUNCH;
  const dim3 grid(static_cast<unsigned>((M + kBQ - 1) / kBQ), static_cast<unsigned>(heads));
  attention_kernel<<<grid, kThreads, kSmemBytes, s>>>(tm_q, tm_k, tm_vt, static_cast<int>(M), hidden,
                                                      static_cast<__nv_bfloat16*>(out), ldo, err, wait_timeout_ns());
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_LAUNCH;
}

}  // namespace nvfp4
