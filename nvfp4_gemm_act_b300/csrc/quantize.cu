// bf16 -> NVFP4 quantization kernels for sm_103a: tensor amax, activation quantizer and the
// offline weight packer (transpose + optional gated pair interleave + quantize).
//
// Format (page "How fal made Ideogram V4 6x faster", NVFP4 paragraph): E2M1 codes, one
// unsigned E4M3 scale per 16 contiguous K-elements, fp32 tensor scale ts = amax / (6 * 448).
// Per block: s = E4M3(fp32(bamax / fp32(6 ts))); d = fp32(dec(s) ts); a block with
// d < 2^-126 is stored as scale 0 / codes +0; otherwise code = E2M1(fp32(x * fp32(1 / d))).
// All roundings are IEEE round-to-nearest-even in fp32 (explicit __fmul_rn / __fdiv_rn and
// the saturating cvt instructions), so codes and scales are reproducible bit for bit.

#include <cuda_bf16.h>

#include <algorithm>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr float kTsDivisor = 2688.0f;        // 6 (E2M1 max) * 448 (E4M3 max)

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 32 bytes in one 256-bit load (address 32-byte aligned).
__device__ __forceinline__ void ld_nc_v8(const void* p, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
               : "l"(p));
}

struct BlockScale {
  uint32_t code;  // E4M3 code actually stored (0 for a zero block)
  float inv;      // fp32(1 / fp32(dec(code) * ts)); unused for a zero block
  bool live;
};

__device__ __forceinline__ BlockScale block_scale(float bamax, float ts, float six_ts) {
  BlockScale r;
  if (!(ts > 0.0f)) {
    r.code = 0u;
    r.inv = 0.0f;
    r.live = false;
    return r;
  }
  const uint32_t code = cvt_e4m3(__fdiv_rn(bamax, six_ts));
  const float d = __fmul_rn(e4m3_to_f32(code), ts);
  r.live = d >= kFltMin;
  r.code = r.live ? code : 0u;
  r.inv = r.live ? __fdiv_rn(1.0f, d) : 0.0f;
  return r;
}

// ---------------------------------------------------------------------------------------
// amax: 128-bit loads, packed 16-bit max, warp reduce, one atomicMax per block.
// ---------------------------------------------------------------------------------------
constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 4;

template <bool kContiguous>
__global__ void __launch_bounds__(kAmaxThreads)
    amax_kernel(const uint4* __restrict__ x, uint32_t vec_per_row, uint64_t ld_vec,
                uint32_t total_vec, unsigned* __restrict__ amax_bits) {
  uint32_t m = 0;
  const uint32_t stride = gridDim.x * kAmaxThreads;
  uint32_t i = blockIdx.x * kAmaxThreads + threadIdx.x;
  for (; i + (kAmaxUnroll - 1) * stride < total_vec; i += kAmaxUnroll * stride) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      const uint32_t j = i + u * stride;
      const uint64_t off =
          kContiguous ? j : (uint64_t)(j / vec_per_row) * ld_vec + (j % vec_per_row);
      v[u] = ld_nc_v4(x + off);
    }
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      m = __vmaxu2(m, v[u].x & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].y & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].z & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].w & 0x7FFF7FFFu);
    }
  }
  for (; i < total_vec; i += stride) {
    const uint64_t off = kContiguous ? i : (uint64_t)(i / vec_per_row) * ld_vec + (i % vec_per_row);
    const uint4 v = ld_nc_v4(x + off);
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  }
  uint32_t mx = max(m & 0xFFFFu, m >> 16);
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  __shared__ uint32_t warp_max[kAmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < kAmaxThreads / 32 ? warp_max[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0 && v != 0u) atomicMax(amax_bits, v << 16);
  }
}

// ---------------------------------------------------------------------------------------
// Activation quantizer (after amax_kernel when the tensor scale is dynamic). Work item = one
// 512-element chunk of a row; lane l owns the 16-element block c * 32 + l (one 32-byte or
// two 16-byte loads), so a warp reads 1 KB of a row per item and writes 256 contiguous code
// bytes. Items are visited in reverse order (a grid-stride walk from the end of x), so the
// data the amax pass read last -- still in L2 -- is quantized first. Rows in [M, Mpad) only
// write their zero scale bytes.
//
// Per block, without a division in the common case:
//  * scale code s = E4M3(fp32(bamax / fp32(6 ts))): the quotient is approximated as
//    bamax * fp32(1 / (6 ts)) (within 2 ulp of the rounded quotient) and rounded to E4M3 at
//    both ends of a +-2^-20 relative window; when the two ends disagree the quotient is
//    within a few ulp of an E4M3 rounding boundary and the exact IEEE division decides, so
//    s always equals the code of the correctly rounded quotient;
//  * fp32(1 / d) with d = fp32(dec(s) ts) takes one of 127 values for the whole tensor: each
//    CTA tabulates them in shared memory (with the stored code, 0 for a zero block).
//
// Workspace words (zero between calls): ws[0] = amax bits (amax_kernel's atomic max),
// ws[1] = count of finished CTAs. Every CTA reads ws[0] before it counts itself finished;
// the last CTA to finish therefore knows all reads are done and zeroes both words.
// ---------------------------------------------------------------------------------------
constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;

template <bool kLoad32>  // one 32-byte load per lane (x 32-byte aligned, ldx % 16 == 0)
__global__ void __launch_bounds__(kQuantThreads, 4)
    quantize_kernel(const __nv_bfloat16* __restrict__ x, uint64_t ldx, uint32_t M,
                    uint32_t blocks_per_row, uint32_t chunks_per_row, uint32_t total_items,
                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, unsigned* ws,
                    const float* __restrict__ ts_in, float* __restrict__ ts_out) {
  __shared__ float inv_tab[128];     // fp32(1 / fp32(dec(s) ts)) per E4M3 code s (0: zero block)
  __shared__ uint32_t code_tab[128];  // code stored for s (0 for a zero block)
  const float ts = ts_in != nullptr
                       ? *ts_in
                       : __fdiv_rn(__uint_as_float(*reinterpret_cast<volatile unsigned*>(ws)), kTsDivisor);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;
  if (threadIdx.x < 128) build_scale_table_entry(threadIdx.x, ts, inv_tab, code_tab);
  const ScaleRoute sr = scale_route(ts);
  __syncthreads();

  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = (blockIdx.x * kQuantThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kQuantThreads) >> 5;
  const uint32_t gpr = blocks_per_row >> 2;
  const uint64_t row_code_bytes = (uint64_t)blocks_per_row * 8u;
  const uint32_t lane_sf = (lane >> 2) * 512u + (lane & 3u);  // this lane's byte in 8 scale atoms
  const int32_t cpr = static_cast<int32_t>(chunks_per_row);
  // slot u visits items total - 1 - (warp + u * nwarps + k * step), k = 0, 1, ...; its
  // (row, chunk) is stepped without a division
  const int32_t step = static_cast<int32_t>(nwarps * kQuantUnroll);
  const int32_t step_rows = step / cpr, step_chunks = step % cpr;
  int32_t row[kQuantUnroll], chunk[kQuantUnroll];
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const int32_t item = static_cast<int32_t>(total_items) - 1 - static_cast<int32_t>(warp + u * nwarps);
    row[u] = item >= 0 ? item / cpr : -1;
    chunk[u] = item >= 0 ? item % cpr : 0;
  }

  while (row[0] >= 0) {  // slot 0 holds the largest remaining item
    uint4 lo[kQuantUnroll], hi[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const uint32_t blk = static_cast<uint32_t>(chunk[u]) * 32u + lane;
      lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row[u] >= 0 && static_cast<uint32_t>(row[u]) < M && blk < blocks_per_row) {
        const __nv_bfloat16* src = x + static_cast<uint64_t>(row[u]) * ldx + blk * 16u;
        if (kLoad32) {
          ld_nc_v8(src, lo[u], hi[u]);
        } else {
          lo[u] = ld_nc_v4(src);
          hi[u] = ld_nc_v4(src + 8);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int32_t r = row[u];
      const uint32_t blk = static_cast<uint32_t>(chunk[u]) * 32u + lane;
      if (r >= 0 && blk < blocks_per_row) {
        const uint32_t ru = static_cast<uint32_t>(r);
        uint32_t stored = 0u;
        if (ru < M) {
          uint2 c;
          stored = quantize_block(lo[u], hi[u], sr, inv_tab, code_tab, c);
          if (NVFP4_INDEX_OK(blk < blocks_per_row &&
                             (uint64_t)ru * row_code_bytes + blk * 8u + 8u <= (uint64_t)M * row_code_bytes))
            *reinterpret_cast<uint2*>(codes + ru * row_code_bytes + blk * 8u) = c;
        }
        const uint64_t sidx = ((ru >> 7) * gpr + static_cast<uint32_t>(chunk[u]) * 8u) * 512u + (ru & 31u) * 16u +
                              ((ru >> 5) & 3u) * 4u + lane_sf;
        if (NVFP4_INDEX_OK(sidx < (uint64_t)((M + 127u) / 128u) * gpr * 512u && sidx == scale_offset(ru, blk, gpr)))
          scales[sidx] = static_cast<uint8_t>(stored);
      }
      chunk[u] -= step_chunks;
      row[u] -= step_rows;
      if (chunk[u] < 0) {
        chunk[u] += cpr;
        row[u] -= 1;
      }
    }
  }
  if (ts_in == nullptr) {
    __syncthreads();  // every thread of this CTA has read the amax word (long ago)
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(ws + 1, 1u) == gridDim.x - 1u) {  // last CTA: all CTAs have read it
        ws[0] = 0u;
        ws[1] = 0u;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Single-pass quantizer (a dynamic tensor scale only): one cooperative launch, one CTA per
// SM. CTA b reads rows [b R, b R + R) of x -- all 1024 threads, 16-byte loads in batches of
// six, so each SM keeps ~100 KB of x in flight (bulk copies from HBM keep far fewer bytes in
// flight per SM) -- taking the amax from the registers on the way and keeping its first S
// rows (S = R when they fit, else as many as 200 KB hold) in shared memory, and joins a
// grid-wide barrier on workspace words (bounded spin; the cooperative launch guarantees every
// CTA is resident). It then reads the tensor amax and quantizes its rows: the S resident rows
// from shared memory, the others from global memory again, last-read first (the part of them
// still in L2). When all rows are resident x is read from HBM once instead of twice; else
// the S rows are not read twice, and the amax pass needs no launch of its own.
//
// Workspace words: ws[0] amax bits (atomic max), ws[1] CTAs arrived, ws[2] CTAs departed,
// ws[3] failure flag. The CTA that departs last has seen every CTA pass the barrier and zeroes
// all four. A wait that runs out of time marks the failure: every CTA then writes no codes and
// the tensor scale written is NaN.
// ---------------------------------------------------------------------------------------
constexpr int kFusedThreads = 1024;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedSmemData = 200 * 1024;      // bytes of x per CTA held in shared memory
constexpr int kFusedBatch = 6;                  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kFusedThreads, 1)
    quantize_fused_kernel(const __nv_bfloat16* __restrict__ x, uint64_t ldx, uint32_t M, uint32_t Mpad,
                          uint32_t K, uint32_t rows_per_cta, uint32_t res_rows, uint8_t* __restrict__ codes,
                          uint8_t* __restrict__ scales, unsigned* ws, float* __restrict__ ts_out,
                          uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t xs[];  // the first res_rows rows of x, K * 2 bytes each
  __shared__ float inv_tab[128];
  __shared__ uint32_t code_tab[128];
  __shared__ uint32_t warp_max[kFusedWarps];
  __shared__ float ts_s;
  __shared__ int failed;

  const uint32_t r0 = blockIdx.x * rows_per_cta;
  const uint32_t r_end = min(Mpad, r0 + rows_per_cta);  // rows [r0, r_end), padding included
  const uint32_t n_real = min(M, r_end) > r0 ? min(M, r_end) - r0 : 0u;  // rows holding data
  const uint32_t row_bytes = K * 2u;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) failed = 0;
  // 16-byte chunk c of the CTA's rows: row c / vpr, column chunk c % vpr; in shared memory
  // the rows are contiguous, so chunk c sits at byte 16 c
  const uint32_t vpr = K / 8u;
  const uint32_t nchunks = n_real * vpr;
  const uint32_t res_chunks = min(n_real, res_rows) * vpr;  // chunks of the resident rows
  uint32_t m = 0u;
  for (uint32_t c0 = threadIdx.x; c0 < nchunks; c0 += kFusedBatch * kFusedThreads) {
    uint4 v[kFusedBatch];
#pragma unroll
    for (int j = 0; j < kFusedBatch; ++j) {
      const uint32_t c = c0 + j * kFusedThreads;
      v[j] = make_uint4(0u, 0u, 0u, 0u);
      if (c < nchunks) {
        const uint32_t r = c / vpr;
        v[j] = ld_nc_v4(x + (uint64_t)(r0 + r) * ldx + (c - r * vpr) * 8u);
      }
    }
#pragma unroll
    for (int j = 0; j < kFusedBatch; ++j) {
      const uint32_t c = c0 + j * kFusedThreads;
      if (c < nchunks) {
        m = bf16x2_max_abs(m, bf16x2_max_abs(bf16x2_max_abs(v[j].x, v[j].y), bf16x2_max_abs(v[j].z, v[j].w)));
        if (c < res_chunks) reinterpret_cast<uint4*>(xs)[c] = v[j];
      }
    }
  }
  uint32_t h = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
  h = __reduce_max_sync(0xFFFFFFFFu, h);
  if (lane == 0) warp_max[warp] = h;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t cm = 0u;
    for (int w = 0; w < kFusedWarps; ++w) cm = max(cm, warp_max[w]);
    // publish the amax (and a failure), then arrive; the release orders them before it
    if (cm != 0u) red_max_relaxed_gpu(ws, cm << 16);
    if (failed) red_or_relaxed_gpu(ws + 3, 1u);
    red_add_release_gpu(ws + 1, 1u);
    // grid barrier: every CTA has published its amax
    const uint64_t t0 = global_timer_ns();
    bool all_in = false;
    while (!(all_in = ld_acquire_gpu(ws + 1) >= gridDim.x)) {
      if (global_timer_ns() - t0 > timeout_ns) break;
    }
    // (the acquire loads order the reads below after every CTA's release)
    const bool bad = !all_in || ld_acquire_gpu(ws + 3) != 0u;
    const uint32_t amax_bits = ld_acquire_gpu(ws);
    failed = bad ? 1 : 0;
    ts_s = bad ? __int_as_float(0x7FC00000) : __fdiv_rn(__uint_as_float(amax_bits), kTsDivisor);
  }
  __syncthreads();
  const float ts = ts_s;
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;
  if (!failed) {
    if (threadIdx.x < 128) build_scale_table_entry(threadIdx.x, ts, inv_tab, code_tab);
    const ScaleRoute sr = scale_route(ts);
    __syncthreads();
    // quantize: item = (row, 512-element chunk) -- last item first when some rows are read
    // again (the rows read last are the ones most likely still in L2) --; lane = one
    // 16-element block of the chunk; a warp takes two items at a time
    const uint32_t bpr = K / 16u, cpr = (bpr + 31u) / 32u, gpr = bpr >> 2;
    const uint32_t items = (r_end - r0) * cpr;
    const uint64_t row_code_bytes = (uint64_t)bpr * 8u;
    for (uint32_t it0 = warp; it0 < items; it0 += 2 * kFusedWarps) {
      uint4 lo[2], hi[2];
      uint32_t rr[2], bb[2];
      bool data[2], valid[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t idx = it0 + u * kFusedWarps;
        const uint32_t it = idx < items ? (res_rows < r_end - r0 ? items - 1u - idx : idx) : 0u;
        const uint32_t i = it / cpr;
        bb[u] = (it - i * cpr) * 32u + lane;
        rr[u] = r0 + i;
        valid[u] = idx < items && bb[u] < bpr;
        data[u] = valid[u] && i < n_real;
        lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
        if (data[u]) {
          if (i < res_rows) {
            if (NVFP4_INDEX_OK(i * row_bytes + bb[u] * 32u + 32u <= res_rows * row_bytes)) {
              const uint4* src = reinterpret_cast<const uint4*>(xs + i * row_bytes + bb[u] * 32u);
              lo[u] = src[0];
              hi[u] = src[1];
            }
          } else if (NVFP4_INDEX_OK(rr[u] < M && bb[u] < bpr)) {
            const __nv_bfloat16* g = x + (uint64_t)rr[u] * ldx + bb[u] * 16u;
            lo[u] = ld_nc_v4(g);
            hi[u] = ld_nc_v4(g + 8);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (!valid[u]) continue;
        uint32_t stored = 0u;
        if (data[u]) {
          uint2 c;
          stored = quantize_block(lo[u], hi[u], sr, inv_tab, code_tab, c);
          if (NVFP4_INDEX_OK(rr[u] < M && bb[u] < bpr))
            *reinterpret_cast<uint2*>(codes + rr[u] * row_code_bytes + bb[u] * 8u) = c;
        }
        if (NVFP4_INDEX_OK(rr[u] < Mpad && bb[u] < bpr))
          scales[scale_offset(rr[u], bb[u], gpr)] = static_cast<uint8_t>(stored);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // every CTA that departs has passed the grid barrier and read the words; the last one
    // to depart resets them for the next call
    if (atomicAdd(ws + 2, 1u) == gridDim.x - 1u) {
      ws[0] = 0u;
      ws[1] = 0u;
      ws[2] = 0u;
      ws[3] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------------------
// Weight packer: a CTA transposes a 64 (k) x 64 (n) tile of W through shared memory; each
// thread then quantizes one 16-element K-block of one column into packed row p(n).
// ---------------------------------------------------------------------------------------
template <bool kGated>
__global__ void __launch_bounds__(256)
    pack_weights_kernel(const __nv_bfloat16* __restrict__ w, uint32_t K, uint32_t N,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                        const unsigned* __restrict__ amax_bits, float* __restrict__ ts_out) {
  __shared__ uint32_t tile[64][33];  // [k][n/2] bf16 pairs, padded against bank conflicts
  const float ts = __fdiv_rn(__uint_as_float(*amax_bits), kTsDivisor);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ts_out = ts;
  const float six_ts = __fmul_rn(6.0f, ts);
  const uint32_t n0 = blockIdx.x * 64u, k0 = blockIdx.y * 64u;
  const uint32_t t = threadIdx.x;
  // load: thread t reads row k0 + t/4, columns n0 + (t%4)*16 .. +16 (two 16-byte vectors)
  {
    const uint32_t kr = t >> 2, c = (t & 3u) * 16u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t n = n0 + c + h * 8u;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < N) v = ld_nc_v4(w + (uint64_t)(k0 + kr) * N + n);
      uint32_t* dst = &tile[kr][(c + h * 8u) >> 1];
      dst[0] = v.x;
      dst[1] = v.y;
      dst[2] = v.z;
      dst[3] = v.w;
    }
  }
  __syncthreads();
  const uint32_t nl = t & 63u, b = t >> 6;  // column in tile, 16-row block in tile
  const uint32_t n = n0 + nl;
  if (n >= N) return;
  float vals[16];
  float bamax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = tile[b * 16u + i][nl >> 1];
    vals[i] = (nl & 1u) ? bf16_hi(word) : bf16_lo(word);
    bamax = fmaxf(bamax, fabsf(vals[i]));
  }
  const BlockScale bs = block_scale(bamax, ts, six_ts);
  uint32_t lo = 0u, hi = 0u;
  if (bs.live) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= cvt_e2m1x2(__fmul_rn(vals[2 * i], bs.inv), __fmul_rn(vals[2 * i + 1], bs.inv)) << (8 * i);
      hi |= cvt_e2m1x2(__fmul_rn(vals[8 + 2 * i], bs.inv), __fmul_rn(vals[9 + 2 * i], bs.inv))
            << (8 * i);
    }
  }
  const uint32_t half = N >> 1;
  const uint32_t p = kGated ? (n < half ? 2u * n : 2u * (n - half) + 1u) : n;
  const uint32_t kb = (k0 >> 4) + b;
  if (!NVFP4_INDEX_OK(p < N && kb < (K >> 4))) return;
  *reinterpret_cast<uint2*>(codes + (uint64_t)p * (K >> 1) + (kb << 3)) = make_uint2(lo, hi);
  const uint32_t gpr = K >> 6;
  scales[((p >> 7) * gpr + (kb >> 2)) * 512u + (p & 31u) * 16u + ((p >> 5) & 3u) * 4u + (kb & 3u)] =
      static_cast<uint8_t>(bs.code);
}

// ---------------------------------------------------------------------------------------
// FP8 (E4M3) with one scale per tensor: ts = amax / 448, code = E4M3(fp32(x * fp32(1 / ts))),
// nearest even, saturating at +-448, sign kept; a tensor with ts < 2^-126 is stored as +0.
// ---------------------------------------------------------------------------------------
constexpr float kFp8TsDivisor = 448.0f;
constexpr int kFp8Threads = 256;

// 16 values -> 16 E4M3 codes, element i in byte i.
__device__ __forceinline__ uint4 encode_e4m3x16(const float (&v)[16], float inv) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = cvt_e4m3x2(__fmul_rn(v[4 * i], inv), __fmul_rn(v[4 * i + 1], inv)) |
           (cvt_e4m3x2(__fmul_rn(v[4 * i + 2], inv), __fmul_rn(v[4 * i + 3], inv)) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Activation quantizer: item = 16 consecutive elements of a row (32 bytes in, 16 bytes out),
// grid-stride. Workspace words as for quantize_kernel: ws[0] = amax bits (from amax_kernel),
// ws[1] = CTAs finished; the last CTA to finish zeroes both (dynamic scale only).
__global__ void __launch_bounds__(kFp8Threads)
    fp8_quantize_kernel(const __nv_bfloat16* __restrict__ x, uint64_t ldx, uint32_t M, uint32_t items_per_row,
                        uint8_t* __restrict__ codes, unsigned* __restrict__ ws, const float* __restrict__ ts_in,
                        float* __restrict__ ts_out) {
  const float ts = ts_in != nullptr ? __ldg(ts_in)
                                    : __fdiv_rn(__uint_as_float(*reinterpret_cast<volatile unsigned*>(ws)),
                                                kFp8TsDivisor);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;
  const bool live = ts >= kFltMin;
  const float inv = live ? __frcp_rn(ts) : 0.0f;
  const uint64_t total = static_cast<uint64_t>(M) * items_per_row;
  const uint64_t K = static_cast<uint64_t>(items_per_row) * 16u;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kFp8Threads + threadIdx.x; i < total;
       i += static_cast<uint64_t>(gridDim.x) * kFp8Threads) {
    const uint64_t r = i / items_per_row, c = (i - r * items_per_row) * 16u;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (live) {
      const __nv_bfloat16* src = x + r * ldx + c;
      const uint4 lo = ld_nc_v4(src), hi = ld_nc_v4(src + 8);
      const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[2 * j] = bf16_lo(wv[j]);
        v[2 * j + 1] = bf16_hi(wv[j]);
      }
      out = encode_e4m3x16(v, inv);
    }
    if (NVFP4_INDEX_OK(r < M && c + 16u <= K)) *reinterpret_cast<uint4*>(codes + r * K + c) = out;
  }
  if (ts_in == nullptr) {
    __syncthreads();  // every thread of this CTA has read the amax word
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(ws + 1, 1u) == gridDim.x - 1u) {
        ws[0] = 0u;
        ws[1] = 0u;
      }
    }
  }
}

// Weight packer: a CTA transposes a 64 (k) x 64 (n) tile of W through shared memory; each
// thread then encodes 16 consecutive K-elements of one column into packed row p(n).
template <bool kGated>
__global__ void __launch_bounds__(256)
    fp8_pack_weights_kernel(const __nv_bfloat16* __restrict__ w, uint32_t K, uint32_t N, uint8_t* __restrict__ codes,
                            const unsigned* __restrict__ amax_bits, float* __restrict__ ts_out) {
  __shared__ uint32_t tile[64][33];  // [k][n/2] bf16 pairs, padded against bank conflicts
  const float ts = __fdiv_rn(__uint_as_float(*amax_bits), kFp8TsDivisor);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ts_out = ts;
  const bool live = ts >= kFltMin;
  const float inv = live ? __frcp_rn(ts) : 0.0f;
  const uint32_t n0 = blockIdx.x * 64u, k0 = blockIdx.y * 64u;
  const uint32_t t = threadIdx.x;
  {
    const uint32_t kr = t >> 2, c = (t & 3u) * 16u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t n = n0 + c + h * 8u;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < N) v = ld_nc_v4(w + (uint64_t)(k0 + kr) * N + n);
      uint32_t* dst = &tile[kr][(c + h * 8u) >> 1];
      dst[0] = v.x;
      dst[1] = v.y;
      dst[2] = v.z;
      dst[3] = v.w;
    }
  }
  __syncthreads();
  const uint32_t nl = t & 63u, b = t >> 6;  // column in tile, 16-row block in tile
  const uint32_t n = n0 + nl;
  if (n >= N) return;
  float vals[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = tile[b * 16u + i][nl >> 1];
    vals[i] = (nl & 1u) ? bf16_hi(word) : bf16_lo(word);
  }
  const uint4 out = live ? encode_e4m3x16(vals, inv) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t half = N >> 1;
  const uint32_t p = kGated ? (n < half ? 2u * n : 2u * (n - half) + 1u) : n;
  if (NVFP4_INDEX_OK(p < N && k0 + b * 16u + 16u <= K)) *reinterpret_cast<uint4*>(codes + (uint64_t)p * K + k0 + b * 16u) = out;
}

__global__ void wait_timeout_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait runs out, records the time-out, returns.
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0u, limit_ns, err);
}

}  // namespace

cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                        unsigned* amax_bits, cudaStream_t s) {
  const uint32_t vpr = static_cast<uint32_t>(cols / 8);
  const uint32_t total = static_cast<uint32_t>(rows * (cols / 8));
  if (total == 0) return cudaSuccess;
  static const int per_sm = resident_blocks((const void*)amax_kernel<true>, kAmaxThreads, 0);
  const uint32_t want = (total + kAmaxThreads * kAmaxUnroll - 1) / (kAmaxThreads * kAmaxUnroll);
  const uint32_t grid = std::min<uint32_t>(want, (uint32_t)(sm_count() * per_sm));
  if (ld == cols)
    amax_kernel<true><<<grid, kAmaxThreads, 0, s>>>(static_cast<const uint4*>(x), vpr, ld / 8,
                                                    total, amax_bits);
  else
    amax_kernel<false><<<grid, kAmaxThreads, 0, s>>>(static_cast<const uint4*>(x), vpr, ld / 8,
                                                     total, amax_bits);
  return cudaGetLastError();
}

namespace {

// Rows per CTA of the single-pass quantizer for x [M, K] and how many of them stay in shared
// memory ({0, 0}: x rows not 16-byte aligned, a row larger than the shared-memory budget, or
// fewer than a quarter of each CTA's rows resident, where the two-pass path is the better one).
struct FusedPlan {
  uint32_t rows;
  uint32_t res_rows;
};

FusedPlan fused_plan(const void* x, int64_t M, int64_t K, int64_t ldx) {
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || (ldx * 2) % 16 != 0) return {0, 0};
  static const int per_sm = [] {
    int n = 0;
    if (cudaFuncSetAttribute(quantize_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFusedSmemData) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_fused_kernel, kFusedThreads, kFusedSmemData) !=
            cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    return n;
  }();
  if (per_sm < 1) return {0, 0};
  const int64_t mpad = (M + 127) / 128 * 128;
  const int64_t ctas = static_cast<int64_t>(sm_count()) * per_sm;
  const int64_t rows = (mpad + ctas - 1) / ctas;
  const int64_t res = std::min<int64_t>(rows, kFusedSmemData / (K * 2));
  if (res < 1 || res * 4 < rows) return {0, 0};
  return {static_cast<uint32_t>(rows), static_cast<uint32_t>(res)};
}

}  // namespace

cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, unsigned* ws, const float* ts_in, float* ts_out,
                            cudaStream_t s) {
  if (ts_in == nullptr && M > 0) {
    if (const FusedPlan plan = fused_plan(x, M, K, ldx); plan.rows != 0) {
      const int64_t mpad = (M + 127) / 128 * 128;
      const unsigned grid = static_cast<unsigned>((mpad + plan.rows - 1) / plan.rows);
      const __nv_bfloat16* xp = static_cast<const __nv_bfloat16*>(x);
      uint64_t ld = static_cast<uint64_t>(ldx);
      uint32_t m = static_cast<uint32_t>(M), mp = static_cast<uint32_t>(mpad), k = static_cast<uint32_t>(K);
      uint32_t r = plan.rows, rr = plan.res_rows;
      uint64_t limit = wait_timeout_ns();
      void* args[] = {&xp, &ld, &m, &mp, &k, &r, &rr, &codes, &scales, &ws, &ts_out, &limit};
      return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(quantize_fused_kernel), dim3(grid),
                                         dim3(kFusedThreads), args, static_cast<size_t>(plan.res_rows) * K * 2,
                                         s);
    }
  }
  if (ts_in == nullptr) {
    const cudaError_t e = launch_amax(x, M, K, ldx, ws, s);
    if (e != cudaSuccess) return e;
  }
  const uint32_t bpr = static_cast<uint32_t>(K / 16);
  const uint32_t cpr = (bpr + 31u) / 32u;
  const int64_t mpad = (M + 127) / 128 * 128;
  const uint32_t total = static_cast<uint32_t>(mpad * cpr);
  static const int per_sm = resident_blocks((const void*)quantize_kernel<true>, kQuantThreads, 0);
  const uint32_t items_per_block = (kQuantThreads / 32) * kQuantUnroll;
  const uint32_t want = (total + items_per_block - 1) / items_per_block;
  const uint32_t grid = std::max<uint32_t>(1u, std::min<uint32_t>(want, (uint32_t)(sm_count() * per_sm)));
  const bool load32 = (reinterpret_cast<uintptr_t>(x) & 31u) == 0 && ldx % 16 == 0;
  auto kern = load32 ? quantize_kernel<true> : quantize_kernel<false>;
  kern<<<grid, kQuantThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), static_cast<uint64_t>(ldx),
                                      static_cast<uint32_t>(M), bpr, cpr, total, codes, scales, ws, ts_in,
                                      ts_out);
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const void* w, int64_t K, int64_t N, bool gated,
                                uint8_t* codes, uint8_t* scales, const unsigned* amax_bits,
                                float* ts_out, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((N + 63) / 64), static_cast<unsigned>(K / 64));
  if (gated)
    pack_weights_kernel<true><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w),
                                                   (uint32_t)K, (uint32_t)N, codes, scales,
                                                   amax_bits, ts_out);
  else
    pack_weights_kernel<false><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w),
                                                    (uint32_t)K, (uint32_t)N, codes, scales,
                                                    amax_bits, ts_out);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes, unsigned* ws,
                               const float* ts_in, float* ts_out, cudaStream_t s) {
  if (ts_in == nullptr) {
    const cudaError_t e = launch_amax(x, M, K, ldx, ws, s);
    if (e != cudaSuccess) return e;
  }
  const uint32_t per_row = static_cast<uint32_t>(K / 16);
  const uint64_t total = static_cast<uint64_t>(M) * per_row;
  static const int per_sm = resident_blocks((const void*)fp8_quantize_kernel, kFp8Threads, 0);
  const uint64_t want = (total + kFp8Threads - 1) / kFp8Threads;
  const uint32_t grid = static_cast<uint32_t>(
      std::max<uint64_t>(1u, std::min<uint64_t>(want, static_cast<uint64_t>(sm_count()) * per_sm)));
  fp8_quantize_kernel<<<grid, kFp8Threads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), static_cast<uint64_t>(ldx),
                                                   static_cast<uint32_t>(M), per_row, codes, ws, ts_in, ts_out);
  return cudaGetLastError();
}

cudaError_t launch_fp8_pack_weights(const void* w, int64_t K, int64_t N, bool gated, uint8_t* codes,
                                    const unsigned* amax_bits, float* ts_out, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((N + 63) / 64), static_cast<unsigned>(K / 64));
  const __nv_bfloat16* wp = static_cast<const __nv_bfloat16*>(w);
  if (gated)
    fp8_pack_weights_kernel<true><<<grid, 256, 0, s>>>(wp, (uint32_t)K, (uint32_t)N, codes, amax_bits, ts_out);
  else
    fp8_pack_weights_kernel<false><<<grid, 256, 0, s>>>(wp, (uint32_t)K, (uint32_t)N, codes, amax_bits, ts_out);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}


// Failed index checks counted by this file's kernels since the last call (debug builds; always
// 0 otherwise); reading clears the counter. Call with the device idle.
cudaError_t take_index_failures_quantize(unsigned* n) {
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
