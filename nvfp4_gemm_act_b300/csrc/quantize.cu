// bf16 -> NVFP4 quantization kernels for sm_103a: tensor amax, activation quantizer and the
// offline weight packer (transpose + optional gated pair interleave + quantize).
//
// Format (page "How fal made Ideogram V4 6x faster", NVFP4 paragraph): E2M1 codes, one
// unsigned E4M3 scale per 16 contiguous K-elements, fp32 tensor scale ts = amax / (6 * 448).
// Per block: s = E4M3(bamax / fp32(6 ts)); d = fp32(dec(s) ts); a block with d < 2^-126 is
// stored as scale 0 / codes +0; otherwise code = E2M1(fp32(x * fp32(1 / d))).
// All roundings are IEEE round-to-nearest-even in fp32 (explicit __fmul_rn / __fdiv_rn and
// the saturating cvt instructions), so codes and scales are reproducible bit for bit.

#include <cuda_bf16.h>

#include <algorithm>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr float kTsDivisor = 2688.0f;        // 6 (E2M1 max) * 448 (E4M3 max)
constexpr float kFltMin = 1.17549435082e-38f;  // 2^-126

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

// |bf16| maximum of the 8 values in v, as the fp32 value (exact).
__device__ __forceinline__ float absmax8(const uint4& v) {
  uint32_t m = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  const uint32_t hi = max(m & 0xFFFFu, m >> 16);
  return __uint_as_float(hi << 16);
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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 8 bf16 values (in memory order) -> 4 bytes of E2M1 codes, element 2j in the low nibble.
__device__ __forceinline__ uint32_t encode8(const uint4& v, float inv) {
  const uint32_t b0 = cvt_e2m1x2(__fmul_rn(bf16_lo(v.x), inv), __fmul_rn(bf16_hi(v.x), inv));
  const uint32_t b1 = cvt_e2m1x2(__fmul_rn(bf16_lo(v.y), inv), __fmul_rn(bf16_hi(v.y), inv));
  const uint32_t b2 = cvt_e2m1x2(__fmul_rn(bf16_lo(v.z), inv), __fmul_rn(bf16_hi(v.z), inv));
  const uint32_t b3 = cvt_e2m1x2(__fmul_rn(bf16_lo(v.w), inv), __fmul_rn(bf16_hi(v.w), inv));
  return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
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
// 512-element chunk of a row; lane l owns the 16-element block c * 32 + l (two 16-byte
// loads), so a warp reads 1 KB of a row per item and writes 256 contiguous code bytes.
// Items are visited in reverse order (a grid-stride walk from the end of x), so the data
// the amax pass read last -- still in L2 -- is quantized first. Rows in [M, Mpad) only
// write their zero scale bytes.
//
// Workspace words (zero between calls): ws[0] = amax bits (amax_kernel's atomic max),
// ws[1] = count of finished CTAs. Every CTA reads ws[0] before it counts itself finished;
// the last CTA to finish therefore knows all reads are done and zeroes both words.
// ---------------------------------------------------------------------------------------
constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;

struct QuantItem {
  uint32_t row, blk;
  bool live, real;
};

__device__ __forceinline__ QuantItem quant_item(uint32_t item, uint32_t lane, uint32_t M,
                                                uint32_t blocks_per_row, uint32_t chunks_per_row) {
  QuantItem q;
  q.row = item / chunks_per_row;
  q.blk = (item - q.row * chunks_per_row) * 32u + lane;
  q.live = q.blk < blocks_per_row;
  q.real = q.live && q.row < M;
  return q;
}

template <bool kLoad32>  // one 32-byte load per lane (x 32-byte aligned, ldx % 16 == 0)
__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(const __nv_bfloat16* __restrict__ x, uint64_t ldx, uint32_t M,
                    uint32_t blocks_per_row, uint32_t chunks_per_row, uint32_t total_items,
                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, unsigned* ws,
                    const float* __restrict__ ts_in, float* __restrict__ ts_out) {
  float ts;
  if (ts_in != nullptr) {
    ts = *ts_in;
  } else {
    ts = __fdiv_rn(__uint_as_float(*reinterpret_cast<volatile unsigned*>(ws)), kTsDivisor);
    __syncthreads();  // every thread of this CTA has read the amax word
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(ws + 1, 1u) == gridDim.x - 1u) {  // last CTA: all CTAs have read it
        ws[0] = 0u;
        ws[1] = 0u;
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;
  const float six_ts = __fmul_rn(6.0f, ts);
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = (blockIdx.x * kQuantThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kQuantThreads) >> 5;
  const uint32_t gpr = blocks_per_row >> 2;
  const uint64_t row_code_bytes = (uint64_t)blocks_per_row * 8u;

  for (uint32_t base = warp; base < total_items; base += nwarps * kQuantUnroll) {
    uint4 lo[kQuantUnroll], hi[kQuantUnroll];
    QuantItem q[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const uint32_t i = base + u * nwarps;
      const bool in = i < total_items;
      q[u] = quant_item(in ? total_items - 1u - i : 0u, lane, M, blocks_per_row, chunks_per_row);
      q[u].live = q[u].live && in;
      q[u].real = q[u].real && in;
      lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
      if (q[u].real) {
        const __nv_bfloat16* src = x + q[u].row * ldx + q[u].blk * 16u;
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
      if (!q[u].live) continue;
      uint32_t scale = 0u;
      if (q[u].real) {
        const BlockScale bs = block_scale(fmaxf(absmax8(lo[u]), absmax8(hi[u])), ts, six_ts);
        uint2 c = make_uint2(0u, 0u);
        if (bs.live) c = make_uint2(encode8(lo[u], bs.inv), encode8(hi[u], bs.inv));
        *reinterpret_cast<uint2*>(codes + q[u].row * row_code_bytes + q[u].blk * 8u) = c;
        scale = bs.code;
      }
      const uint32_t r = q[u].row, b = q[u].blk;
      scales[((r >> 7) * gpr + (b >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u + (b & 3u)] =
          static_cast<uint8_t>(scale);
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
  *reinterpret_cast<uint2*>(codes + (uint64_t)p * (K >> 1) + (kb << 3)) = make_uint2(lo, hi);
  const uint32_t gpr = K >> 6;
  scales[((p >> 7) * gpr + (kb >> 2)) * 512u + (p & 31u) * 16u + ((p >> 5) & 3u) * 4u + (kb & 3u)] =
      static_cast<uint8_t>(bs.code);
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

cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, unsigned* ws, const float* ts_in, float* ts_out,
                            cudaStream_t s) {
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

cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace nvfp4
