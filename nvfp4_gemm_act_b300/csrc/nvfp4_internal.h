// Internal host-side interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Default bound on any single device-side wait (2 s); NVFP4_WAIT_TIMEOUT_NS overrides it.
uint64_t wait_timeout_ns();

// Blocks per SM the kernel can keep resident with `threads` threads and `smem` dynamic bytes.
int resident_blocks(const void* kernel, int threads, size_t smem);
int sm_count();

// amax(|x|) of bf16 x [rows, cols] (row stride ld) into *amax_bits (fp32 bit pattern,
// atomic max; the caller zeroes it first).
cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                        unsigned* amax_bits, cudaStream_t s);

// Host checks of nvfp4_quantize, in order: shapes (then M == 0 returns NVFP4_OK), NULL
// pointers, alignment, the device, and that every pointer is memory of the current device.
// `library_scratch`: the workspace is the library's own array (no NULL check on it).
nvfp4_status check_quantize_args(const void* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* codes,
                                 const uint8_t* scales, const float* tensor_scale, const float* tensor_scale_in,
                                 const void* workspace, bool library_scratch);

// Quantize x [M, K] (row stride ldx). ts = *ts_in if ts_in, else amax/2688 of x: either one
// cooperative single-pass launch (x fits in the SMs' shared memory) or amax_kernel reducing
// into ws[0] and the quantize kernel reading it; both leave ws[0..3] zeroed again.
cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, unsigned* ws, const float* ts_in, float* ts_out,
                            cudaStream_t s);

// W [K, N] -> packed K-major codes [N, K/2] + tiled scales (scales pre-zeroed by caller).
cudaError_t launch_pack_weights(const void* w, int64_t K, int64_t N, bool gated,
                                uint8_t* codes, uint8_t* scales, const unsigned* amax_bits,
                                float* ts_out, cudaStream_t s);

// FP8 (E4M3, one scale per tensor): x [M, K] (row stride ldx) -> codes [M, K]; ts = *ts_in if
// ts_in, else amax/448 of x (amax_kernel into ws[0], which the quantize kernel zeroes again).
cudaError_t launch_fp8_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes, unsigned* ws,
                               const float* ts_in, float* ts_out, cudaStream_t s);

// W [K, N] -> E4M3 codes [N, K] (K-major, packed column order if gated), ts = amax/448.
cudaError_t launch_fp8_pack_weights(const void* w, int64_t K, int64_t N, bool gated, uint8_t* codes,
                                    const unsigned* amax_bits, float* ts_out, cudaStream_t s);

struct GemmArgs {
  const uint8_t* a_codes;
  const uint8_t* a_scales;
  const float* a_ts;
  const uint8_t* b_codes;
  const uint8_t* b_scales;
  const float* b_ts;
  int64_t M, N, K;
  int epi;
  const float* bias;
  const float* gamma;
  int head_dim;
  int64_t norm_cols;
  float eps;
  int out_fp32;
  void* out;
  int64_t ldo;
  int* err;
  // NVFP4 output instead of `out` (codes [M, out_cols/2], tiled scales, static tensor scale)
  int out_nvfp4 = 0;
  uint8_t* out_codes = nullptr;
  uint8_t* out_scales = nullptr;
  const float* out_ts = nullptr;
  // operands: 0 = NVFP4 (codes [rows, K/2] + tiled block scales), 1 = FP8 E4M3 (codes
  // [rows, K], no block scales; a_scales / b_scales unused)
  int fp8 = 0;
};

// Validated arguments in, kernel launched (or an error code out).
nvfp4_status launch_gemm(const GemmArgs& a, cudaStream_t s);

// Row stride (elements) of the V^T workspace [heads * 256, attention_vt_ld(M)] bf16.
int64_t attention_vt_ld(int64_t M);

// Attention over qkv [M, 3 * heads * 256] (Q | K | V, heads contiguous in each, row stride
// ld_qkv) -> out [M, heads * 256] (row stride ldo): V^T into `vt`, then the attention kernel.
nvfp4_status launch_attention(const void* qkv, int64_t M, int64_t ld_qkv, int heads, void* vt, void* out,
                              int64_t ldo, int* err, cudaStream_t s);

cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t s);

// Failed index checks of the quantize / GEMM kernels since the last call (debug builds), cleared.
cudaError_t take_index_failures_quantize(unsigned* n);
cudaError_t take_index_failures_gemm(unsigned* n);

// Validated arguments of nvfp4_debug_mma_rate in, the probe kernel launched.
nvfp4_status launch_mma_probe(int kind, int cta_group, int n, int iters, int ctas, long long* out, int* err,
                              cudaStream_t s);

}  // namespace nvfp4
