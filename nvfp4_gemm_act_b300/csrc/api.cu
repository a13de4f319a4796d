// C ABI of the fused NVFP4 linear layer (declared in include/nvfp4.h): argument checks,
// device check, and dispatch to the kernels. Every check runs before anything is launched.

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <initializer_list>
#include <mutex>

#include "../../include/nvfp4.h"
#include "nvfp4_internal.h"
#include "pointer_check.h"

namespace nvfp4 {

uint64_t wait_timeout_ns() {
  static const uint64_t v = [] {
    const char* s = std::getenv("NVFP4_WAIT_TIMEOUT_NS");
    if (s != nullptr) {
      const unsigned long long t = std::strtoull(s, nullptr, 10);
      if (t > 0) return static_cast<uint64_t>(t);
    }
    return static_cast<uint64_t>(2000000000ull);
  }();
  return v;
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int resident_blocks(const void* kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n <= 0) n = 1;
  return n;
}

}  // namespace nvfp4

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 34;  // M * K bound of the 32-bit work indices

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device must be compute capability 10.3 (B300). Cached per device.
nvfp4_status check_device() {
  static std::atomic<int> state[64];  // 0 unknown, 1 ok, 2 bad
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    (void)cudaGetLastError();
    return NVFP4_ERR_DEVICE;
  }
  if (dev < 64) {
    const int st = state[dev].load(std::memory_order_relaxed);
    if (st == 1) return NVFP4_OK;
    if (st == 2) return NVFP4_ERR_DEVICE;
  }
  int major = 0, minor = 0;
  bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
            major == 10 && minor == 3;
  if (!ok) (void)cudaGetLastError();
  if (dev < 64) state[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? NVFP4_OK : NVFP4_ERR_DEVICE;
}

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_LAUNCH; }

// Every non-NULL pointer of the list names memory of the current device (classify_pointer);
// runs after check_device, before anything is launched.
nvfp4_status check_pointers(std::initializer_list<const void*> ptrs) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return NVFP4_ERR_DEVICE;
  }
  for (const void* p : ptrs) {
    if (p == nullptr) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      (void)cudaGetLastError();
      return NVFP4_ERR_ARG;
    }
    if (nvfp4_status st = nvfp4::classify_pointer(at.type, at.device, dev); st != NVFP4_OK) return st;
  }
  return NVFP4_OK;
}

}  // namespace

namespace nvfp4 {

nvfp4_status check_quantize_args(const void* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* codes,
                                 const uint8_t* scales, const float* tensor_scale, const float* tensor_scale_in,
                                 const void* workspace, bool library_scratch) {
  if (M < 0 || K <= 0 || K % 64 != 0 || ldx < K) return NVFP4_ERR_SHAPE;
  if (M > 0 && K > kMaxElems / M) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;  // empty: nothing is read or written (pointers may be NULL)
  if (x == nullptr || codes == nullptr || scales == nullptr || tensor_scale == nullptr)
    return NVFP4_ERR_NULL;
  if (!library_scratch && tensor_scale_in == nullptr && workspace == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(x) || ldx % 8 != 0 || !aligned16(codes) || !aligned16(scales) ||
      (workspace != nullptr && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return NVFP4_ERR_ALIGN;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  return check_pointers({x, codes, scales, tensor_scale, tensor_scale_in, workspace});
}

}  // namespace nvfp4

extern "C" {

size_t nvfp4_scales_bytes(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0 || K % 64 != 0) return 0;
  return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>(K / 64) * 512u;
}

int64_t nvfp4_scale_offset(int64_t row, int64_t kblock, int64_t K) {
  if (row < 0 || kblock < 0 || K <= 0 || K % 64 != 0 || kblock >= K / 16) return -1;
  return ((row / 128) * (K / 64) + kblock / 4) * 512 + (row % 32) * 16 + ((row / 32) % 4) * 4 + kblock % 4;
}

size_t nvfp4_workspace_bytes(void) { return 16; }

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_NULL: return "NVFP4_ERR_NULL";
    case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE";
    case NVFP4_ERR_ALIGN: return "NVFP4_ERR_ALIGN";
    case NVFP4_ERR_DEVICE: return "NVFP4_ERR_DEVICE";
    case NVFP4_ERR_LAUNCH: return "NVFP4_ERR_LAUNCH";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
    case NVFP4_ERR_ARG: return "NVFP4_ERR_ARG";
  }
  return "NVFP4_ERR_UNKNOWN";
}

nvfp4_status nvfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, float* tensor_scale, const float* tensor_scale_in,
                            void* workspace, nvfp4_stream_t stream) {
  if (nvfp4_status st = nvfp4::check_quantize_args(x, M, K, ldx, codes, scales, tensor_scale, tensor_scale_in,
                                                   workspace, false);
      st != NVFP4_OK || M == 0)
    return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(nvfp4::launch_quantize(x, M, K, ldx, codes, scales, static_cast<unsigned*>(workspace),
                                          tensor_scale_in, tensor_scale, s));
}

nvfp4_status nvfp4_pack_weights(const void* w, int64_t K, int64_t N, int gated_interleave, uint8_t* codes,
                                uint8_t* scales, float* tensor_scale, void* workspace, nvfp4_stream_t stream) {
  if (w == nullptr || codes == nullptr || scales == nullptr || tensor_scale == nullptr || workspace == nullptr)
    return NVFP4_ERR_NULL;
  if (gated_interleave != 0 && gated_interleave != 1) return NVFP4_ERR_ARG;
  if (K <= 0 || K % 64 != 0 || N <= 0 || N % 8 != 0) return NVFP4_ERR_SHAPE;
  if (K > kMaxElems / N || K / 64 > 65535) return NVFP4_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return NVFP4_ERR_ALIGN;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (nvfp4_status st = check_pointers({w, codes, scales, tensor_scale, workspace}); st != NVFP4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* amax = static_cast<unsigned*>(workspace);
  if (cudaMemsetAsync(amax, 0, nvfp4_workspace_bytes(), s) != cudaSuccess) return NVFP4_ERR_LAUNCH;
  if (cudaMemsetAsync(scales, 0, nvfp4_scales_bytes(N, K), s) != cudaSuccess) return NVFP4_ERR_LAUNCH;
  if (nvfp4_status st = from_cuda(nvfp4::launch_amax(w, K, N, N, amax, s)); st != NVFP4_OK) return st;
  if (nvfp4_status st = from_cuda(nvfp4::launch_pack_weights(w, K, N, gated_interleave == 1, codes, scales,
                                                               amax, tensor_scale, s));
      st != NVFP4_OK)
    return st;
  // leave the workspace zeroed, the state nvfp4_quantize expects of a fresh workspace
  return from_cuda(cudaMemsetAsync(amax, 0, nvfp4_workspace_bytes(), s));
}

namespace {

// Shape / argument checks and argument packing shared by the two GEMM entry points; the
// output-specific checks are the callers'.
nvfp4_status gemm_args(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_ts,
                       const uint8_t* b_codes, const uint8_t* b_scales, const float* b_ts, int64_t M, int64_t N,
                       int64_t K, nvfp4_epilogue epi, const float* bias, const float* gamma, int head_dim,
                       int64_t norm_cols, float eps, int* device_error, nvfp4::GemmArgs& a, int64_t& out_cols) {
  if (epi != NVFP4_EPI_BIAS && epi != NVFP4_EPI_HEAD_RMSNORM && epi != NVFP4_EPI_GATED_SILU)
    return NVFP4_ERR_ARG;
  if (epi == NVFP4_EPI_HEAD_RMSNORM) {
    if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256) return NVFP4_ERR_ARG;
    if (!(eps >= 0.0f) || eps != eps) return NVFP4_ERR_ARG;
  }
  if (M < 0 || N <= 0 || N % 32 != 0 || K <= 0 || K % 64 != 0) return NVFP4_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return NVFP4_ERR_SHAPE;
  // operands no larger than the quantizer and packer produce (M * K and N * K below 2^34), and
  // the kernel's pair-tile index and row coordinates within 32 bits
  if ((M > 0 && K > kMaxElems / M) || K > kMaxElems / N) return NVFP4_ERR_SHAPE;
  if (((M + 255) / 256) * ((N + 255) / 256) > int64_t{INT32_MAX}) return NVFP4_ERR_SHAPE;
  if (epi == NVFP4_EPI_HEAD_RMSNORM && (norm_cols < 0 || norm_cols > N || norm_cols % head_dim != 0))
    return NVFP4_ERR_SHAPE;
  out_cols = epi == NVFP4_EPI_GATED_SILU ? N / 2 : N;
  a.a_codes = a_codes;
  a.a_scales = a_scales;
  a.a_ts = a_ts;
  a.b_codes = b_codes;
  a.b_scales = b_scales;
  a.b_ts = b_ts;
  a.M = M;
  a.N = N;
  a.K = K;
  a.epi = static_cast<int>(epi);
  a.bias = bias;
  a.gamma = gamma;
  a.head_dim = epi == NVFP4_EPI_HEAD_RMSNORM ? head_dim : 256;
  a.norm_cols = epi == NVFP4_EPI_HEAD_RMSNORM ? norm_cols : 0;
  a.eps = eps;
  a.err = device_error;
  return NVFP4_OK;
}

// Input pointer checks (after M == 0 has returned); FP8 operands have no block scales.
nvfp4_status gemm_inputs_ok(const nvfp4::GemmArgs& a) {
  if (a.a_codes == nullptr || a.a_ts == nullptr || a.b_codes == nullptr || a.b_ts == nullptr)
    return NVFP4_ERR_NULL;
  if (!a.fp8 && (a.a_scales == nullptr || a.b_scales == nullptr)) return NVFP4_ERR_NULL;
  if (a.epi == NVFP4_EPI_HEAD_RMSNORM && a.gamma == nullptr && a.norm_cols > 0) return NVFP4_ERR_NULL;
  if (!aligned16(a.a_codes) || !aligned16(a.b_codes)) return NVFP4_ERR_ALIGN;
  if (!a.fp8 && (!aligned16(a.a_scales) || !aligned16(a.b_scales))) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

// Device check, then every pointer the GEMM kernel will read or write (tensor maps included)
// must be memory of the current device.
nvfp4_status gemm_memory_ok(const nvfp4::GemmArgs& a) {
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  return check_pointers({a.a_codes, a.a_scales, a.a_ts, a.b_codes, a.b_scales, a.b_ts, a.bias, a.gamma, a.out,
                         a.out_codes, a.out_scales, a.out_ts, a.err});
}

}  // namespace

nvfp4_status nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_ts,
                        const uint8_t* b_codes, const uint8_t* b_scales, const float* b_ts, int64_t M,
                        int64_t N, int64_t K, nvfp4_epilogue epi, const float* bias, const float* gamma,
                        int head_dim, int64_t norm_cols, float eps, nvfp4_out_dtype out_dtype, void* out,
                        int64_t ldo, int* device_error, nvfp4_stream_t stream) {
  nvfp4::GemmArgs a;
  int64_t out_cols = 0;
  if (nvfp4_status st = gemm_args(a_codes, a_scales, a_ts, b_codes, b_scales, b_ts, M, N, K, epi, bias, gamma,
                                  head_dim, norm_cols, eps, device_error, a, out_cols);
      st != NVFP4_OK)
    return st;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_ARG;
  if (ldo < out_cols) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;  // empty: nothing is read or written (pointers may be NULL)
  if (nvfp4_status st = gemm_inputs_ok(a); st != NVFP4_OK) return st;
  if (out == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(out) || ldo % (out_dtype == NVFP4_OUT_BF16 ? 8 : 4) != 0) return NVFP4_ERR_ALIGN;
  a.out_fp32 = out_dtype == NVFP4_OUT_FP32 ? 1 : 0;
  a.out = out;
  a.ldo = ldo;
  if (nvfp4_status st = gemm_memory_ok(a); st != NVFP4_OK) return st;
  return nvfp4::launch_gemm(a, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm_nvfp4_out(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_ts,
                                  const uint8_t* b_codes, const uint8_t* b_scales, const float* b_ts, int64_t M,
                                  int64_t N, int64_t K, nvfp4_epilogue epi, const float* bias,
                                  const float* gamma, int head_dim, int64_t norm_cols, float eps,
                                  const float* out_tensor_scale, uint8_t* out_codes, uint8_t* out_scales,
                                  int* device_error, nvfp4_stream_t stream) {
  nvfp4::GemmArgs a;
  int64_t out_cols = 0;
  if (nvfp4_status st = gemm_args(a_codes, a_scales, a_ts, b_codes, b_scales, b_ts, M, N, K, epi, bias, gamma,
                                  head_dim, norm_cols, eps, device_error, a, out_cols);
      st != NVFP4_OK)
    return st;
  if (out_cols % 64 != 0) return NVFP4_ERR_SHAPE;  // the output is the next GEMM's K
  if (M == 0) return NVFP4_OK;
  if (nvfp4_status st = gemm_inputs_ok(a); st != NVFP4_OK) return st;
  if (out_tensor_scale == nullptr || out_codes == nullptr || out_scales == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(out_codes) || !aligned16(out_scales)) return NVFP4_ERR_ALIGN;
  a.out_fp32 = 0;
  a.out = nullptr;
  a.ldo = out_cols;
  a.out_nvfp4 = 1;
  a.out_codes = out_codes;
  a.out_scales = out_scales;
  a.out_ts = out_tensor_scale;
  if (nvfp4_status st = gemm_memory_ok(a); st != NVFP4_OK) return st;
  return nvfp4::launch_gemm(a, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status fp8_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes, float* tensor_scale,
                          const float* tensor_scale_in, void* workspace, nvfp4_stream_t stream) {
  if (M < 0 || K <= 0 || K % 64 != 0 || ldx < K) return NVFP4_ERR_SHAPE;
  if (M > 0 && K > kMaxElems / M) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (x == nullptr || codes == nullptr || tensor_scale == nullptr) return NVFP4_ERR_NULL;
  if (tensor_scale_in == nullptr && workspace == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(x) || ldx % 8 != 0 || !aligned16(codes) || (workspace != nullptr && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return NVFP4_ERR_ALIGN;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (nvfp4_status st = check_pointers({x, codes, tensor_scale, tensor_scale_in, workspace}); st != NVFP4_OK)
    return st;
  return from_cuda(nvfp4::launch_fp8_quantize(x, M, K, ldx, codes, static_cast<unsigned*>(workspace),
                                              tensor_scale_in, tensor_scale, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status fp8_pack_weights(const void* w, int64_t K, int64_t N, int gated_interleave, uint8_t* codes,
                              float* tensor_scale, void* workspace, nvfp4_stream_t stream) {
  if (w == nullptr || codes == nullptr || tensor_scale == nullptr || workspace == nullptr) return NVFP4_ERR_NULL;
  if (gated_interleave != 0 && gated_interleave != 1) return NVFP4_ERR_ARG;
  if (K <= 0 || K % 64 != 0 || N <= 0 || N % 8 != 0) return NVFP4_ERR_SHAPE;
  if (K > kMaxElems / N || K / 64 > 65535) return NVFP4_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return NVFP4_ERR_ALIGN;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (nvfp4_status st = check_pointers({w, codes, tensor_scale, workspace}); st != NVFP4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* amax = static_cast<unsigned*>(workspace);
  if (cudaMemsetAsync(amax, 0, nvfp4_workspace_bytes(), s) != cudaSuccess) return NVFP4_ERR_LAUNCH;
  if (nvfp4_status st = from_cuda(nvfp4::launch_amax(w, K, N, N, amax, s)); st != NVFP4_OK) return st;
  if (nvfp4_status st = from_cuda(nvfp4::launch_fp8_pack_weights(w, K, N, gated_interleave == 1, codes, amax,
                                                                   tensor_scale, s));
      st != NVFP4_OK)
    return st;
  return from_cuda(cudaMemsetAsync(amax, 0, nvfp4_workspace_bytes(), s));
}

nvfp4_status fp8_gemm(const uint8_t* a_codes, const float* a_ts, const uint8_t* b_codes, const float* b_ts, int64_t M,
                      int64_t N, int64_t K, nvfp4_epilogue epi, const float* bias, const float* gamma, int head_dim,
                      int64_t norm_cols, float eps, nvfp4_out_dtype out_dtype, void* out, int64_t ldo,
                      int* device_error, nvfp4_stream_t stream) {
  nvfp4::GemmArgs a;
  int64_t out_cols = 0;
  if (nvfp4_status st = gemm_args(a_codes, nullptr, a_ts, b_codes, nullptr, b_ts, M, N, K, epi, bias, gamma,
                                  head_dim, norm_cols, eps, device_error, a, out_cols);
      st != NVFP4_OK)
    return st;
  a.fp8 = 1;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_ARG;
  if (ldo < out_cols) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (nvfp4_status st = gemm_inputs_ok(a); st != NVFP4_OK) return st;
  if (out == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(out) || ldo % (out_dtype == NVFP4_OUT_BF16 ? 8 : 4) != 0) return NVFP4_ERR_ALIGN;
  a.out_fp32 = out_dtype == NVFP4_OUT_FP32 ? 1 : 0;
  a.out = out;
  a.ldo = ldo;
  if (nvfp4_status st = gemm_memory_ok(a); st != NVFP4_OK) return st;
  return nvfp4::launch_gemm(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t attention_workspace_bytes(int64_t M, int heads) {
  if (M <= 0 || heads <= 0) return 0;
  return static_cast<size_t>(heads) * 256u * static_cast<size_t>(nvfp4::attention_vt_ld(M)) * 2u;
}

nvfp4_status attention_fwd(const void* qkv, int64_t M, int64_t ld_qkv, int heads, int head_dim, void* workspace,
                           void* out, int64_t ldo, int* device_error, nvfp4_stream_t stream) {
  if (head_dim != 256) return NVFP4_ERR_ARG;
  if (heads <= 0 || heads > 256 || M < 0 || M > (int64_t(1) << 31) - 1) return NVFP4_ERR_SHAPE;
  const int64_t hidden = static_cast<int64_t>(heads) * head_dim;
  if (ld_qkv < 3 * hidden || ldo < hidden) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (qkv == nullptr || workspace == nullptr || out == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(qkv) || !aligned16(workspace) || !aligned16(out) || ld_qkv % 8 != 0 || ldo % 8 != 0)
    return NVFP4_ERR_ALIGN;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (nvfp4_status st = check_pointers({qkv, workspace, out, device_error}); st != NVFP4_OK) return st;
  return nvfp4::launch_attention(qkv, M, ld_qkv, heads, workspace, out, ldo, device_error,
                                 reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_get_device_error(int* device_error, int* code, nvfp4_stream_t stream) {
  if (device_error == nullptr || code == nullptr) return NVFP4_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, device_error, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return NVFP4_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_LAUNCH;
  *code = host;
  if (cudaMemsetAsync(device_error, 0, sizeof(int), s) != cudaSuccess) return NVFP4_ERR_LAUNCH;
  return NVFP4_OK;
}

nvfp4_status nvfp4_debug_wait_timeout(int* device_error, int64_t timeout_ns, nvfp4_stream_t stream) {
  if (device_error == nullptr) return NVFP4_ERR_NULL;
  if (timeout_ns < 1 || timeout_ns > 10000000000ll) return NVFP4_ERR_ARG;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (nvfp4_status st = check_pointers({device_error}); st != NVFP4_OK) return st;
  return from_cuda(nvfp4::launch_wait_timeout(device_error, static_cast<uint64_t>(timeout_ns),
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int nvfp4_debug_build(void) {
#ifdef NVFP4_DEBUG
  return 1;
#else
  return 0;
#endif
}

nvfp4_status nvfp4_debug_index_failures(int64_t* count) {
  if (count == nullptr) return NVFP4_ERR_NULL;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_LAUNCH;
  unsigned q = 0u, g = 0u;
  if (nvfp4::take_index_failures_quantize(&q) != cudaSuccess || nvfp4::take_index_failures_gemm(&g) != cudaSuccess)
    return NVFP4_ERR_LAUNCH;
  *count = static_cast<int64_t>(q) + static_cast<int64_t>(g);
  return NVFP4_OK;
}

nvfp4_status nvfp4_debug_mma_rate(nvfp4_probe_kind kind, int cta_group, int n, int64_t iters, int ctas,
                                  int64_t* out, int* device_error, nvfp4_stream_t stream) {
  if (kind != NVFP4_PROBE_NVFP4 && kind != NVFP4_PROBE_FP8 && kind != NVFP4_PROBE_BF16) return NVFP4_ERR_ARG;
  if (cta_group != 1 && cta_group != 2) return NVFP4_ERR_ARG;
  if (n != 64 && n != 128 && n != 192 && n != 256) return NVFP4_ERR_SHAPE;
  if (iters < 1 || iters > 4000000) return NVFP4_ERR_ARG;
  if (out == nullptr) return NVFP4_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return NVFP4_ERR_ALIGN;
  if (nvfp4_status st = check_device(); st != NVFP4_OK) return st;
  if (ctas < 1 || ctas > nvfp4::sm_count() / cta_group) return NVFP4_ERR_SHAPE;
  if (nvfp4_status st = check_pointers({out, device_error}); st != NVFP4_OK) return st;
  return nvfp4::launch_mma_probe(static_cast<int>(kind), cta_group, n, static_cast<int>(iters), ctas,
                                 reinterpret_cast<long long*>(out), device_error,
                                 reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
