// nvfp4_quantize_noalloc: the activation quantizer for callers that cannot allocate device
// memory (see include/nvfp4.h). Its scratch -- the quantizer's 16 workspace bytes (the amax
// word, two grid-barrier counters and a failure flag) -- lives in a fixed array inside this
// library instead of a caller-provided workspace.

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "nvfp4_internal.h"

namespace {

// Fixed scratch for nvfp4_quantize_noalloc. Every GPU that loads the library holds these
// bytes until the process exits. All calls share them.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_dev_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device. In host code the array's name
// only stands in for the symbol; the address a kernel may use comes from
// cudaGetSymbolAddress, resolved once per device with that device current.
nvfp4_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return NVFP4_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return NVFP4_ERR_LAUNCH;
    }
    g_scratch_dev_ptr[dev] = p;
  }
  *out = g_scratch_dev_ptr[dev];
  return NVFP4_OK;
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                                    uint8_t* scales, float* tensor_scale, nvfp4_stream_t stream) {
  // Every check nvfp4_quantize makes (shapes, NULL, alignment, device, memory of the current
  // device) comes first: a refused call touches neither the scratch nor the stream.
  if (nvfp4_status st = nvfp4::check_quantize_args(x, M, K, ldx, codes, scales, tensor_scale, nullptr, nullptr,
                                                   true);
      st != NVFP4_OK || M == 0)
    return st;
  // The quantizer's scratch must fit the fixed array; a larger need is refused, not truncated.
  if (nvfp4_workspace_bytes() > kNoAllocScratchBytes) return NVFP4_ERR_SHAPE;
  void* scratch = nullptr;
  if (nvfp4_status st = scratch_address(&scratch); st != NVFP4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Start from a zeroed scratch every call, so an earlier call that was interrupted (or timed
  // out) cannot leave this shared array in a bad state.
  if (cudaMemsetAsync(scratch, 0, nvfp4_workspace_bytes(), s) != cudaSuccess) return NVFP4_ERR_LAUNCH;
  return nvfp4::launch_quantize(x, M, K, ldx, codes, scales, static_cast<unsigned*>(scratch), nullptr,
                                tensor_scale, s) == cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_LAUNCH;
}

}  // extern "C"
