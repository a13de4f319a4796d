// Which memory a pointer passed to the library may name: host-side decision logic, kept apart
// from the CUDA calls that gather its inputs so that it can be exercised without a GPU.
#pragma once

#include <cuda_runtime_api.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// NVFP4_OK when memory of kind `type` that belongs to device `owner` may be read or written by
// kernels launched on device `current`, and described by their TMA tensor maps: device memory
// or managed memory of that same device. Anything else -- pageable or pinned host memory,
// unregistered addresses, or another GPU's memory reached through unified addressing -- is
// NVFP4_ERR_ARG, so no kernel of the library ever touches another device's memory.
inline nvfp4_status classify_pointer(cudaMemoryType type, int owner, int current) {
  if (type != cudaMemoryTypeDevice && type != cudaMemoryTypeManaged) return NVFP4_ERR_ARG;
  return owner == current ? NVFP4_OK : NVFP4_ERR_ARG;
}

}  // namespace nvfp4
