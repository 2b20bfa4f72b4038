// Host helpers for the tensor-core kernels: TMA tensor-map encoding through the
// driver entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mla {

// Encodes a bf16 tensor map of rank 2 or 3 with 128-byte swizzle (or the
// given swizzle).  dims[0] is the contiguous axis; strides_bytes[i] is the
// byte stride of dims[i+1].  Returns false (and sets the error detail) on
// failure.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe.  Returns the CUDA error of
// the attribute call (cudaSuccess when already set).
cudaError_t set_max_dynamic_smem(const void* kernel, int bytes);
template <typename... KArgs>
cudaError_t set_max_dynamic_smem(void (*kernel)(KArgs...), int bytes) {
  return set_max_dynamic_smem(reinterpret_cast<const void*>(kernel), bytes);
}

// Launch with programmatic dependent launch allowed: the kernel may start its
// prologue while the previous kernel in the stream drains; every kernel
// launched this way calls griddepcontrol.wait before it touches memory the
// previous kernels write, and griddepcontrol.launch_dependents when done.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace mla
