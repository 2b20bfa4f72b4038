// Host helpers for the tensor-core kernels: TMA tensor-map encoding through the
// driver entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Encodes a bf16 tensor map of rank 2 or 3 with 128-byte swizzle.
// dims[0] is the contiguous axis; strides_bytes[i] is the byte stride of
// dims[i+1].  Returns false (and sets the error detail) on failure.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace mla
