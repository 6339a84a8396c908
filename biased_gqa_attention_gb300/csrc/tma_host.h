// tma_host.h -- host-side creation of TMA tensor maps through the driver
// entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace extkv {

// Encodes a tiled bf16 tensor map over a row-major tensor of up to three
// dimensions (dims[0] innermost).  strides_bytes[i] is the stride of
// dimension i+1.  Returns false if the driver rejects it.
bool make_tensor_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box,
                          CUtensorMapSwizzle swizzle);

}  // namespace extkv
