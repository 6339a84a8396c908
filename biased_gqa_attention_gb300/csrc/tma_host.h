// tma_host.h -- host-side creation of TMA tensor maps through the driver
// entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace extkv {

// Encodes a tiled bf16 tensor map over a row-major tensor of up to five
// dimensions (dims[0] innermost).  strides_bytes[i] is the stride of
// dimension i+1.  Returns false if the driver rejects it.  The last maps a
// thread encoded are kept and handed out again for the same arguments.
bool make_tensor_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box,
                          CUtensorMapSwizzle swizzle);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for the current device,
// called only when `bytes` exceeds what was already set for that kernel.
cudaError_t set_max_dynamic_smem(const void* kernel, size_t bytes);

}  // namespace extkv
