// tma_host.cu -- tensor map encoding (host).
#include <cstring>
#include <mutex>

#include "tma_host.h"

namespace extkv {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The arguments of one encode; a tensor map is a function of them alone.
struct MapKey {
  const void* base;
  int rank, swizzle;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
};

// The last few maps this thread encoded: a caller repeating a step over the
// same buffers encodes each map once.
struct MapCache {
  static constexpr int kSlots = 16;
  MapKey key[kSlots];
  CUtensorMap map[kSlots];
  int used = 0, next = 0;
};
thread_local MapCache t_maps;

}  // namespace

bool make_tensor_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box,
                          CUtensorMapSwizzle swizzle) {
  if (rank < 1 || rank > 5) return false;
  MapKey k;
  std::memset(&k, 0, sizeof k);
  k.base = base;
  k.rank = rank;
  k.swizzle = static_cast<int>(swizzle);
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides_bytes[i];
  }
  MapCache& c = t_maps;
  for (int i = 0; i < c.used; ++i)
    if (std::memcmp(&c.key[i], &k, sizeof k) == 0) {
      *map = c.map[i];
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                  const_cast<void*>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  const int slot = c.next;
  c.key[slot] = k;
  c.map[slot] = *map;
  c.next = (c.next + 1) % MapCache::kSlots;
  if (c.used < MapCache::kSlots) ++c.used;
  return true;
}

cudaError_t set_max_dynamic_smem(const void* kernel, size_t bytes) {
  // per (kernel, device): the largest size set so far; a smaller request needs no call
  static std::mutex mu;
  struct Entry {
    const void* kernel;
    int dev;
    size_t bytes;
  };
  static Entry entries[256];
  static int n = 0;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  for (int i = 0; i < n; ++i)
    if (entries[i].kernel == kernel && entries[i].dev == dev) {
      if (entries[i].bytes >= bytes) return cudaSuccess;
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
      if (e == cudaSuccess) entries[i].bytes = bytes;
      return e;
    }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && n < 256) entries[n++] = Entry{kernel, dev, bytes};
  return e;
}

}  // namespace extkv
