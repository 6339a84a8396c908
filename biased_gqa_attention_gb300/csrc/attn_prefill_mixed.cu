// attn_prefill_mixed.cu -- the tensor-core prefill kernel for a value head
// size that differs from the query-key head size (128 or 256):
// ("Skill: Attention Optimization", "ORT CUDA Attention Kernel Dispatch":
// head_size != v_head_size, e.g. a KV-shared layer borrowing the cache of a
// layer with another head size).
#include "attn_prefill.cuh"

namespace extkv {

cudaError_t launch_attn_prefill_mixed(const AttnArgs& a, const char** name) {
  if (a.D == 128 && (a.Dv == 256 || a.Dv == 512)) return launch_kv<128, 256>(a, name);
  if (a.D == 256 && a.Dv == 128) return launch_kv<256, 128>(a, name);
  return cudaErrorInvalidValue;
}

}  // namespace extkv
