// attn_prefill.cu -- tcgen05 prefill kernel (placeholder until the fast path lands).
#include "common.cuh"
#include "internal.h"

namespace extkv {
bool prefill_supported(const AttnArgs&) { return false; }
cudaError_t launch_attn_prefill(const AttnArgs&, const char** name) {
  *name = "";
  return cudaErrorNotSupported;
}
}  // namespace extkv
