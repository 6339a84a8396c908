// attn_decode.cu -- split-KV decode kernel (placeholder until the fast path lands).
#include "common.cuh"
#include "internal.h"

namespace extkv {
bool decode_supported(const AttnArgs&) { return false; }
cudaError_t launch_attn_decode(const AttnArgs&, const char** name) {
  *name = "";
  return cudaErrorNotSupported;
}
}  // namespace extkv
