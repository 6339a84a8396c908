// attn_prefill_dk512.cu -- the tensor-core prefill kernel for a query-key head
// size of 512: Q stays in shared memory (128 KB), each K tile streams as four
// 128-column units, and a value head size of 512 is written as two 256-column
// chunks by two CTAs.
#include "attn_prefill.cuh"

namespace extkv {

cudaError_t launch_attn_prefill_dk512(const AttnArgs& a, const char** name) {
  if (a.D != 512) return cudaErrorInvalidValue;
  switch (a.Dv) {
    case 128: return launch_kv<512, 128>(a, name);
    case 256:
    case 512: return launch_kv<512, 256>(a, name);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace extkv
