// attn_decode_mixed.cu -- the decode kernel for a value head size unlike the
// query-key one (each of 128, 256, 512): a KV-shared layer borrowing the
// cache of a layer with another head size ("Skill: Attention Optimization",
// "ORT CUDA Attention Kernel Dispatch": head_size != v_head_size).  Q and K
// carry Dk, V and Y carry Dv; no fused scatter, no softcap.
#include "attn_decode.cuh"

namespace extkv {

DecodeShape decode_shape_mixed(int64_t Dk, int64_t Dv, int64_t B, int64_t items_max) {
  if (Dk == 128 && Dv == 256) return decode_shape<128, 256>(B, items_max);
  if (Dk == 128 && Dv == 512) return decode_shape<128, 512>(B, items_max);
  if (Dk == 256 && Dv == 128) return decode_shape<256, 128>(B, items_max);
  if (Dk == 256 && Dv == 512) return decode_shape<256, 512>(B, items_max);
  if (Dk == 512 && Dv == 128) return decode_shape<512, 128>(B, items_max);
  return decode_shape<512, 256>(B, items_max);
}

cudaError_t launch_attn_decode_mixed(const AttnArgs& a, const char** name) {
  if (a.D == 128 && a.Dv == 256) return launch_d<128, 256>(a, name);
  if (a.D == 128 && a.Dv == 512) return launch_d<128, 512>(a, name);
  if (a.D == 256 && a.Dv == 128) return launch_d<256, 128>(a, name);
  if (a.D == 256 && a.Dv == 512) return launch_d<256, 512>(a, name);
  if (a.D == 512 && a.Dv == 128) return launch_d<512, 128>(a, name);
  if (a.D == 512 && a.Dv == 256) return launch_d<512, 256>(a, name);
  return cudaErrorInvalidValue;
}

}  // namespace extkv
