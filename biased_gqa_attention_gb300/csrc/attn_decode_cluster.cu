// attn_decode_cluster.cu -- which decode calls the cluster kernel takes, and
// its dispatch over the head sizes.
#include "attn_decode_cluster.cuh"

namespace extkv {

int decode_cluster_size(const AttnArgs& a) {
  if (a.dtype != EXTKV_BF16 || a.Dv != a.D) return 0;
  if (a.D != 64 && a.D != 128 && a.D != 256 && a.D != 512) return 0;
  if (a.Hkv <= 0 || a.Hq % a.Hkv) return 0;
  // units of at most 8 query rows, up to 8 per KV head; a stage's bias block
  // holds the 16 keys of every query position (S_q <= 8)
  if ((a.Hq / a.Hkv) * a.S_q > kRows * kMaxRowGroups || a.S_q > kRows) return 0;
  // the fused specification's live tiles in closed form (several positions
  // with spans need a per-tile test)
  if (a.fused && needs_plan(a)) return 0;
  // 16-byte rows for the bias / extra-term copies; a materialised bias is
  // scanned from one copy of the batch's rows
  if ((a.bias || (a.fused && a.extra)) && a.max_seq % 8) return 0;
  if (a.bias && a.S_q * a.max_seq * 2 > kScanBytes) return 0;
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  if (max_tiles > 65535 || a.B * a.Hq * a.S_q > 0x7fffffff) return 0;
  const int64_t units = a.B * a.Hkv * row_groups((a.Hq / a.Hkv) * a.S_q);
  if (units <= 0 || units > (1 << 20)) return 0;
  switch (a.D) {
    case 64: return cluster_size_for<64, 64>(units);
    case 128: return cluster_size_for<128, 128>(units);
    case 256: return cluster_size_for<256, 256>(units);
    default: return cluster_size_for<512, 512>(units);
  }
}

int decode_cluster_split(const AttnArgs& a, int C) {
  if (C <= 0) return 0;
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  const int64_t units = a.B * a.Hkv * row_groups((a.Hq / a.Hkv) * a.S_q);
  switch (a.D) {
    case 64: return cluster_split_for<64>(a.B, units, max_tiles, C);
    case 128: return cluster_split_for<128>(a.B, units, max_tiles, C);
    case 256: return cluster_split_for<256>(a.B, units, max_tiles, C);
    default: return cluster_split_for<512>(a.B, units, max_tiles, C);
  }
}

cudaError_t launch_attn_decode_cluster(const AttnArgs& a, int C, int M, const char** name) {
  switch (a.D) {
    case 64: return launch_dc<64>(a, C, M, name);
    case 128: return launch_dc<128>(a, C, M, name);
    case 256: return launch_dc<256>(a, C, M, name);
    case 512: return launch_dc<512>(a, C, M, name);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace extkv
