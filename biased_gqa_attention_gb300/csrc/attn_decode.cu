// attn_decode.cu -- the decode kernel for one head size of queries, keys and
// values, which shapes the decode path takes, its workspace, and the dispatch
// over the head sizes (pairs of two head sizes are compiled in their own
// translation unit).
#include "attn_decode.cuh"

namespace extkv {

namespace {

DecodeShape shape_for(int64_t Dk, int64_t Dv, int64_t B, int64_t items_max) {
  if (Dk != Dv) return decode_shape_mixed(Dk, Dv, B, items_max);
  switch (Dk) {
    case 64: return decode_shape<64, 64>(B, items_max);
    case 128: return decode_shape<128, 128>(B, items_max);
    case 256: return decode_shape<256, 256>(B, items_max);
    default: return decode_shape<512, 512>(B, items_max);
  }
}

// Pairs of two head sizes the decode kernel runs (without a softcap).
bool mixed_pair(int64_t Dk, int64_t Dv) {
  auto in = [](int64_t d) { return d == 128 || d == 256 || d == 512; };
  return Dk != Dv && in(Dk) && in(Dv);
}

// Whether the cluster kernel should take a call it can run with C CTAs per
// unit.  Its time follows the unit with the most live tiles, shared by C
// CTAs; stream-K's the average over its grid of G CTAs plus its fixed costs
// (plan, tables, merge: about kClusterSlack tiles of one CTA's streaming).  A
// unit's live tiles are bounded by max_seq, or, for the fused specification
// with a causal window and no spans, by the window; a materialised bias
// gives no bound without reading it.
constexpr double kClusterSlack = 8.0;
// the merge kernel a split into M > 1 clusters per unit adds (its launch and
// two dependent round trips), in the same units (measured: the split wins
// against stream-K from one to four long sequences)
constexpr double kMergeTiles = 2.0;

bool cluster_pays(const AttnArgs& a, int C, int M) {
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  int64_t L = max_tiles;
  if (a.fused && !a.spans && a.causal && a.window > 0)
    L = std::min<int64_t>(max_tiles, (a.window + a.S_q - 1 + kTile - 1) / kTile + 1);
  const int64_t units = a.B * a.Hkv * row_groups((a.Hq / a.Hkv) * a.S_q);
  const DecodeShape d = shape_for(a.D, a.Dv, a.B, units * max_tiles);
  const double excess =
      static_cast<double>(L) * (1.0 / (static_cast<double>(C) * M) - static_cast<double>(units) / std::max(d.G, 1));
  return excess <= kClusterSlack - (M > 1 ? kMergeTiles : 0.0);
}

}  // namespace

size_t decode_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk,
                              int64_t Dv) {
  const int64_t max_tiles = (max_seq + kTile - 1) / kTile;
  const int64_t gr = Hq / Hkv * S_q, n_rg = row_groups(gr);
  return ws_layout(B, Hkv * n_rg, max_tiles, shape_for(Dk, Dv, B, B * Hkv * n_rg * max_tiles).G,
                   std::min<int64_t>(gr, kRows), Dv).total;
}

bool decode_supported(const AttnArgs& a) {
  if (a.decode_variant == kDecodeCluster) return decode_cluster_size(a) > 0;
  if (a.dtype != EXTKV_BF16) return false;
  if (a.Dv != a.D) {
    if (!mixed_pair(a.D, a.Dv) || a.softcap > 0.f) return false;
  } else if (a.D != 64 && a.D != 128 && a.D != 256 && a.D != 512) {
    return false;
  }
  // up to kMaxRowGroups units of 8 query rows per KV head; a stage's bias or
  // extra-term block holds the 16 keys of every query position (S_q <= 8)
  if ((a.Hq / a.Hkv) * a.S_q > kRows * kMaxRowGroups || a.S_q > kRows) return false;
  // 16-byte rows for the bias / extra-term block copies
  if ((a.bias || (a.fused && a.extra)) && a.max_seq % 8) return false;
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  const int64_t units = a.B * a.Hkv * row_groups((a.Hq / a.Hkv) * a.S_q);
  if (a.B > kMaxBatches || units >= (1 << 20) || max_tiles > 65535) return false;
  if (a.B * a.Hq * a.S_q > 0x7fffffff || units * max_tiles > 0x7fffffff) return false;
  // the per-batch tables and the longest slice's work list fit shared memory
  const DecodeShape d = shape_for(a.D, a.Dv, a.B, units * max_tiles);
  return d.occ > 0 && d.slice <= d.wc;
}

cudaError_t launch_attn_decode(const AttnArgs& a, const char** name) {
  // The cluster kernel (no plan, tables or merge) where its longest share is
  // not much longer than stream-K's average one (cluster_pays); stream-K
  // otherwise.  Measured: the decode workload (64 units, 8 CTAs each) 16.0 us
  // against 21.7 us; one sequence of 8000 keys (8 units) 60.7 us against
  // 24.5 us; the global-layer decode (64 units, 4 CTAs each at head size 512)
  // 141 us against 86 us.
  if (a.decode_variant != kDecodeStreamK) {
    const int C = decode_cluster_size(a);
    const int M = decode_cluster_split(a, C);
    if (C > 0 && (a.decode_variant == kDecodeCluster || cluster_pays(a, C, M)))
      return launch_attn_decode_cluster(a, C, M, name);
    if (a.decode_variant == kDecodeCluster) return cudaErrorInvalidValue;
  }
  if (a.Dv != a.D) return launch_attn_decode_mixed(a, name);
  switch (a.D) {
    case 64: return launch_d<64, 64>(a, name);
    case 128: return launch_d<128, 128>(a, name);
    case 256: return launch_d<256, 256>(a, name);
    case 512: return launch_d<512, 512>(a, name);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace extkv
