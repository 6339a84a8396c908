// attn_prefill.cu -- the tensor-core prefill kernel for one head size of
// queries, keys and values up to 256 (and value head sizes that are whole
// multiples of it), which shapes it takes, its workspace, and the dispatch
// over the head-size groups (each group compiled in its own translation unit).
#include "attn_prefill_pair.cuh"

namespace extkv {

namespace {

// Head size 256 on CTA pairs: the two query heads of a pair share a KV head
// (an even group size), the grid is large enough not to split keys, and the
// rows are not packed (a pair holds one tile of each of its two heads).
bool pair_ok(const AttnArgs& a) {
  return a.prefill_pairs && a.D == 256 && a.Dv == 256 && (a.Hq / a.Hkv) % 2 == 0 &&
         !packs_rows(a.Hq, a.Hkv, a.S_q) && prefill_splits(a.B, a.Hq, a.S_q) == 1;
}

template <bool CAP>
cudaError_t launch_pair_c(const AttnArgs& a, const char** name) {
  if (a.bias) return launch_pair<kBias, CAP>(a, name);
  if (a.fused) return a.extra ? launch_pair<kFusedExtra, CAP>(a, name) : launch_pair<kFused, CAP>(a, name);
  return launch_pair<kNone, CAP>(a, name);
}

}  // namespace

cudaError_t launch_attn_prefill_equal(const AttnArgs& a, const char** name) {
  switch (a.D) {
    case 64: return launch_kv<64, 64>(a, name);
    case 128: return launch_kv<128, 128>(a, name);
    case 256:
      if (pair_ok(a)) return a.softcap > 0.f ? launch_pair_c<true>(a, name) : launch_pair_c<false>(a, name);
      return launch_kv<256, 256>(a, name);
    default: return cudaErrorInvalidValue;
  }
}

size_t prefill_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk,
                               int64_t Dv, bool term) {
  (void)Dk;
  const int64_t n_vc = Dv / v_chunk(Dv);
  const int ns = prefill_call_splits(B, Hq, Hkv, S_q, n_vc);
  if (!term && ns == 1) return 0;
  const size_t part = ns > 1 ? static_cast<size_t>(ns) * B * Hq * S_q * part_stride(static_cast<int>(Dv)) * 4 : 0;
  return term_tables_bytes(B, S_q, max_seq) + part;  // the partials follow the (maybe unused) term tables
}

bool prefill_supported(const AttnArgs& a) {
  if (a.dtype != EXTKV_BF16) return false;
  if (!prefill_pair_supported(a.D, a.Dv)) return false;
  // 16-byte rows for the bias / extra-term copies
  if ((a.bias || (a.fused && a.extra)) && a.max_seq % 8) return false;
  if (a.B * a.Hq * a.S_q > 0x7fffffff || a.B * a.S_q > 0x7fffffff) return false;
  if (a.max_seq > 0x7fffffff - 2 * kPlanKeys || a.B > 65535 || n_query_tiles(a.S_q) > 65535) return false;
  if (a.Hq * (a.Dv / v_chunk(a.Dv)) * kMaxSplit > 0x7fffffff) return false;
  return true;
}

cudaError_t launch_attn_prefill(const AttnArgs& a, const char** name) {
  if (!prefill_pair_supported(a.D, a.Dv)) return cudaErrorInvalidValue;
  if (a.D == 512) return launch_attn_prefill_dk512(a, name);
  if (a.D == v_chunk(a.Dv)) return launch_attn_prefill_equal(a, name);  // Dv == D, or Dv == 512 in chunks of D
  return launch_attn_prefill_mixed(a, name);
}

}  // namespace extkv
