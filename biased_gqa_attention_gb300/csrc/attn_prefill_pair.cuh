// attn_prefill_pair.cuh -- prefill attention at head size 256 on CTA pairs:
// the two query heads that share a KV head ("ONNX Domain Attention (Opset
// 23/24) CUDA Patterns", section 1: query head h reads KV head h / (Hq/Hkv))
// run as one M = 256 tcgen05 MMA over the two SMs of a 2-CTA cluster
// (cta_group::2).
//
// Why: at head size 256 the single-SM kernel keeps Q in shared memory (S_0,
// S_1 and O fill the 512 tensor-memory columns), so every Q K^T MMA reads A
// and B from shared memory while the K/V tiles stream in through the same
// port: about 320 KB of shared-memory traffic per 128-key tile, more than the
// tensor cores' time for it.  On a pair, each SM stores half of every K and V
// tile (64 keys of K, 128 columns of V) and serves that half to both tensor
// cores: about 190 KB per SM per tile, below the tensor-core time.
// Measured, the pair is slower than the single-SM kernel on the shapes tried
// (a 128-key tile every 2.0 us against 1.5 us: each P V waits for the softmax
// of both halves, and Q K_{j+2} for P_j V_j, across the two SMs), so it runs
// only when asked for (EXTKV_ALGO_PREFILL_PAIR).
//
// Layout of the work: cluster (b, head pair, tile of 128 query rows); CTA
// rank r (0 or 1) holds query head 2m + r: its Q tile, its S and O in its own
// tensor memory (128 lanes), its softmax.  The even CTA's MMA thread issues
//   S_j  = Q K_j^T  M=256, N=128 keys (64 in each CTA's shared memory), K=256
//   O   += P_j V_j  M=256, N=256 (128 columns of V in each CTA), K=128 keys
// and commits to the same barrier in both CTAs (multicast).  Each CTA's
// producer loads its halves with TMA onto its own barriers; the odd CTA's
// warp 1 relays each landing to the even CTA's barrier, so the MMA thread
// knows both halves are there and each CTA can still wait for its own copies
// before it exits.  The softmax warps of both CTAs release P_j on the even
// CTA's barrier.  The two heads of a pair see the same query positions, so
// their allowed keys (and dead V rows) are the same.
//
// The scores, masking, online softmax, zero rows and epilogue are those of
// the single-SM kernel (attn_prefill.cuh).
#pragma once

#include "attn_prefill.cuh"

namespace extkv {

namespace {

template <int MODE>
struct PairCfg {
  static constexpr bool kTerm = MODE == kBias || MODE == kFusedExtra;
  static constexpr int kThreads = 192;  // producer, MMA (relay in the odd CTA), 4 softmax warps
  static constexpr int kUnitBytes = 32 * 1024;  // a K half (64 keys x 256) or a V half (128 keys x 128)
  static constexpr int kQBytes = kBM * 256 * 2;
  static constexpr int kTermBytes = kTerm ? kBM * kBN * 2 : 0;
  static constexpr int kTermBufs = kTerm ? 1 : 0;
  static constexpr int kBudget = 232448 - 1024 - 1024;
  static constexpr int kFit = (kBudget - kQBytes - kTermBufs * kTermBytes) / kUnitBytes;
  static constexpr int kNU = kFit > kMaxUnits ? kMaxUnits : kFit;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffT = kOffKV + kNU * kUnitBytes;
  static constexpr int kOffBar = kOffT + kTermBufs * kTermBytes;
  static constexpr int kSmem = kOffBar + 1024 + 1024;
  static constexpr uint32_t kOCol = 256;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(2 * kBM, kBN, 0, 0);
  static constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(2 * kBM, 256, 0, 1);
  static_assert(kNU >= 3, "shared memory holds fewer than three load units");
  static_assert(kNU * kUnitBytes >= 4 * 4 * 4096, "the epilogue stages 128 rows x 256 in the K/V ring");
};

struct PairBars {
  uint64_t q_full;                                  // own Q landed (+ the peer's relay, even CTA)
  uint64_t u_full[kMaxUnits], u_empty[kMaxUnits];   // own half landed (+ relay) / slot free in both
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t v_ready[2];
  uint64_t t_full[2], t_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int range_lo, range_hi;
  int abort;
};
static_assert(sizeof(PairBars) <= 1024, "barrier block");

template <int MODE, bool CAP>
__global__ void __launch_bounds__(PairCfg<MODE>::kThreads, 1)
    attn_prefill_pair_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap tmap,
                             const __grid_constant__ CUtensorMap ymap, const PrefillParams p) {
  using C = PairCfg<MODE>;
  constexpr int DV = 256;
  constexpr bool kFusedMode = MODE == kFused || MODE == kFusedExtra;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sKV = sm + C::kOffKV;
  uint8_t* sT = sm + C::kOffT;
  PairBars& bar = *reinterpret_cast<PairBars*>(sm + C::kOffBar);
  volatile int* abort = &bar.abort;
  const uint32_t lim = p.polls;  // pipeline waits; the drains keep the full limit

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;
  const int h = blockIdx.x, pt = blockIdx.y, b = blockIdx.z;  // head h = 2m + rank
  const int g = p.Hq / p.Hkv;
  const int hk = h / g;
  const int q0 = pt * kBM;

  if (tid == 0) {
    // the even CTA's full barriers also count the odd CTA's relay
    ptx::mbar_init(&bar.q_full, leader ? 2 : 1);
    for (int s = 0; s < C::kNU; ++s) {
      ptx::mbar_init(&bar.u_full[s], leader ? 2 : 1);
      ptx::mbar_init(&bar.u_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar.s_full[s], 1);
      ptx::mbar_init(&bar.p_full[s], 2 * 4);  // one per softmax warp of each CTA
      ptx::mbar_init(&bar.pv_done[s], 1);
      ptx::mbar_init(&bar.v_ready[s], 1);
      ptx::mbar_init(&bar.t_full[s], 1);
      ptx::mbar_init(&bar.t_empty[s], 4);
    }
    ptx::mbar_init(&bar.drain, 1);
    bar.range_lo = INT_MAX;
    bar.range_hi = 0;
    bar.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&qmap);
    ptx::prefetch_tensormap(&kmap);
    ptx::prefetch_tensormap(&vmap);
    if (C::kTerm) ptx::prefetch_tensormap(&tmap);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&bar.tmem_base, C::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncwarp();  // every warp converged at the (aligned) cluster barrier
  // both CTAs' barriers exist before either signals the other
  ptx::cluster_sync();
  ptx::tc_fence_after();
  ptx::grid_dependency_wait();  // the preceding kernels' writes (cache, bias, plan) are visible

  if (warp == 0 && lane == 0) {
    ptx::mbar_arrive_expect_tx(&bar.q_full, C::kQBytes);
    ptx::tma_load_3d(sQ, &qmap, &bar.q_full, 0, (b * p.Hq + h) * p.S_q + q0, 0);
  }

  const int64_t np64 = p.nonpad[b];
  const bool bad = bad_nonpad(np64, p.max_seq);
  if (bad && tid == 0 && h == 0 && pt == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int64_t qs = bad ? 0 : query_start(p.spec.q_start, b, np64, p.S_q);
  const uint64_t* cmrow = C::kTerm ? p.colmask + (static_cast<int64_t>(b) * p.n_pt + pt) * p.n_tiles : nullptr;
  const int64_t imp0 = MODE == kBias ? (static_cast<int64_t>(b) * p.n_pt + pt) * p.n_kt : 0;

  // softmax threads: this thread's query row and its allowed key intervals
  const bool is_sm = warp >= 2;
  const int row = 32 * (warp & 3) + lane;
  const bool row_valid = is_sm && q0 + row < p.S_q;
  int a1 = 0, b1 = np, a2 = 0, b2 = 0;  // allowed keys: [a1, b1) U [a2, b2)
  if (kFusedMode && is_sm) {
    const RowWindow w = row_window(p.spec, b, qs + q0 + row, np);
    const int64_t bl = w.band_lo < 0 ? 0 : w.band_lo, bh = w.band_hi < np ? w.band_hi : np;
    const int64_t sl = w.span_lo < 0 ? 0 : w.span_lo, sh = w.span_hi < np ? w.span_hi : np;
    a1 = static_cast<int>(bl < bh ? bl : 0);
    b1 = static_cast<int>(bl < bh ? bh : 0);
    a2 = static_cast<int>(sl < sh ? sl : 0);
    b2 = static_cast<int>(sl < sh ? sh : 0);
    if (MODE == kFused && row_valid) {
      int lo = INT_MAX, hi = 0;
      if (a1 < b1) {
        lo = a1;
        hi = b1;
      }
      if (a2 < b2) {
        lo = min(lo, a2);
        hi = max(hi, b2);
      }
      if (lo < hi) {
        atomicMin(&bar.range_lo, lo);
        atomicMax(&bar.range_hi, hi);
      }
    }
  }
  if (MODE == kNone) {
    if (tid == 0 && np > 0) {
      bar.range_lo = 0;
      bar.range_hi = np;
    }
  } else if (C::kTerm && warp == 1) {
    // first and last 64-key block with a live key in the plan's column masks
    int lo = INT_MAX, hi = 0;
    const int nw = (np + 63) / 64;
    for (int t = lane; t < nw; t += 32)
      if (cmrow[t]) {
        lo = min(lo, t);
        hi = max(hi, t + 1);
      }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0 && lo < hi) {
      bar.range_lo = lo * 64;
      bar.range_hi = min(hi * 64, np);
    }
  }
  __syncthreads();
  // the two CTAs compute the same range (the same query positions)
  const int rlo = bar.range_lo, rhi = bar.range_hi;
  const int t_lo = rlo < rhi ? rlo / kBN : 0;
  const int T = rlo < rhi ? (rhi + kBN - 1) / kBN - t_lo : 0;  // KV tiles of the query tile
  const uint32_t tbase = bar.tmem_base;
  const uint32_t peer_q_full = ptx::map_cluster(&bar.q_full, 0);

  if (warp == 0) {
    // ---------------- TMA producer: this CTA's halves ----------------
    if (lane == 0) {
      const int unit = b * p.Hkv + hk;
      int issued = 0, t_issued = 0;
      bool ok = true;
      bool imp_next = MODE != kBias || (T > 0 && p.impure[imp0 + t_lo] != 0);
      auto load_term = [&](int j) -> bool {
        const bool imp = imp_next;
        if (MODE == kBias && j + 1 < T) imp_next = p.impure[imp0 + t_lo + j + 1] != 0;
        if (!imp) return true;  // the row bits suffice
        const int tb = t_issued % 1;
        if (t_issued >= 1 && !wait_or_abort(&bar.t_empty[tb], (t_issued - 1) & 1, abort, lim)) return false;
        uint8_t* dst = sT;
        ptx::mbar_arrive_expect_tx(&bar.t_full[tb], C::kTermBytes);
        ptx::tma_load_2d(dst, &tmap, &bar.t_full[tb], (t_lo + j) * kBN, b * p.S_q + q0);
        ptx::tma_load_2d(dst + C::kTermBytes / 2, &tmap, &bar.t_full[tb], (t_lo + j) * kBN + 64, b * p.S_q + q0);
        ++t_issued;
        return true;
      };
      for (int idx = 0; idx < 2 * T && ok; ++idx) {
        const bool is_v = idx == 2 * T - 1 ? true : (idx == 0 ? false : (idx & 1) == 0);
        const int j = idx == 2 * T - 1 ? T - 1 : (is_v ? idx / 2 - 1 : (idx + 1) / 2);
        const int key0 = (t_lo + j) * kBN;
        const int u = issued, slot = u % C::kNU;  // units leave in sequence order
        if (u >= C::kNU && !wait_or_abort(&bar.u_empty[slot], ((u / C::kNU) - 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        uint8_t* dst = sKV + slot * C::kUnitBytes;
        ptx::mbar_arrive_expect_tx(&bar.u_full[slot], C::kUnitBytes);
        if (is_v)  // 128 keys x this CTA's 128 value columns
          ptx::tma_load_4d(dst, &vmap, &bar.u_full[slot], 0, key0, 2 * static_cast<int>(rank), unit);
        else  // this CTA's 64 keys x 256
          ptx::tma_load_4d(dst, &kmap, &bar.u_full[slot], 0, key0 + 64 * static_cast<int>(rank), 0, unit);
        ++issued;
        if (C::kTerm) {
          if (idx == 0) ok = load_term(0);
          else if (is_v && j + 1 < T) ok = load_term(j + 1);
        }
      }
      // the copies still in flight land before the CTA leaves (the newest
      // request of each slot; older phases are complete)
      ptx::mbar_wait_bounded(&bar.q_full, 0, kWaitPolls);
      for (int u = issued > C::kNU ? issued - C::kNU : 0; u < issued; ++u)
        ptx::mbar_wait_bounded(&bar.u_full[u % C::kNU], (u / C::kNU) & 1, kWaitPolls);
      if (C::kTerm && t_issued > 0) ptx::mbar_wait_bounded(&bar.t_full[0], (t_issued - 1) & 1, kWaitPolls);
    }
  } else if (warp == 1) {
    if (!leader) {
      // ---------------- relay (odd CTA): each own landing onto the even CTA's barrier ----------------
      if (lane == 0) {
        bool ok = wait_or_abort(&bar.q_full, 0, abort, lim);
        if (ok) ptx::mbar_arrive_cluster(peer_q_full);
        for (int u = 0; u < 2 * T && ok; ++u) {
          const int slot = u % C::kNU;
          if (!(ok = wait_or_abort(&bar.u_full[slot], (u / C::kNU) & 1, abort, lim))) break;
          ptx::mbar_arrive_cluster(ptx::map_cluster(&bar.u_full[slot], 0));
        }
      }
    } else if (lane == 0 && T > 0) {
      // ---------------- MMA issuer (even CTA) ----------------
      const uint32_t kv_addr = ptx::smem_u32(sKV), q_addr = ptx::smem_u32(sQ);
      const uint64_t kdesc0 = ptx::smem_desc_sw128(kv_addr, 16, 1024);
      const uint64_t vdesc0 = ptx::smem_desc_sw128(kv_addr, kBN * 128, 1024);
      const uint64_t qdesc0 = ptx::smem_desc_sw128(q_addr, 16, 1024);
      const uint32_t peer_v_ready0 = ptx::map_cluster(&bar.v_ready[0], 1), peer_v_ready1 = ptx::map_cluster(&bar.v_ready[1], 1);
      // Readiness tests of the next steps, placed a few MMAs before the end of
      // the current batch (the issuing thread blocks while the tensor pipe's
      // queue is full, so a test there overlaps its round trip with queued
      // work); the blocking waits remain for what is not there yet.
      auto k_ready = [&](int j) -> bool {
        const int u = k_unit<1, 1>(j);
        return ptx::mbar_test_wait(&bar.u_full[u % C::kNU], (u / C::kNU) & 1);
      };
      auto pv_ready = [&](int j) -> bool {
        const int u = v_unit<1, 1>(j, T);
        bool r = ptx::mbar_test_wait(&bar.p_full[j & 1], (j >> 1) & 1);
        r = ptx::mbar_test_wait(&bar.u_full[u % C::kNU], (u / C::kNU) & 1) && r;
        return r;
      };
      bool k_known = false, pv_known = false;
      // Q K_j^T into S_{j & 1}; tests P_pj / V_pj on the way when pj >= 0
      auto issue_qk = [&](int j, int pj) -> bool {
        const int u = k_unit<1, 1>(j), slot = u % C::kNU;
        if (!k_known && !wait_or_abort(&bar.u_full[slot], (u / C::kNU) & 1, abort, lim)) return false;
        k_known = false;
        ptx::tc_fence_after();
        const uint32_t d = tbase + (j & 1) * kBN;
        const uint64_t kd = kdesc0 + ((slot * C::kUnitBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {  // K steps of 16 over the head dim
          const uint64_t ad = qdesc0 + (((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
          const uint64_t bd = kd + (((kk >> 2) * (64 * 128) + (kk & 3) * 32) >> 4);
          ptx::umma_bf16_pair(d, ad, bd, C::kIdescQK, kk > 0);
          if (pj >= 0 && kk == 12) pv_known = pv_ready(pj);
        }
        ptx::umma_commit_pair(&bar.u_empty[slot]);
        ptx::umma_commit_pair(&bar.s_full[j & 1]);
        return true;
      };
      bool ok = wait_or_abort(&bar.q_full, 0, abort, lim);  // both Q tiles
      if (ok) {
        ptx::tc_fence_after();
        ok = issue_qk(0, -1);
      }
      for (int j = 0; j < T && ok; ++j) {
        pv_known = false;
        if (j + 1 < T && !(ok = issue_qk(j + 1, j))) break;
        const int u = v_unit<1, 1>(j, T), slot = u % C::kNU;
        if (!pv_known && !(ok = wait_or_abort(&bar.u_full[slot], (u / C::kNU) & 1, abort, lim))) break;
        // V_j landed in both CTAs: their softmax warps may zero its dead rows
        ptx::mbar_arrive(&bar.v_ready[j & 1]);
        ptx::mbar_arrive_cluster((j & 1) ? peer_v_ready1 : peer_v_ready0);
        if (!pv_known && !(ok = wait_or_abort(&bar.p_full[j & 1], (j >> 1) & 1, abort, lim))) break;
        ptx::tc_fence_after();
        const uint64_t vd = vdesc0 + ((slot * C::kUnitBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {  // K steps of 16 keys
          ptx::umma_bf16_ts_pair(tbase + C::kOCol, tbase + (j & 1) * kBN + ks * 8, vd + ((ks * 2048) >> 4),
                                 C::kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
          if (j + 2 < T && ks == kBN / 16 - 3) k_known = k_ready(j + 2);
        }
        ptx::umma_commit_pair(&bar.u_empty[slot]);
        ptx::umma_commit_pair(&bar.pv_done[j & 1]);
      }
      // every MMA issued has completed before tensor memory is released
      ptx::umma_commit_pair(&bar.drain);
      if (!ptx::mbar_wait_bounded(&bar.drain, 0, kWaitPolls)) *abort = 1;
    }
  } else {
    // ---------------- softmax and epilogue (one query row per thread) ----------------
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const float sc = p.scale;
    const float lowest = Elem<__nv_bfloat16>::lowest();
    const uint32_t peer_p_full0 = ptx::map_cluster(&bar.p_full[0], 0), peer_p_full1 = ptx::map_cluster(&bar.p_full[1], 0);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int t_seen = 0;  // term blocks consumed
    bool pure_next = MODE == kBias && T > 0 && p.impure[imp0 + t_lo] == 0;
    for (int j = 0; j < T; ++j) {
      const int tile = t_lo + j, key0 = tile * kBN;
      const bool pure = pure_next;
      if (MODE == kBias && j + 1 < T) pure_next = p.impure[imp0 + tile + 1] == 0;
      uint64_t dead0, dead1;
      if (C::kTerm) {
        dead0 = ~cmrow[2 * tile];
        dead1 = 2 * tile + 1 < p.n_tiles ? ~cmrow[2 * tile + 1] : ~0ull;
      } else {
        dead0 = ~bit_range(rlo - key0, rhi - key0);
        dead1 = ~bit_range(rlo - key0 - 64, rhi - key0 - 64);
      }
      uint64_t al0, al1;
      if (pure) {
        const uint4 rb = *reinterpret_cast<const uint4*>(
            p.rowmask + ((static_cast<int64_t>(b) * p.n_pt + pt) * kBM + row) * p.rm_stride + tile * 16);
        al0 = rb.x | (static_cast<uint64_t>(rb.y) << 32);
        al1 = rb.z | (static_cast<uint64_t>(rb.w) << 32);
      } else if (kFusedMode) {
        al0 = bit_range(a1 - key0, b1 - key0) | bit_range(a2 - key0, b2 - key0);
        al1 = bit_range(a1 - key0 - 64, b1 - key0 - 64) | bit_range(a2 - key0 - 64, b2 - key0 - 64);
      } else {
        al0 = bit_range(-key0, np - key0);
        al1 = bit_range(-key0 - 64, np - key0 - 64);
      }
      const bool part0 = !__all_sync(0xffffffffu, al0 == ~0ull);
      const bool part1 = !__all_sync(0xffffffffu, al1 == ~0ull);
      if (!__all_sync(0xffffffffu, wait_or_abort(&bar.s_full[j & 1], (j >> 1) & 1, abort, lim))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t ts = tl + (j & 1) * kBN;
      float t[kBN];
      {
        const bool termed = C::kTerm && !pure;
        const uint8_t* tblk = sT;
        if (termed && !__all_sync(0xffffffffu, wait_or_abort(&bar.t_full[0], t_seen & 1, abort, lim))) {
          ok = false;
          break;
        }
        if (termed) ++t_seen;
        uint32_t sa[32], sb[32], tw[32];
        ptx::tmem_ld32(ts, sa);
        ptx::tmem_ld32(ts + 32, sb);
        if (termed) load_swizzled_row(tw, tblk, row);
        ptx::tmem_wait_ld();
        if constexpr (CAP) {
          if (termed) {
            if (part0) half_scores_capped<0, true, true>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
            else half_scores_capped<0, true, false>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
          } else if (part0) {
            half_scores_capped<0, false, true>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
          } else {
            half_scores_capped<0, false, false>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
          }
        } else if (termed) {
          if (part0) half_scores<0, true, true>(t, sa, sb, tw, al0, sc, lowest);
          else half_scores<0, true, false>(t, sa, sb, tw, al0, sc, lowest);
        } else if (part0) {
          half_scores<0, false, true>(t, sa, sb, tw, al0, sc, lowest);
        } else {
          half_scores<0, false, false>(t, sa, sb, tw, al0, sc, lowest);
        }
        ptx::tmem_ld32(ts + 64, sa);
        ptx::tmem_ld32(ts + 96, sb);
        if (termed) {
          load_swizzled_row(tw, tblk + C::kTermBytes / 2, row);
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bar.t_empty[0]);
        }
        ptx::tmem_wait_ld();
        if constexpr (CAP) {
          if (termed) {
            if (part1) half_scores_capped<1, true, true>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
            else half_scores_capped<1, true, false>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
          } else if (part1) {
            half_scores_capped<1, false, true>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
          } else {
            half_scores_capped<1, false, false>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
          }
        } else if (termed) {
          if (part1) half_scores<1, true, true>(t, sa, sb, tw, al1, sc, lowest);
          else half_scores<1, true, false>(t, sa, sb, tw, al1, sc, lowest);
        } else if (part1) {
          half_scores<1, false, true>(t, sa, sb, tw, al1, sc, lowest);
        } else {
          half_scores<1, false, false>(t, sa, sb, tw, al1, sc, lowest);
        }
      }
      const float mt = tile_max(t);
      // lazy rescale: only when the running maximum grows by more than 8 ln 2
      const float m_new = fmaxf(m_run, mt);
      const bool grow = m_new > m_run + kRescaleGrow;  // false while the row has no unmasked key
      const bool rescale_o = grow && m_run != -INFINITY;
      const float factor = rescale_o ? ptx::ex2((m_run - m_new) * kLog2e) : 1.f;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // the output accumulator holds P_{j-1} V_{j-1} once that product completes
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, lim))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tl + C::kOCol + 32 * c, o);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          ptx::tmem_st32(tl + C::kOCol + 32 * c, o);
        }
        ptx::tmem_wait_st();
      }
      if (grow) {
        l_run *= factor;
        m_run = m_new;
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      uint64_t ls[4] = {0, 0, 0, 0};
      // P_j over the first half of S_j (this CTA's tensor memory): QK_{j+2},
      // the next writer of this buffer, is issued after P_j V_j
      {
        uint32_t pk[32];
        exp_pairs<0>(t, m_use, pk, ls);
        ptx::tmem_st32(ts, pk);
      }
      {
        uint32_t pk[32];
        exp_pairs<64>(t, m_use, pk, ls);
        ptx::tmem_st32(ts + 32, pk);
      }
      const uint64_t lsum = ptx::add2(ptx::add2(ls[0], ls[1]), ptx::add2(ls[2], ls[3]));
      l_run += ptx::f2_lo(lsum) + ptx::f2_hi(lsum);
      if (dead0 | dead1) {
        // zero the dead keys' rows of this CTA's half of V_j once it has
        // landed in both CTAs (the MMA thread says so)
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.v_ready[j & 1], (j >> 1) & 1, abort, lim))) {
          ok = false;
          break;
        }
        const int slot = v_unit<1, 1>(j, T) % C::kNU;
        uint8_t* vt = sKV + slot * C::kUnitBytes;
        constexpr int kLines = kBN * 2 * 8;  // 16-byte pieces: 128 keys x 2 chunks x 8
        for (int w = tid - 64; w < kLines; w += 128) {
          const int key = w >> 4, rem = w & 15;
          const uint64_t dm = key < 64 ? dead0 : dead1;
          if ((dm >> (key & 63)) & 1)
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kBN * 128) + key * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        ptx::fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      // P_j of this warp's rows (and its dead V rows) ready: on the even CTA's barrier
      if (lane == 0) {
        if (leader) ptx::mbar_arrive(&bar.p_full[j & 1]);
        else ptx::mbar_arrive_cluster((j & 1) ? peer_p_full1 : peer_p_full0);
      }
    }
    // epilogue: O / l, zero rows without an unmasked key
    if (ok && T > 0 &&
        !__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort, lim)))
      ok = false;
    ptx::tc_fence_after();
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    constexpr int kNB = DV / 64;  // 64-column blocks
    // the warp's 32 rows through shared memory (the K/V ring is idle: every
    // MMA that read either CTA's ring has completed), one TMA store per block
    uint8_t* stage = sKV + (warp & 3) * kNB * 4096;
#pragma unroll 1
    for (int cb = 0; cb < kNB; ++cb) {
      uint32_t o[64];
      if (ok && T > 0) {
        ptx::tmem_ld32(tl + C::kOCol + 64 * cb, *reinterpret_cast<uint32_t(*)[32]>(o));
        ptx::tmem_ld32(tl + C::kOCol + 64 * cb + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
        ptx::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) o[e] = 0;
      }
      uint8_t* blk = stage + cb * 4096 + lane * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv, __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
        *reinterpret_cast<uint4*>(blk + ((q ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    ptx::fence_proxy_async_smem();  // the staged rows, visible to the TMA store
    __syncwarp();
    if (ok && lane == 0 && q0 + 32 * (warp & 3) < p.S_q) {  // a box wholly past S_q writes nothing
      for (int cb = 0; cb < kNB; ++cb)
        ptx::tma_store_3d(&ymap, stage + cb * 4096, cb * 64, q0 + 32 * (warp & 3), b * p.Hq + h);
      ptx::bulk_commit_group();
      ptx::bulk_wait_read_all();  // shared memory stays valid until the stores have read it
    }
    __syncwarp();
  }
  ptx::grid_launch_dependents();
  if (tid == 0 && *abort) report(p.status, EXTKV_DEV_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  __syncwarp();
  // neither CTA leaves (or frees tensor memory) while the other may still
  // signal it or read its shared memory
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tbase, C::kTmemCols);
}

// Launch of the pair kernel: D = Dk = Dv = 256, an even number of query heads
// per KV head, no key splits.
template <int MODE, bool CAP>
cudaError_t launch_pair(const AttnArgs& a, const char** name) {
  using C = PairCfg<MODE>;
  if (cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_prefill_pair_kernel<MODE, CAP>),
                                           C::kSmem);
      e != cudaSuccess)
    return e;
  CUtensorMap qmap, kmap, vmap, tmap, ymap;
  const uint64_t units = static_cast<uint64_t>(a.B * a.Hkv);
  const uint64_t k_dims[4] = {64, static_cast<uint64_t>(a.max_seq), 4, units};
  const uint64_t k_strides[3] = {512, 128, static_cast<uint64_t>(a.max_seq) * 512};
  const uint32_t k_box[4] = {64, 64, 4, 1};   // 64 keys x 256
  const uint32_t v_box[4] = {64, 128, 2, 1};  // 128 keys x 128 columns
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 4, k_dims, k_strides, k_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 4, k_dims, k_strides, v_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t q_dims[3] = {64, static_cast<uint64_t>(a.B * a.Hq * a.S_q), 4};
  const uint64_t q_strides[2] = {512, 128};
  const uint32_t q_box[3] = {64, kBM, 4};
  if (!make_tensor_map_bf16(&qmap, a.q, 3, q_dims, q_strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t y_dims[3] = {256, static_cast<uint64_t>(a.S_q), static_cast<uint64_t>(a.B * a.Hq)};
  const uint64_t y_strides[2] = {512, static_cast<uint64_t>(a.S_q) * 512};
  const uint32_t y_box[3] = {64, 32, 1};
  if (!make_tensor_map_bf16(&ymap, a.y, 3, y_dims, y_strides, y_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  std::memset(&tmap, 0, sizeof tmap);
  const void* term = MODE == kBias ? a.bias : (MODE == kFusedExtra ? a.extra : nullptr);
  if (term) {
    const uint64_t t_dims[2] = {static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(a.B * a.S_q)};
    const uint64_t t_strides[1] = {static_cast<uint64_t>(a.max_seq) * 2};
    const uint32_t t_box[2] = {64, kBM};
    if (!make_tensor_map_bf16(&tmap, term, 2, t_dims, t_strides, t_box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  PrefillParams prm;
  std::memset(&prm, 0, sizeof prm);
  if (cudaError_t e = prefill_setup(a, MODE, 256, &prm); e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.Hq), static_cast<unsigned>(prm.n_pt), static_cast<unsigned>(a.B));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_prefill_pair_kernel<MODE, CAP>, qmap, kmap, vmap, tmap, ymap, prm);
  if (e != cudaSuccess) return e;
  *name = "attn_prefill_tcgen05_pair";
  note_launches(C::kTerm ? 2 : 1);
  return cudaGetLastError();
}

}  // namespace

}  // namespace extkv
