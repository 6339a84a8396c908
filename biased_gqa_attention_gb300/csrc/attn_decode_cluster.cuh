// attn_decode_cluster.cuh -- decode attention for calls whose units fit the
// GPU at once: thread-block clusters per (batch, KV head, row group).
//
// The stream-K decode (attn_decode.cuh) balances any number of units over a
// fixed grid, at the price of a plan kernel (a materialised bias), per-batch
// tables of the whole call in every CTA and a merge kernel: fixed costs that
// dominate a call of a few tens of MB ("Skill: Attention Optimization":
// decode is memory-bandwidth bound, so what is not streaming is overhead).
// When every unit can hold a cluster of C CTAs resident at once, this kernel
// removes all three (the merge stays only where a unit is split over several
// clusters):
//
//   Unit: one (batch b, KV head, row group): up to 8 of the KV head's
//     GR = (Hq/Hkv) * S_q <= 64 query rows (GQA by reshaping Q, "ONNX Domain
//     Attention (Opset 23/24) CUDA Patterns", section 1); the row groups of a
//     KV head read the same tiles.  A cluster of C one-warp CTAs (C <= 8) per
//     unit.
//   Live tiles: every CTA of the unit finds the unit's live 16-key tiles by
//     itself -- without a bias, the tiles below nonpad; with the fused
//     specification, the closed-form runs of the rows' allowed intervals;
//     with a materialised bias, one bulk copy of the batch's S_q bias rows,
//     multicast by the cluster's first CTA into every CTA's shared memory,
//     and a scan (a tile is live when some key below nonpad has a bias above
//     lowest(T), section 6 of the ORT page).
//   Streaming: CTA r of the cluster takes the r-th of C equal contiguous
//     shares of the live tiles (of its cluster's block, below) and streams them with the stream-K kernel's
//     per-tile pipeline (TMA K/V stages, mma.sync QK^T and PV, online
//     softmax in natural units, dead keys' V rows zeroed).
//   Combine: each CTA leaves (max, sum, unnormalised output) of its share in
//     its own shared memory; after a cluster barrier CTA r reads column block
//     r of every share through distributed shared memory and writes those
//     columns of Y, combining the shares in rank order (the result does not
//     depend on timing); a second barrier keeps every CTA's shared memory
//     alive until its peers have read it.  A row with no unmasked key in any
//     share is written as zeros.
//   Few units (one long sequence, say): M clusters per unit, cluster m taking
//     the m-th of M blocks of the unit's live tiles; each cluster's combine
//     writes one partial (max, sum, unnormalised output) in the stream-K
//     kernel's layout instead of Y, and the stream-K merge kernel combines the
//     M partials in order.
#pragma once

#include "attn_decode.cuh"

namespace extkv {
namespace {

constexpr int kMaxCluster = 8;                  // portable cluster size
constexpr int kScanBytes = 16 * 1024;           // bias rows one CTA scans (S_q * max_seq * 2)
constexpr int kMaxListTiles = kScanBytes / 32;  // live-tile list of one unit

// Stages of a cluster decode CTA's ring: as many as keep four CTAs on an SM
// (a unit's eight CTAs of the decode workload's 64 units resident at once).
template <int D>
struct ClusterCfg;
template <>
struct ClusterCfg<64> {
  static constexpr int SPW = 4;
};
template <>
struct ClusterCfg<128> {
  static constexpr int SPW = 4;
};
template <>
struct ClusterCfg<256> {
  static constexpr int SPW = 3;
};
template <>
struct ClusterCfg<512> {
  static constexpr int SPW = 2;
};

// Shared memory of a cluster decode CTA.  The stage ring doubles as the
// buffer of the bias rows, which are scanned before the first K/V request,
// and, once every copy into it has landed, as the share's unnormalised O.
template <int DK, int DV, int SPW>
struct CSmem {
  using S = Smem<DK, DV, SPW>;
  static constexpr int kStages = SPW * S::kStageBytes;
  static_assert(kStages >= kScanBytes, "the stage ring holds the scanned bias rows");
  static_assert(kStages >= kRows * DV * 4, "the stage ring holds the share's O");
  static constexpr int kQ = kStages;                               // Q slot (DK = 512)
  static constexpr int kTerm = kQ + (S::kQReg ? 0 : S::kQBytes);   // per stage: S_q rows x 16 keys
  static constexpr int kPart = kTerm + SPW * 256;                  // fp32 max[8], sum[8]
  static constexpr int kList = kPart + 2 * kRows * 4;              // uint16 live tiles
  static constexpr int kBars = kList + kMaxListTiles * 2;          // SPW stages, Q, scan
  static constexpr int kEnd = kBars + (SPW + 2) * 8;
  static constexpr size_t bytes() { return 1024 + kEnd; }
};

// Whether any of 8 bf16 values is above lowest(bf16), i.e. unmasked.
__device__ __forceinline__ bool any_above_lowest(const uint4 v) {
  const __nv_bfloat162 lo2 = __halves2bfloat162(__ushort_as_bfloat16(Elem<__nv_bfloat16>::kLowestBits),
                                                  __ushort_as_bfloat16(Elem<__nv_bfloat16>::kLowestBits));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 x;
    *reinterpret_cast<uint32_t*>(&x) = w[i];
    const __nv_bfloat162 c = __hgt2(x, lo2);  // 1.0 where x > lowest
    r |= *reinterpret_cast<const uint32_t*>(&c);
  }
  return r != 0;
}

template <int DK, int DV, int SPW, int MODE, bool CAP>
__global__ void __launch_bounds__(32) attn_decode_cluster_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap tmap,
    const DecodeParams p, const int C, const int M) {
  using S = Smem<DK, DV, SPW>;
  using L = CSmem<DK, DV, SPW>;
  constexpr bool kOneSize = DK == DV;  // the fused scatter takes one head size
  constexpr bool kTerm = MODE == kBias || MODE == kFusedExtra;  // per-tile bias block
  constexpr bool kQReg = S::kQReg;
  constexpr int kKSteps = DK / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* qbar = bars + SPW;
  uint64_t* sbar = bars + SPW + 1;
  float* pm = reinterpret_cast<float*>(smem + L::kPart);  // max of each row
  float* pl = pm + kRows;                                  // sum of each row
  float* po = reinterpret_cast<float*>(smem);              // unnormalised O [kRows][DV], over the ring
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  const int lane = threadIdx.x;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int cl = static_cast<int>(blockIdx.x) / C;  // cluster
  const int unit = cl / M, m = cl - unit * M;        // the unit, and which of its M clusters
  const int bh = unit / p.n_rg, rg = unit - bh * p.n_rg;  // bh: the K/V views' unit coordinate
  const int b = bh / p.Hkv, kvh = bh - b * p.Hkv;
  const float lowest = Elem<__nv_bfloat16>::lowest();
  const int max_seq = p.max_seq;

  if (lane == 0) {
    for (int s = 0; s < SPW + 2; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&kmap);
    ptx::prefetch_tensormap(&vmap);
    if (!kQReg) ptx::prefetch_tensormap(&qmap);
    if (kTerm) ptx::prefetch_tensormap(&tmap);
  }
  __syncwarp();
  // every CTA's barriers are initialised before the first CTA multicasts into them
  // (the CTAs would wait for the previous kernel here anyway)
  if (MODE == kBias) ptx::cluster_sync();
  // Nothing above reads an input; everything below may read what the
  // previous kernel in the stream wrote.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  // the batch's bias rows: one bulk copy by the first CTA, delivered to all
  // (issued before nonpad is known); each CTA's barrier expects the bytes
  if (MODE == kBias && lane == 0) {
    const uint32_t bytes = static_cast<uint32_t>(p.S_q) * static_cast<uint32_t>(max_seq) * 2u;
    ptx::mbar_arrive_expect_tx(sbar, bytes);
    if (rank == 0 && EXTKV_IN(static_cast<int64_t>(b) * p.S_q * max_seq, static_cast<int64_t>(p.S_q) * max_seq,
                              static_cast<int64_t>(p.B) * p.S_q * max_seq, p.status))
      ptx::bulk_load_multicast(smem, p.bias + static_cast<int64_t>(b) * p.S_q * max_seq, bytes, sbar,
                               static_cast<uint16_t>((1u << C) - 1u));
  }
  const int64_t np64 = EXTKV_IN(b, 1, p.B, p.status) ? p.nonpad[b] : 0;
  const bool bad = bad_nonpad(np64, max_seq);
  if (bad && kvh == 0 && rg == 0 && m == 0 && rank == 0 && lane == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int n_range = (np + kTile - 1) / kTile;

  // this lane's two query rows of the unit (row r of group rg is the KV head's
  // row 8 rg + r: head (8 rg + r) / S_q of the group, position (8 rg + r) % S_q),
  // and the unit's first row of Y
  const int R = min(kRows, p.GR - rg * kRows);
  const int64_t row0 =
      (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(kvh) * p.g) * p.S_q + rg * kRows;
  const int r0 = 2 * (lane & 3), r1 = r0 + 1;
  const bool ok0 = r0 < R, ok1 = r1 < R;
  const int i0 = (rg * kRows + r0) % p.S_q, i1 = (rg * kRows + r1) % p.S_q;

  // Q: mma B fragments in registers (DK <= 256), else one TMA box in shared memory
  uint32_t qf[kQReg ? kKSteps : 1][2];
  if constexpr (kQReg) {
    // B fragment of k-step ks: the bf16 pair at (row lane/4, d = 16 ks + 2 (lane%4)), and d + 8
    const int row = lane >> 2;
    const bool qok = row < R && EXTKV_IN(row0 + row, 1, static_cast<int64_t>(p.B) * p.Hq * p.S_q, p.status);
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(p.q + (row0 + row) * static_cast<int64_t>(DK)) + (lane & 3);
#pragma unroll
    for (int ks = 0; ks < kKSteps; ++ks) {
      qf[ks][0] = qok ? __ldg(qrow + 8 * ks) : 0u;
      qf[ks][1] = qok ? __ldg(qrow + 8 * ks + 4) : 0u;
    }
  } else if (lane == 0) {
    ptx::mbar_arrive_expect_tx(qbar, S::kQBytes);
    ptx::tma_load_3d(smem + L::kQ, &qmap, qbar, 0, static_cast<int32_t>(row0), 0);
  }

  // ---- the unit's live tiles ----
  bool failed = false;
  int n_live = 0;
  Runs runs{0, 0, 0, 0};
  if (MODE == kNone) {
    n_live = n_range;
  } else if (MODE == kFused || MODE == kFusedExtra) {
    runs = batch_runs<MODE>(p, b, np64);
    n_live = runs.count();
  } else {
    if (__any_sync(0xffffffffu, !ptx::mbar_wait_spin_bounded(sbar, 0, p.polls))) {
      failed = true;
    } else {
      for (int t0 = 0; t0 < n_range; t0 += 32) {
        const int t = t0 + lane;
        bool live = false;
        if (t < n_range) {
          const int j0 = t * kTile;
          for (int i = 0; i < p.S_q && !live; ++i) {
            const uint16_t* row = reinterpret_cast<const uint16_t*>(smem + static_cast<size_t>(i) * max_seq * 2);
            if (j0 + kTile <= np) {
              // a whole tile below nonpad: 8 packed comparisons (NaN compares false)
              const uint4 v0 = *reinterpret_cast<const uint4*>(row + j0);
              const uint4 v1 = *reinterpret_cast<const uint4*>(row + j0 + 8);
              live = any_above_lowest(v0) || any_above_lowest(v1);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (j0 + 8 * h >= np) break;
                const uint4 v = *reinterpret_cast<const uint4*>(row + j0 + 8 * h);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const uint16_t bits = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
                  live = live || (j0 + 8 * h + e < np && bf16_bits_to_float(bits) > lowest);
                }
              }
            }
          }
        }
        const unsigned m = __ballot_sync(0xffffffffu, live);
        if (live) list[n_live + __popc(m & ((1u << lane) - 1u))] = static_cast<uint16_t>(t);
        n_live += __popc(m);
      }
    }
    __syncwarp();
    ptx::fence_proxy_async_smem();  // the scan's reads precede the stages' TMA fills
  }
  // this CTA's share of the live tiles: share m*C + rank of M*C, [lo, lo + n)
  const int sh = m * C + rank, n_sh = M * C;
  const int lo = static_cast<int>(static_cast<int64_t>(sh) * n_live / n_sh);
  const int n = static_cast<int>(static_cast<int64_t>(sh + 1) * n_live / n_sh) - lo;
  auto tile_of = [&](int k) -> int {
    const int x = lo + k;
    if (MODE == kBias) return list[x];
    if (MODE == kNone) return x;
    return runs.tile(x);
  };

  // ---- producer: lane 0 arms a stage, lanes 0-2 issue its requests ----
  const uint32_t stage_tx = S::kStageBytes + (kTerm ? 32u * p.S_q : 0u);
  int pk = 0;
  auto fill = [&](int consumed) {
    while (pk < n && pk < consumed + SPW) {
      const int st = pk % SPW;
      const int key0 = tile_of(pk) * kTile;
      uint8_t* dst = smem + st * S::kStageBytes;
      if (lane == 0) ptx::mbar_arrive_expect_tx(&bars[st], stage_tx);
      __syncwarp();
      if (lane == 0) ptx::tma_load_4d(dst, &kmap, &bars[st], 0, key0, 0, bh);
      else if (lane == 1) ptx::tma_load_4d(dst + S::kKTileBytes, &vmap, &bars[st], 0, key0, 0, bh);
      else if (kTerm && lane == 2) ptx::tma_load_2d(smem + L::kTerm + st * 256, &tmap, &bars[st], key0, b * p.S_q);
      ++pk;
    }
  };
  if (!failed) fill(0);

  // The fused scatter: the KV head's new rows, split over the CTAs of its
  // first row group's cluster.  Loads of the KV head's other CTAs may see a
  // row before or after it is written; a tile that holds new rows is patched
  // from k_new / v_new below.
  int w_new = -1;  // first new slot of the batch, -1: none or out of range (skipped)
  if (kOneSize && p.k_new) {
    const int64_t w = EXTKV_IN(b, 1, p.B, p.status) ? p.write_idx[b] : -1;
    if (w < 0 || w + p.S_new > max_seq) {
      if (kvh == 0 && rg == 0 && m == 0 && rank == 0 && lane == 0) report(p.status, EXTKV_DEV_BAD_WRITE_IDX);
    } else {
      w_new = static_cast<int>(w);
      constexpr int vpr = DK / 8;  // 16-byte vectors per row
      for (int sn = rank; rg == 0 && m == 0 && sn < p.S_new; sn += C)
        for (int v = lane; v < vpr; v += 32) {
          const int64_t dst = (static_cast<int64_t>(bh) * max_seq + w + sn) * DK + v * 8;
          const int64_t src = (static_cast<int64_t>(bh) * p.S_new + sn) * DK + v * 8;
          const int64_t n_bh = static_cast<int64_t>(p.B) * p.Hkv;
          if (!EXTKV_IN(dst, 8, n_bh * max_seq * DK, p.status) || !EXTKV_IN(src, 8, n_bh * p.S_new * DK, p.status))
            continue;
          *reinterpret_cast<uint4*>(p.kc_w + dst) = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
          *reinterpret_cast<uint4*>(p.vc_w + dst) = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
        }
    }
  }

  // ---- consumer ----
  constexpr int kAcc = kKSteps >= 16 ? 4 : 2;  // independent QK^T accumulator chains
  float o[DV / 16][4];
#pragma unroll
  for (int mt = 0; mt < DV / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  Win32 w0{}, w1{};
  if (MODE == kFused || MODE == kFusedExtra) {
    const int64_t qs = query_start(p.spec.q_start, b, np, p.S_q);
    w0 = win32(p.spec, b, qs + i0, np, max_seq);
    w1 = win32(p.spec, b, qs + i1, np, max_seq);
  }
  const uint32_t q_s = ptx::smem_u32(smem + L::kQ);
  auto q_frag = [&](int kp, uint32_t* f4) {  // k-steps 2kp and 2kp+1
    const int cb = kp >> 1, jb = (kp & 1) * 4 + (lane >> 3), r = lane & 7;
    ptx::ldmatrix_x4(f4[0], f4[1], f4[2], f4[3], q_s + cb * 1024 + r * 128 + ((jb ^ r) << 4));
  };
  bool q_ready = kQReg;
  int done = 0;  // items consumed
  for (int k = 0; k < n && !failed; ++k) {
    if (!q_ready) {
      if (__any_sync(0xffffffffu, !ptx::mbar_wait_spin_bounded(qbar, 0, p.polls))) {
        failed = true;
        break;
      }
      q_ready = true;
    }
    const int st = k % SPW;
    if (__any_sync(0xffffffffu, !ptx::mbar_wait_spin_bounded(&bars[st], (k / SPW) & 1, p.polls))) {
      failed = true;
      break;
    }
    uint8_t* kst = smem + st * S::kStageBytes;
    const uint32_t k_s = ptx::smem_u32(kst), v_s = k_s + S::kKTileBytes;
    const uint16_t* term = reinterpret_cast<const uint16_t*>(smem + L::kTerm + st * 256);
    const int key0 = tile_of(k) * kTile;
    if (kOneSize && w_new >= 0 && key0 < w_new + p.S_new && key0 + kTile > w_new) {
      // new rows of this tile straight from k_new / v_new (what the cache
      // holds after the scatter), into the 128-byte-swizzled stage layout
      const int lo_k = max(key0, w_new), hi_k = min(key0 + kTile, w_new + p.S_new);
      constexpr int D = DK;
      constexpr int vpr = D / 8;
      const int64_t nb = static_cast<int64_t>(bh) * p.S_new;
      for (int idx = lane; idx < (hi_k - lo_k) * vpr; idx += 32) {
        const int key = lo_k + idx / vpr;
        const int r = key - key0, ch = idx % vpr;
        const int off = (ch >> 3) * (kTile * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        const int64_t src = (nb + (key - w_new)) * D + ch * 8;
        if (!EXTKV_IN(src, 8, static_cast<int64_t>(p.B) * p.Hkv * p.S_new * D, p.status)) continue;
        *reinterpret_cast<uint4*>(kst + off) = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
        *reinterpret_cast<uint4*>(kst + S::kKTileBytes + off) = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
      }
      ptx::fence_proxy_async_smem();  // these generic writes precede the stage's next TMA fill
      __syncwarp();
    }

    // S^T (16 keys x 8 rows) = K (16 x DK) Q^T (DK x 8), kAcc interleaved chains
    float sa[kAcc][4];
#pragma unroll
    for (int a = 0; a < kAcc; ++a) sa[a][0] = sa[a][1] = sa[a][2] = sa[a][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < kKSteps / 2; ++kp) {
      uint32_t f[4];
      if constexpr (kQReg) {
        f[0] = qf[2 * kp][0];
        f[1] = qf[2 * kp][1];
        f[2] = qf[2 * kp + 1][0];
        f[3] = qf[2 * kp + 1][1];
      } else {
        q_frag(kp, f);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ks = 2 * kp + h;
        const int cb = ks >> 2, j0 = (ks & 3) * 2;
        const int key = (lane & 7) + ((lane >> 3) & 1) * 8, j = j0 + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ptx::ldmatrix_x4(a0, a1, a2, a3, k_s + cb * (kTile * 128) + key * 128 + ((j ^ (key & 7)) << 4));
        ptx::mma_bf16_16816(sa[ks % kAcc], a0, a1, a2, a3, f[2 * h], f[2 * h + 1]);
      }
    }
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[e] = sa[0][e];
#pragma unroll
      for (int a = 1; a < kAcc; ++a) s[e] += sa[a][e];
    }

    // mask + bias in natural units: s = scale*qk + bias; the base-2 scaling
    // comes only after the row maximum is subtracted.
    // s[0]: key ja, row r0; s[1]: ja, r1; s[2]: jb, r0; s[3]: jb, r1.
    const int kla = lane >> 2, klb = kla + 8;
    const int ja = key0 + kla, jb = key0 + klb;
    bool live[4];
    float bv[4] = {0.f, 0.f, 0.f, 0.f};
    if (MODE == kNone) {
      live[0] = ok0 && ja < np;
      live[1] = ok1 && ja < np;
      live[2] = ok0 && jb < np;
      live[3] = ok1 && jb < np;
    } else if (MODE == kBias) {
      bv[0] = bf16_bits_to_float(term[i0 * kTile + kla]);
      bv[1] = bf16_bits_to_float(term[i1 * kTile + kla]);
      bv[2] = bf16_bits_to_float(term[i0 * kTile + klb]);
      bv[3] = bf16_bits_to_float(term[i1 * kTile + klb]);
      live[0] = ok0 && ja < np && bv[0] > lowest;
      live[1] = ok1 && ja < np && bv[1] > lowest;
      live[2] = ok0 && jb < np && bv[2] > lowest;
      live[3] = ok1 && jb < np && bv[3] > lowest;
    } else {
      live[0] = ok0 && w0.allowed(ja);
      live[1] = ok1 && w1.allowed(ja);
      live[2] = ok0 && w0.allowed(jb);
      live[3] = ok1 && w1.allowed(jb);
      if (MODE == kFusedExtra) {
        bv[0] = bf16_bits_to_float(term[i0 * kTile + kla]);
        bv[1] = bf16_bits_to_float(term[i1 * kTile + kla]);
        bv[2] = bf16_bits_to_float(term[i0 * kTile + klb]);
        bv[3] = bf16_bits_to_float(term[i1 * kTile + klb]);
#pragma unroll
        for (int e = 0; e < 4; ++e) live[e] = live[e] && bv[e] > lowest;
      }
    }
    if constexpr (CAP) {
      // softcap on the scaled score, before the bias ("ONNX Domain Attention
      // (Opset 23/24) CUDA Patterns", section 4 op order)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = p.softcap * tanhf(s[e] * p.scale / p.softcap);
        s[e] = live[e] ? x + bv[e] : -INFINITY;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[e] = live[e] ? fmaf(s[e], p.scale, bv[e]) : -INFINITY;
    }

    // Keys no row attends: zero their V rows (poison must not reach PV).
    const unsigned da = __ballot_sync(0xffffffffu, !live[0] && !live[1]);
    const unsigned db = __ballot_sync(0xffffffffu, !live[2] && !live[3]);
    const unsigned fa = da & (da >> 1) & (da >> 2) & (da >> 3) & 0x11111111u;
    const unsigned fb = db & (db >> 1) & (db >> 2) & (db >> 3) & 0x11111111u;
    if (fa | fb) {
      uint8_t* vt = kst + S::kKTileBytes;  // a key's row: kVBoxes lines of 128 B
      for (int w = lane; w < kTile * S::kVBoxes * 8; w += 32) {
        const int key = w / (S::kVBoxes * 8), rem = w % (S::kVBoxes * 8);
        const unsigned f = key < 8 ? fa : fb;
        if ((f >> (4 * (key & 7))) & 1) {
          const int cb = rem >> 3, ch = rem & 7;
          *reinterpret_cast<uint4*>(vt + cb * (kTile * 128) + key * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      ptx::fence_proxy_async_smem();  // these generic writes precede the stage's next TMA fill
      __syncwarp();
    }

    // online softmax for rows r0, r1: weights 2^((s - m) log2 e)
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 4));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 4));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 8));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 8));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 16));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 16));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float ref0 = n0 == -INFINITY ? 0.f : n0, ref1 = n1 == -INFINITY ? 0.f : n1;  // never -inf - -inf
    const float c0 = ptx::ex2((m0 - ref0) * kLog2e), c1 = ptx::ex2((m1 - ref1) * kLog2e);
    const float p0 = ptx::ex2((s[0] - ref0) * kLog2e), p1 = ptx::ex2((s[1] - ref1) * kLog2e);
    const float p2 = ptx::ex2((s[2] - ref0) * kLog2e), p3 = ptx::ex2((s[3] - ref1) * kLog2e);
    l0 = fmaf(l0, c0, p0 + p2);
    l1 = fmaf(l1, c1, p1 + p3);
    m0 = n0;
    m1 = n1;
    if (!__all_sync(0xffffffffu, c0 == 1.f && c1 == 1.f)) {
#pragma unroll
      for (int mt = 0; mt < DV / 16; ++mt) {
        o[mt][0] *= c0;
        o[mt][1] *= c1;
        o[mt][2] *= c0;
        o[mt][3] *= c1;
      }
    }
    // P^T as the B operand: transpose the two 8x8 blocks (keys 0-7, 8-15)
    const uint32_t pb0 = ptx::movmatrix_trans(ptx::pack_bf16x2(p0, p1));
    const uint32_t pb1 = ptx::movmatrix_trans(ptx::pack_bf16x2(p2, p3));

    // O^T (DV x 8) += V^T (DV x 16) P^T (16 x 8)
#pragma unroll
    for (int mt = 0; mt < DV / 16; ++mt) {
      const int cb = mt >> 2, j0 = (mt & 3) * 2;
      const int key = (lane & 7) + (lane >> 4) * 8, j = j0 + ((lane >> 3) & 1);
      uint32_t a0, a1, a2, a3;
      ptx::ldmatrix_x4_trans(a0, a1, a2, a3, v_s + cb * (kTile * 128) + key * 128 + ((j ^ (key & 7)) << 4));
      ptx::mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    done = k + 1;
    fill(done);  // refill the stage just consumed
  }
  if (failed) {
    if (lane == 0) report(p.status, EXTKV_DEV_TIMEOUT);
    // wait (bounded, at the full limit) for every copy still in flight before
    // the CTA's shared memory is reused or released: the requests of items
    // done .. pk - 1, the Q box and the bias rows
    for (int j = done; j < pk; ++j) ptx::mbar_wait_bounded(&bars[j % SPW], (j / SPW) & 1, kWaitPolls);
    if (!kQReg) ptx::mbar_wait_bounded(qbar, 0, kWaitPolls);
    if (MODE == kBias) ptx::mbar_wait_bounded(sbar, 0, kWaitPolls);
  } else if (!kQReg && !q_ready) {
    ptx::mbar_wait_bounded(qbar, 0, kWaitPolls);  // a share without tiles: the Q box still landed
  }

  // ---- this CTA's share: (max, sum, unnormalised O) into its shared memory ----
  // O goes over the ring, whose copies have all landed (a failed share, whose
  // copies may not have, writes no O: its max of -inf keeps it out of the combine)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
  if (!failed) {
#pragma unroll
    for (int mt = 0; mt < DV / 16; ++mt) {
      const int d = mt * 16 + (lane >> 2);
      if (ok0) {
        po[r0 * DV + d] = o[mt][0];
        po[r0 * DV + d + 8] = o[mt][2];
      }
      if (ok1) {
        po[r1 * DV + d] = o[mt][1];
        po[r1 * DV + d + 8] = o[mt][3];
      }
    }
  }
  if (lane < 4) {
    pm[r0] = failed ? -INFINITY : m0;
    pm[r1] = failed ? -INFINITY : m1;
    pl[r0] = failed ? 0.f : l0;
    pl[r1] = failed ? 0.f : l1;
  }
  __syncwarp();

  // ---- combine: column block `rank` of every row, over the C shares in rank order ----
  ptx::cluster_sync();
  const int cpc = DV / C;  // columns of Y this CTA writes
  const int g4 = cpc / 4;
  // with several clusters per unit: this cluster's partial, in the stream-K layout
  float* part = M > 1 ? p.part + static_cast<int64_t>(unit * M + m) * 2 * p.PS : nullptr;
  if (M > 1 && m == 0 && rank == 0 && lane == 0 &&
      EXTKV_IN(unit, 1, static_cast<int64_t>(p.B) * p.Hkv * p.n_rg, p.status))
    p.info[unit] = make_int4(unit * M, M, 0, 0);
  for (int it = lane; it < R * g4; it += 32) {
    const int row = it / g4, col = rank * cpc + (it - row * g4) * 4;
    // every share's (max, sum, O columns) in one round of remote loads
    float mj[kMaxCluster], lj[kMaxCluster];
    float4 ov[kMaxCluster];
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
      if (j < C) {
        mj[j] = ptx::ld_cluster_f32(ptx::map_cluster(pm + row, j));
        lj[j] = ptx::ld_cluster_f32(ptx::map_cluster(pl + row, j));
        ov[j] = ptx::ld_cluster_f32x4(ptx::map_cluster(po + row * DV + col, j));
      }
    }
    float M_ = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j)
      if (j < C) M_ = fmaxf(M_, mj[j]);
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
      // a share without an unmasked key (max -inf) adds nothing; its O may not
      // have been written, so it is left out by selection, not by a zero weight
      if (j >= C || mj[j] == -INFINITY) continue;
      const float wj = ptx::ex2((mj[j] - M_) * kLog2e);
      Lsum = fmaf(wj, lj[j], Lsum);
      acc.x = fmaf(ov[j].x, wj, acc.x);
      acc.y = fmaf(ov[j].y, wj, acc.y);
      acc.z = fmaf(ov[j].z, wj, acc.z);
      acc.w = fmaf(ov[j].w, wj, acc.w);
    }
    if (part) {
      // unnormalised, relative to this cluster's max (the merge kernel's input)
      if (!EXTKV_IN(static_cast<int64_t>(unit * M + m) * 2 * p.PS + 2 * kRows + row * DV + col, 4,
                    static_cast<int64_t>(p.G) * 2 * p.PS, p.status))
        continue;
      *reinterpret_cast<float4*>(part + 2 * kRows + row * DV + col) = acc;
      if (rank == 0 && col == 0) {
        part[row] = M_;
        part[kRows + row] = Lsum;
      }
      continue;
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;  // no unmasked key: zero row
    const uint32_t lo2 = ptx::pack_bf16x2(acc.x * inv, acc.y * inv);
    const uint32_t hi2 = ptx::pack_bf16x2(acc.z * inv, acc.w * inv);
    if (EXTKV_IN((row0 + row) * DV + col, 4, static_cast<int64_t>(p.B) * p.Hq * p.S_q * DV, p.status))
      *reinterpret_cast<uint2*>(p.y + (row0 + row) * DV + col) = make_uint2(lo2, hi2);
  }
  __syncwarp();
  ptx::cluster_sync();  // peers may still read this CTA's share until here
}

// ---- host ---------------------------------------------------------------------------

// Co-resident clusters of C CTAs of `kern` at `smem` bytes (per device, kernel
// and C), derated by 1/16: the occupancy query counted 72 clusters of 8 at four
// CTAs per SM, but the hardware placed 68 (136 of the 152 SMs took clusters),
// and the other 4 clusters waited for a whole second wave.
inline int cluster_capacity(const void* kern, size_t smem, int C) {
  static std::mutex mu;
  struct Entry {
    const void* kern;
    int dev, C, n;
  };
  static Entry entries[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> g(mu);
  for (int i = 0; i < used; ++i)
    if (entries[i].kern == kern && entries[i].dev == dev && entries[i].C == C) return entries[i].n;
  int n = 0;
  if (set_max_dynamic_smem(kern, smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    n -= (n + 15) / 16;
  }
  (void)cudaGetLastError();
  if (used < 64) entries[used++] = Entry{kern, dev, C, n};
  return n;
}

// CTAs per unit for `units` units: the largest C <= 8 (a power of two, at most
// DV / 8 so that each CTA combines whole float4 columns) whose clusters all fit
// the GPU at once; 0: not even single CTAs do.
template <int DK, int DV>
int cluster_size_for(int64_t units) {
  constexpr int SPW = ClusterCfg<DK>::SPW;
  const void* kern = reinterpret_cast<const void*>(attn_decode_cluster_kernel<DK, DV, SPW, kBias, false>);
  const size_t smem = CSmem<DK, DV, SPW>::bytes();
  for (int C = kMaxCluster; C >= 1; C >>= 1) {
    if (DV / C < 4 || DV % (4 * C)) continue;
    if (units <= cluster_capacity(kern, smem, C)) return C;
  }
  return 0;
}

template <int DK, int DV, int MODE, bool CAP>
cudaError_t launch_dcl(const AttnArgs& a, const DecodeParams& prm, const CUtensorMap& kmap,
                       const CUtensorMap& vmap, const CUtensorMap& qmap, const CUtensorMap& tmap, int C, int M) {
  constexpr int SPW = ClusterCfg<DK>::SPW;
  const size_t smem = CSmem<DK, DV, SPW>::bytes();
  auto kern = attn_decode_cluster_kernel<DK, DV, SPW, MODE, CAP>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(C);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.Hkv * prm.n_rg * M * C));
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = smem;
  e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, qmap, tmap, prm, C, M);
  if (e != cudaSuccess || M == 1) {
    if (e == cudaSuccess) note_launches(1);
    return e;
  }
  // the M partials of every unit: the stream-K merge kernel
  const int n_cg = merge_groups(prm.R, DV);
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // a dependent launch, no cluster
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.Hkv * prm.n_rg * n_cg));
  cfg.blockDim = dim3(static_cast<unsigned>((prm.R * (DV / 4 / n_cg) + 31) / 32 * 32));
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<MODE>, prm, n_cg);
  if (e == cudaSuccess) note_launches(2);
  return e;
}

template <int DK, int DV, int MODE>
cudaError_t launch_dclc(const AttnArgs& a, const DecodeParams& prm, const CUtensorMap& kmap,
                        const CUtensorMap& vmap, const CUtensorMap& qmap, const CUtensorMap& tmap, int C, int M) {
  return a.softcap > 0.f ? launch_dcl<DK, DV, MODE, true>(a, prm, kmap, vmap, qmap, tmap, C, M)
                         : launch_dcl<DK, DV, MODE, false>(a, prm, kmap, vmap, qmap, tmap, C, M);
}

// Clusters per unit for C CTAs each: as many as fit the GPU at once beside the
// other units' (at most kMaxSplit), and whose partials fit the workspace
// (the stream-K layout: two partial slots per CTA of its grid).
constexpr int kMaxSplit = 16;

template <int D>
int cluster_split_for(int64_t B, int64_t units, int64_t max_tiles, int C) {
  constexpr int SPW = ClusterCfg<D>::SPW;
  const void* kern = reinterpret_cast<const void*>(attn_decode_cluster_kernel<D, D, SPW, kBias, false>);
  const int cap = cluster_capacity(kern, CSmem<D, D, SPW>::bytes(), C);
  const DecodeShape shape = decode_shape<D, D>(B, units * max_tiles);
  int64_t M = std::min<int64_t>(kMaxSplit, cap / std::max<int64_t>(units, 1));
  M = std::min<int64_t>(M, shape.G / std::max<int64_t>(units, 1));
  return static_cast<int>(std::max<int64_t>(M, 1));
}

// One head size D for queries, keys and values.  C: from cluster_size_for; M:
// clusters per unit (from cluster_split_for; M > 1 needs the workspace).
template <int D>
cudaError_t launch_dc(const AttnArgs& a, int C, int M, const char** name) {
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  CUtensorMap kmap, vmap, qmap, tmap;
  // K/V and Q through the same views as the stream-K kernel: one TMA box
  // brings a whole tile as D/64 blocks of (rows x 128 B), 128-byte swizzle
  const uint64_t units = static_cast<uint64_t>(a.B * a.Hkv);
  const uint64_t kv_dims[4] = {64, static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(D / 64), units};
  const uint64_t kv_strides[3] = {static_cast<uint64_t>(D) * 2, 128, static_cast<uint64_t>(a.max_seq) * D * 2};
  const uint32_t kv_box[4] = {64, kTile, static_cast<uint32_t>(D / 64), 1};
  const uint64_t q_dims[3] = {64, static_cast<uint64_t>(a.B * a.Hq * a.S_q), static_cast<uint64_t>(D / 64)};
  const uint64_t q_strides[2] = {static_cast<uint64_t>(D) * 2, 128};
  const uint32_t q_box[3] = {64, kRows, static_cast<uint32_t>(D / 64)};
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 4, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 4, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&qmap, a.q, 3, q_dims, q_strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const void* term = a.bias ? a.bias : (a.fused ? a.extra : nullptr);
  std::memset(&tmap, 0, sizeof tmap);
  if (term) {
    const uint64_t t_dims[2] = {static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(a.B * a.S_q)};
    const uint64_t t_strides[1] = {static_cast<uint64_t>(a.max_seq) * 2};
    const uint32_t t_box[2] = {kTile, static_cast<uint32_t>(a.S_q)};
    if (!make_tensor_map_bf16(&tmap, term, 2, t_dims, t_strides, t_box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  DecodeParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.y = static_cast<__nv_bfloat16*>(a.y);
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.bias = static_cast<const __nv_bfloat16*>(a.bias);
  prm.spec = BiasSpec{a.causal, a.window, a.span_offsets, a.spans, a.extra, a.q_start};
  prm.nonpad = a.nonpad;
  prm.scale = a.scale;
  prm.softcap = a.softcap;
  prm.B = static_cast<int>(a.B);
  prm.Hq = static_cast<int>(a.Hq);
  prm.Hkv = static_cast<int>(a.Hkv);
  prm.S_q = static_cast<int>(a.S_q);
  prm.g = static_cast<int>(a.Hq / a.Hkv);
  prm.GR = static_cast<int>(a.Hq / a.Hkv * a.S_q);
  prm.n_rg = static_cast<int>(row_groups(prm.GR));
  prm.R = std::min(prm.GR, kRows);
  prm.D = D;
  prm.max_seq = static_cast<int>(a.max_seq);
  prm.max_tiles = static_cast<int>(max_tiles);
  prm.status = a.status;
  prm.polls = wait_limit(a.wait_limit_plus1, kWaitPolls);
  prm.kc_w = static_cast<__nv_bfloat16*>(a.kc_w);
  prm.vc_w = static_cast<__nv_bfloat16*>(a.vc_w);
  prm.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  prm.write_idx = a.write_idx;
  prm.S_new = static_cast<int>(a.S_new);
  if (M > 1) {
    // the clusters' partials and the units' slice records, where the stream-K
    // kernels keep theirs
    const int64_t units = a.B * a.Hkv * prm.n_rg;
    const DecodeShape shape = decode_shape<D, D>(a.B, units * max_tiles);
    if (units * M > shape.G) return cudaErrorInvalidValue;
    const WsLayout ws = ws_layout(a.B, a.Hkv * prm.n_rg, max_tiles, shape.G, prm.R, D);
    if (!a.workspace || a.ws_bytes < ws.total) return cudaErrorInvalidValue;
    uint8_t* wsb = static_cast<uint8_t*>(a.workspace);
    prm.info = reinterpret_cast<int4*>(wsb + ws.info);
    prm.part = reinterpret_cast<float*>(wsb + ws.part);
    prm.PS = static_cast<int>(part_floats(prm.R, D));
    prm.G = shape.G;  // the partial slots' extent (two per CTA of the stream-K grid)
  }
  cudaError_t e;
  switch (mode_of(a)) {
    case kNone: e = launch_dclc<D, D, kNone>(a, prm, kmap, vmap, qmap, tmap, C, M); break;
    case kBias: e = launch_dclc<D, D, kBias>(a, prm, kmap, vmap, qmap, tmap, C, M); break;
    case kFused: e = launch_dclc<D, D, kFused>(a, prm, kmap, vmap, qmap, tmap, C, M); break;
    default: e = launch_dclc<D, D, kFusedExtra>(a, prm, kmap, vmap, qmap, tmap, C, M); break;
  }
  if (e != cudaSuccess) return e;
  *name = prm.k_new ? "attn_decode_cluster_scatter" : "attn_decode_cluster";
  return cudaGetLastError();
}

}  // namespace
}  // namespace extkv
