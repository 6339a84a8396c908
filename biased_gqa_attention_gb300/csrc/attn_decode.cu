// attn_decode.cu -- split-KV decode attention over the external static cache.
//
// Work unit: one (batch b, KV head) pair and its R = (Hq/Hkv) * S_q query
// rows (R <= 8), which share every K/V row they read ("ONNX Domain Attention
// (Opset 23/24) CUDA Patterns", section 1: GQA by reshaping Q, no KV
// replication).  A unit is split over the NS CTAs of one thread-block cluster.
//
//   1. Every CTA lists the unit's live 16-key tiles: tiles holding at least
//      one key that some row may attend (the materialised bias row is scanned,
//      or the fused specification's intervals are intersected).  Tiles at or
//      beyond nonpad_kv_seqlen[b], or fully masked, are never loaded.
//   2. CTA c takes an equal share of the live tiles; inside it, warp w takes
//      every NW-th tile and streams it through its own ring of SPW shared
//      memory stages, filled by TMA (128-byte swizzle, one box per 64
//      columns).  HBM bytes are read once.
//   3. Per tile, on the warp's tensor cores (mma.sync m16n8k16 bf16, fp32
//      accumulation): S^T = K Q^T with the 16 keys on M and the <= 8 query
//      rows on N; scale, bias, mask; online softmax in fp32; P^T is moved
//      into the B-operand layout with movmatrix; O^T += V^T P^T.
//   4. Warps of a CTA, then CTAs of the cluster (through distributed shared
//      memory), merge their (max, sum, output) partials; each CTA writes a
//      slice of D of the unit's output rows.
//
// Masking and zero rows follow section 6 of the same page: a key is masked
// iff j >= nonpad[b] or bias <= lowest(T); masked scores become -inf by
// selection; V rows of keys no row may attend are zeroed in shared memory
// before the PV product, so poisoned (even NaN) cache slots cannot reach the
// output; a row with no unmasked key is written as zeros.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace extkv {

namespace {

constexpr int kTile = 16;                 // keys per tile (M of the QK^T mma)
constexpr int kRows = 8;                  // query rows per unit (N of the mma)
constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits

template <int D>
struct DecodeCfg;
template <>
struct DecodeCfg<64> {
  static constexpr int NW = 4, SPW = 4;
};
template <>
struct DecodeCfg<128> {
  static constexpr int NW = 4, SPW = 3;
};
template <>
struct DecodeCfg<256> {
  static constexpr int NW = 2, SPW = 3;
};
template <>
struct DecodeCfg<512> {
  static constexpr int NW = 1, SPW = 3;
};

struct DecodeParams {
  __nv_bfloat16* y;
  const __nv_bfloat16* bias;
  BiasSpec spec;
  int fused;
  const int64_t* nonpad;
  float scale;
  int Hq, Hkv, S_q, g, R;
  int64_t max_seq;
  int32_t* status;
};

// Shared memory map (offsets from a 1024-byte aligned base).
template <int D, int NW, int SPW>
struct Smem {
  static constexpr int kBoxes = D / 64;                       // 64-column TMA boxes
  static constexpr int kTileBytes = kBoxes * kTile * 128;     // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;          // K then V
  static constexpr int kStages = NW * SPW;
  static constexpr int kQ = kStages * kStageBytes;            // Q tile: kBoxes x 8 rows x 128 B
  static constexpr int kBars = kQ + kBoxes * 1024;            // kStages + 1 mbarriers
  static constexpr int kMisc = kBars + (kStages + 1) * 8;     // list length + scan scratch
  static constexpr int kList = kMisc + 64;                    // live tile list (uint16)
  // Combine scratch reuses the stages: per warp O (kRows x (D+4) fp32), m, l;
  // then one CTA partial of the same shape.
  static constexpr int kRowStride = D + 4;
  static constexpr int kPart = kRows * kRowStride * 4 + 2 * kRows * 4;
  static_assert((NW + 1) * kPart <= kQ, "combine scratch must fit in the stages");
  static size_t bytes(int64_t max_tiles) { return 1024 + kList + 2 * max_tiles + 16; }
};

__device__ __forceinline__ float exp2_scaled(float x) { return exp2f(x * kLog2e); }

template <int D, int NW, int SPW>
__global__ void __launch_bounds__(NW * 32) attn_decode_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap qmap, const DecodeParams p) {
  using S = Smem<D, NW, SPW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars);  // [stages], q
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + S::kList);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NS = static_cast<int>(gridDim.x);
  const int crank = static_cast<int>(ptx::cluster_ctarank());
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int64_t max_seq = p.max_seq;
  const int64_t row0 = (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(kvh) * p.g) * p.S_q;
  const int32_t bh = b * p.Hkv + kvh;

  if (tid == 0) {
    for (int s = 0; s < S::kStages + 1; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&kmap);
    ptx::prefetch_tensormap(&vmap);
  }
  __syncthreads();
  if (tid == 0) {
    // Q rows of the unit (rows past R belong to other units or are zero
    // filled; they only feed output columns that are never written).
    ptx::mbar_arrive_expect_tx(&bars[S::kStages], S::kBoxes * 1024);
    for (int c = 0; c < S::kBoxes; ++c)
      ptx::tma_load_2d(smem + S::kQ + c * 1024, &qmap, &bars[S::kStages], c * 64,
                       static_cast<int32_t>(row0));
  }

  const int64_t np = p.nonpad[b];
  const bool bad = bad_nonpad(np, max_seq);
  if (bad && crank == 0 && tid == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);

  // ---- 1. live tiles ----------------------------------------------------------
  // Each lane's two query rows (columns of S^T): r0 = 2*(lane%4), r1 = r0+1.
  const int r_lane[2] = {2 * (lane & 3), 2 * (lane & 3) + 1};
  RowWindow win[2];
  int64_t jlo = 0, jhi = bad ? 0 : np;
  if (p.fused && !bad) {
    int64_t lo = INT64_MAX, hi = INT64_MIN;
    const int64_t qs = query_start(p.spec.q_start, b, np, p.S_q);
    for (int i = 0; i < p.S_q; ++i) {
      RowWindow w = row_window(p.spec, b, qs + i, np);
      lo = min(lo, w.lo());
      hi = max(hi, w.hi());
    }
    jlo = lo;
    jhi = hi;
    for (int e = 0; e < 2; ++e) {
      const int i = r_lane[e] % p.S_q;
      win[e] = row_window(p.spec, b, qs + i, np);
    }
  }
  const int64_t t_begin = jlo >= jhi ? 0 : jlo / kTile;
  const int64_t t_end = jlo >= jhi ? 0 : (jhi + kTile - 1) / kTile;
  const int n_range = static_cast<int>(t_end - t_begin);
  const float lowest = Elem<__nv_bfloat16>::lowest();

  // Each thread owns a contiguous segment of the tile range.
  const int T = NW * 32;
  const int seg = (n_range + T - 1) / T;
  const int my_lo = min(n_range, tid * seg), my_hi = min(n_range, my_lo + seg);
  auto tile_live = [&](int64_t t) -> bool {
    const int64_t k0 = t * kTile;
    if (!p.fused && !p.bias) return true;  // only nonpad masks: every tile below it
    if (p.fused) {
      for (int i = 0; i < p.S_q; ++i) {
        const int64_t qs = query_start(p.spec.q_start, b, np, p.S_q);
        RowWindow w = row_window(p.spec, b, qs + i, np);
        const int64_t a0 = max(k0, max(w.band_lo, int64_t(0))), a1 = min(k0 + kTile, min(w.band_hi, np));
        const int64_t s0 = max(k0, max(w.span_lo, int64_t(0))), s1 = min(k0 + kTile, min(w.span_hi, np));
        if (a0 < a1 || s0 < s1) return true;
      }
      return false;
    }
    for (int i = 0; i < p.S_q; ++i) {
      const __nv_bfloat16* brow = p.bias + (static_cast<int64_t>(b) * p.S_q + i) * max_seq;
      for (int h8 = 0; h8 < 2; ++h8) {
        const int64_t j8 = k0 + 8 * h8;
        if (j8 >= np) break;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(brow + j8));
        const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
        for (int q = 0; q < 8; ++q)
          if (j8 + q < np && bf16_bits_to_float(e[q]) > lowest) return true;
      }
    }
    return false;
  };
  int cnt = 0;
  for (int t = my_lo; t < my_hi; ++t) cnt += tile_live(t_begin + t);
  // Block-wide exclusive scan of the counts.
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  __shared__ int warp_tot[NW];
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
  for (int w2 = 0; w2 < NW; ++w2) {
    if (w2 < warp) base += warp_tot[w2];
    total += warp_tot[w2];
  }
  int pos = base + incl - cnt;
  for (int t = my_lo; t < my_hi; ++t)
    if (tile_live(t_begin + t)) list[pos++] = static_cast<uint16_t>(t_begin + t);
  __syncthreads();

  // ---- 2. this CTA's share, streamed per warp -------------------------------
  const int c_begin = static_cast<int>((static_cast<int64_t>(total) * crank) / NS);
  const int c_end = static_cast<int>((static_cast<int64_t>(total) * (crank + 1)) / NS);
  const int my_first = c_begin + warp;  // warp's tiles: my_first + k*NW
  uint8_t* stage0 = smem + warp * SPW * S::kStageBytes;
  uint64_t* wbars = bars + warp * SPW;

  auto issue = [&](int idx, int st) {
    const int32_t key0 = static_cast<int32_t>(list[idx]) * kTile;
    uint8_t* dst = stage0 + st * S::kStageBytes;
    ptx::mbar_arrive_expect_tx(&wbars[st], S::kStageBytes);
#pragma unroll
    for (int c = 0; c < S::kBoxes; ++c) {
      ptx::tma_load_3d(dst + c * kTile * 128, &kmap, &wbars[st], c * 64, key0, bh);
      ptx::tma_load_3d(dst + S::kTileBytes + c * kTile * 128, &vmap, &wbars[st], c * 64, key0, bh);
    }
  };
  if (lane == 0) {
    for (int k = 0; k < SPW; ++k) {
      const int idx = my_first + k * NW;
      if (idx < c_end) issue(idx, k);
    }
  }

  // Q fragments (B operand of S^T = K Q^T) stay in registers for D <= 256.
  constexpr bool kQReg = D <= 256;
  constexpr int kKSteps = D / 16;
  uint32_t qf[kQReg ? kKSteps : 1][2];
  // Wait results are made warp-uniform so that no lane leaves a loop its
  // warp-mates stay in.
  bool failed = __any_sync(0xffffffffu, !ptx::mbar_wait_bounded(&bars[S::kStages], 0, kWaitPolls));
  const uint32_t q_s = ptx::smem_u32(smem + S::kQ);
  auto q_frag = [&](int kp, uint32_t* f4) {  // k-steps 2kp and 2kp+1
    const int c = kp >> 1, jb = (kp & 1) * 4 + (lane >> 3), r = lane & 7;
    ptx::ldmatrix_x4(f4[0], f4[1], f4[2], f4[3], q_s + c * 1024 + r * 128 + ((jb ^ r) << 4));
  };
  if constexpr (kQReg) {
#pragma unroll
    for (int kp = 0; kp < kKSteps / 2; ++kp) {
      uint32_t f[4];
      q_frag(kp, f);
      qf[2 * kp][0] = f[0];
      qf[2 * kp][1] = f[1];
      qf[2 * kp + 1][0] = f[2];
      qf[2 * kp + 1][1] = f[3];
    }
  }

  float o[D / 16][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const bool row_ok[2] = {r_lane[0] < p.R, r_lane[1] < p.R};

  int k = 0;
  for (int idx = my_first; idx < c_end && !failed; idx += NW, ++k) {
    const int st = k % SPW;
    if (__any_sync(0xffffffffu, !ptx::mbar_wait_bounded(&wbars[st], (k / SPW) & 1, kWaitPolls))) {
      failed = true;
      break;
    }
    uint8_t* kst = stage0 + st * S::kStageBytes;
    const uint32_t k_s = ptx::smem_u32(kst), v_s = k_s + S::kTileBytes;
    const int64_t key0 = static_cast<int64_t>(list[idx]) * kTile;

    // S^T (16 keys x 8 rows) = K (16 x D) Q^T (D x 8)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
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
        const int c = ks >> 2, j0 = (ks & 3) * 2;
        const int key = (lane & 7) + ((lane >> 3) & 1) * 8, j = j0 + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ptx::ldmatrix_x4(a0, a1, a2, a3, k_s + c * (kTile * 128) + key * 128 + ((j ^ (key & 7)) << 4));
        ptx::mma_bf16_16816(s, a0, a1, a2, a3, f[2 * h], f[2 * h + 1]);
      }
    }

    // scale + bias + mask; s[e]: key = lane/4 (+8 for e >= 2), row r_lane[e & 1]
    bool dead[2];  // key (lane/4, +8) masked for both of this lane's rows
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int64_t j = key0 + (lane >> 2) + 8 * kk;
      dead[kk] = true;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float& sv = s[2 * kk + e];
        bool live = row_ok[e] && j < np;
        float bv = 0.f;
        if (live) {
          const int i = r_lane[e] % p.S_q;
          if (p.bias) {
            bv = Elem<__nv_bfloat16>::load(p.bias, (static_cast<int64_t>(b) * p.S_q + i) * max_seq + j);
            live = bv > lowest;
          } else if (p.fused) {
            live = win[e].allowed(j);
            if (live && p.spec.extra) {
              bv = Elem<__nv_bfloat16>::load(static_cast<const __nv_bfloat16*>(p.spec.extra),
                                             (static_cast<int64_t>(b) * p.S_q + i) * max_seq + j);
              live = bv > lowest;
            }
          }
        }
        sv = live ? fmaf(sv, p.scale, bv) : -INFINITY;
        dead[kk] = dead[kk] && !live;
      }
    }
    // Zero the V rows of keys that no row of the unit attends.
    const unsigned dm0 = __ballot_sync(0xffffffffu, dead[0]);
    const unsigned dm1 = __ballot_sync(0xffffffffu, dead[1]);
    unsigned dead_keys = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (((dm0 >> (4 * q)) & 0xF) == 0xF) dead_keys |= 1u << q;
      if (((dm1 >> (4 * q)) & 0xF) == 0xF) dead_keys |= 1u << (q + 8);
    }
    if (dead_keys) {
      // each dead key owns kBoxes lines of 128 B in the V tile
      uint8_t* vt = kst + S::kTileBytes;
      for (int u = lane; u < kTile * S::kBoxes * 8; u += 32) {
        const int key = u / (S::kBoxes * 8), rem = u % (S::kBoxes * 8);
        if ((dead_keys >> key) & 1) {
          const int c = rem >> 3, ch = rem & 7;
          *reinterpret_cast<uint4*>(vt + c * (kTile * 128) + key * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
    }

    // online softmax, rows r_lane[0], r_lane[1]
    float mt[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mt[e] = fmaxf(mt[e], __shfl_xor_sync(0xffffffffu, mt[e], 4));
      mt[e] = fmaxf(mt[e], __shfl_xor_sync(0xffffffffu, mt[e], 8));
      mt[e] = fmaxf(mt[e], __shfl_xor_sync(0xffffffffu, mt[e], 16));
    }
    float pr[4], corr[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float m_new = fmaxf(m_run[e], mt[e]);
      const float ref = m_new == -INFINITY ? 0.f : m_new;  // never -inf - -inf
      corr[e] = exp2_scaled(m_run[e] - ref);
      pr[e] = exp2_scaled(s[e] - ref);
      pr[2 + e] = exp2_scaled(s[2 + e] - ref);
      l_run[e] = fmaf(l_run[e], corr[e], pr[e] + pr[2 + e]);
      m_run[e] = m_new;
    }
    if (!__all_sync(0xffffffffu, corr[0] == 1.f && corr[1] == 1.f)) {
#pragma unroll
      for (int mt2 = 0; mt2 < D / 16; ++mt2) {
        o[mt2][0] *= corr[0];
        o[mt2][1] *= corr[1];
        o[mt2][2] *= corr[0];
        o[mt2][3] *= corr[1];
      }
    }
    // P^T as the B operand: transpose the two 8x8 blocks (keys 0-7, 8-15)
    const uint32_t pb0 = ptx::movmatrix_trans(ptx::pack_bf16x2(pr[0], pr[1]));
    const uint32_t pb1 = ptx::movmatrix_trans(ptx::pack_bf16x2(pr[2], pr[3]));

    // O^T (D x 8) += V^T (D x 16) P^T (16 x 8)
#pragma unroll
    for (int mt2 = 0; mt2 < D / 16; ++mt2) {
      const int c = mt2 >> 2, j0 = (mt2 & 3) * 2;
      const int key = (lane & 7) + (lane >> 4) * 8, j = j0 + ((lane >> 3) & 1);
      uint32_t a0, a1, a2, a3;
      ptx::ldmatrix_x4_trans(a0, a1, a2, a3, v_s + c * (kTile * 128) + key * 128 + ((j ^ (key & 7)) << 4));
      ptx::mma_bf16_16816(o[mt2], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    // refill this stage with the warp's tile SPW steps ahead
    const int nidx = idx + SPW * NW;
    if (lane == 0 && nidx < c_end) {
      ptx::fence_proxy_async_smem();
      issue(nidx, st);
    }
  }
  if (failed) {
    // A wait gave up: report it, then wait (bounded) for this warp's loads
    // still in flight before the stages are reused or the CTA exits.
    if (lane == 0) report(p.status, EXTKV_DEV_TIMEOUT);
    for (int k2 = k; k2 < k + SPW; ++k2)
      if (my_first + k2 * NW < c_end) ptx::mbar_wait_bounded(&wbars[k2 % SPW], (k2 / SPW) & 1, kWaitPolls);
  }

  // ---- 4. merge partials --------------------------------------------------------
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
  }
  // Warp partials, after every warp left the stages (no TMA is in flight:
  // each warp only issued loads it consumed, unless a wait gave up).
  __syncthreads();
  constexpr int RS = S::kRowStride;
  auto part_o = [&](int w2) { return reinterpret_cast<float*>(smem + w2 * S::kPart); };
  auto part_m = [&](int w2) { return part_o(w2) + kRows * RS; };
  auto part_l = [&](int w2) { return part_o(w2) + kRows * RS + kRows; };
  {
    float* po = part_o(warp);
#pragma unroll
    for (int mt2 = 0; mt2 < D / 16; ++mt2) {
      const int d = mt2 * 16 + (lane >> 2);
      po[r_lane[0] * RS + d] = o[mt2][0];
      po[r_lane[1] * RS + d] = o[mt2][1];
      po[r_lane[0] * RS + d + 8] = o[mt2][2];
      po[r_lane[1] * RS + d + 8] = o[mt2][3];
    }
    if (lane < 4) {
      part_m(warp)[r_lane[0]] = m_run[0];
      part_m(warp)[r_lane[1]] = m_run[1];
      part_l(warp)[r_lane[0]] = l_run[0];
      part_l(warp)[r_lane[1]] = l_run[1];
    }
  }
  __syncthreads();
  // CTA partial (unnormalised) in slot NW
  float* co = part_o(NW);
  float* cm = part_m(NW);
  float* cl = part_l(NW);
  if (tid < kRows) {
    float m = -INFINITY;
    for (int w2 = 0; w2 < NW; ++w2) m = fmaxf(m, part_m(w2)[tid]);
    float l = 0.f;
    const float ref = m == -INFINITY ? 0.f : m;
    for (int w2 = 0; w2 < NW; ++w2) l += part_l(w2)[tid] * exp2_scaled(part_m(w2)[tid] - ref);
    cm[tid] = m;
    cl[tid] = l;
  }
  for (int u = tid; u < kRows * D; u += T) {
    const int r = u / D, d = u % D;
    float m = -INFINITY;
    for (int w2 = 0; w2 < NW; ++w2) m = fmaxf(m, part_m(w2)[r]);
    const float ref = m == -INFINITY ? 0.f : m;
    float acc = 0.f;
    for (int w2 = 0; w2 < NW; ++w2) acc += part_o(w2)[r * RS + d] * exp2_scaled(part_m(w2)[r] - ref);
    co[r * RS + d] = acc;
  }
  ptx::cluster_sync();
  // Cluster merge: CTA `crank` writes columns [d0, d1) of the unit's rows.
  const int d0 = (D * crank) / NS, d1 = (D * (crank + 1)) / NS;
  const uint32_t co_s = ptx::smem_u32(co), cm_s = ptx::smem_u32(cm), cl_s = ptx::smem_u32(cl);
  for (int u = tid; u < p.R * (d1 - d0); u += T) {
    const int r = u / (d1 - d0), d = d0 + u % (d1 - d0);
    float M = -INFINITY;
    for (int c = 0; c < NS; ++c) M = fmaxf(M, ptx::ld_cluster_f32(ptx::map_cluster(cm_s + 4 * r, c)));
    const float ref = M == -INFINITY ? 0.f : M;
    float L = 0.f, acc = 0.f;
    for (int c = 0; c < NS; ++c) {
      const float wgt = exp2_scaled(ptx::ld_cluster_f32(ptx::map_cluster(cm_s + 4 * r, c)) - ref);
      L += ptx::ld_cluster_f32(ptx::map_cluster(cl_s + 4 * r, c)) * wgt;
      acc += ptx::ld_cluster_f32(ptx::map_cluster(co_s + 4 * (r * RS + d), c)) * wgt;
    }
    // no unmasked key (or a skipped batch): exact zero by selection
    const float out = (L > 0.f && !bad && !failed) ? acc / L : 0.f;
    p.y[(row0 + r) * D + d] = __float2bfloat16_rn(out);
  }
  ptx::cluster_sync();  // keep this CTA's shared memory alive for the readers
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const char** name) {
  using Cfg = DecodeCfg<D>;
  constexpr int NW = Cfg::NW, SPW = Cfg::SPW;
  using S = Smem<D, NW, SPW>;
  CUtensorMap kmap, vmap, qmap;
  const uint64_t kv_dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.max_seq),
                               static_cast<uint64_t>(a.B * a.Hkv)};
  const uint64_t kv_strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.max_seq) * D * 2};
  const uint32_t kv_box[3] = {64, kTile, 1};
  const uint64_t q_dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.B * a.Hq * a.S_q)};
  const uint64_t q_strides[1] = {static_cast<uint64_t>(D) * 2};
  const uint32_t q_box[2] = {64, kRows};
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 3, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 3, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&qmap, a.q, 2, q_dims, q_strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;

  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  const size_t smem = S::bytes(max_tiles);
  auto kern = attn_decode_kernel<D, NW, SPW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;

  // Split each unit over a cluster so that about two waves of CTAs cover the GPU.
  const int64_t units = a.B * a.Hkv;
  const int64_t target = 2 * static_cast<int64_t>(num_sms());
  int ns = 1;
  while (ns < 8 && units * ns < target && ns * 2 <= max_tiles) ns *= 2;

  DecodeParams prm;
  prm.y = static_cast<__nv_bfloat16*>(a.y);
  prm.bias = static_cast<const __nv_bfloat16*>(a.bias);
  prm.spec = BiasSpec{a.causal, a.window, a.span_offsets, a.spans, a.extra, a.q_start};
  prm.fused = a.fused;
  prm.nonpad = a.nonpad;
  prm.scale = a.scale;
  prm.Hq = static_cast<int>(a.Hq);
  prm.Hkv = static_cast<int>(a.Hkv);
  prm.S_q = static_cast<int>(a.S_q);
  prm.g = static_cast<int>(a.Hq / a.Hkv);
  prm.R = static_cast<int>(a.Hq / a.Hkv * a.S_q);
  prm.max_seq = a.max_seq;
  prm.status = a.status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ns, static_cast<unsigned>(a.Hkv), static_cast<unsigned>(a.B));
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ns;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, qmap, prm);
  if (e != cudaSuccess) return e;
  *name = "attn_decode_splitkv_mma";
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(const AttnArgs& a) {
  if (a.dtype != EXTKV_BF16) return false;
  if (a.D != 64 && a.D != 128 && a.D != 256 && a.D != 512) return false;
  if ((a.Hq / a.Hkv) * a.S_q > kRows) return false;
  if (a.bias && a.max_seq % 8) return false;  // 16-byte bias row loads
  if (a.max_seq > 16 * 65535 || a.B > 65535 || a.Hkv > 65535) return false;
  if (a.B * a.Hkv > 0x7fffffff || a.B * a.Hq * a.S_q > 0x7fffffff) return false;
  return true;
}

cudaError_t launch_attn_decode(const AttnArgs& a, const char** name) {
  switch (a.D) {
    case 64: return launch_d<64>(a, name);
    case 128: return launch_d<128>(a, name);
    case 256: return launch_d<256>(a, name);
    case 512: return launch_d<512>(a, name);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace extkv
