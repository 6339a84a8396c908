// attn_decode.cu -- stream-K split-KV decode attention over the external
// static cache.
//
// Work unit: one (batch b, KV head) pair and its R = (Hq/Hkv) * S_q query
// rows (R <= 8), which share every K/V row they read ("ONNX Domain Attention
// (Opset 23/24) CUDA Patterns", section 1: GQA by reshaping Q, no KV
// replication).  The decode step is HBM-bound ("Skill: Attention
// Optimization": decode is memory-bandwidth bound regardless of kernel), so
// the design goal is to stream every live K/V row exactly once, with every SM
// busy until the end:
//
//   plan kernel (one CTA per batch): lists the batch's live 16-key tiles --
//     tiles holding at least one key that some query row may attend.  With a
//     materialised bias the bias rows are bulk-copied into shared memory and
//     scanned; with the fused specification the rows' allowed intervals are
//     intersected; without either, every tile below nonpad is live.  Tiles at
//     or beyond nonpad_kv_seqlen[b], or fully masked, are never loaded.
//   decode kernel (persistent, one warp per CTA, G CTAs filling the GPU):
//     the live tiles of all units form one sequence of T work items
//     (unit-major); CTA c takes the contiguous slice [c*T/G, (c+1)*T/G) --
//     equal work per CTA whatever the lengths (stream-K).  The warp streams
//     its slice through a ring of SPW shared-memory stages filled by TMA (K
//     and V tiles with a 128-byte swizzle, one box per 64 columns, plus the
//     tile's bias or extra-term block), running ahead across unit boundaries;
//     Q tiles are double-buffered per unit.  Per tile, on the tensor cores
//     (mma.sync m16n8k16 bf16, fp32 accumulation): S^T = K Q^T with the 16
//     keys on M and the <= 8 query rows on N; scale, bias, mask; online
//     softmax in fp32; P^T moved into the B-operand layout with movmatrix;
//     O^T += V^T P^T.  A unit wholly inside one slice is written directly;
//     a unit split across slices leaves fp32 (max, sum, output) partials in
//     the workspace, and the last slice to finish (an atomic ticket, no
//     waiting) merges them.
//
// Masking and zero rows follow section 6 of the ORT page: a key is masked iff
// j >= nonpad[b] or bias <= lowest(T); masked scores become -inf by
// selection; V rows of keys no row of the unit attends are zeroed in shared
// memory before the PV product, so poisoned (even NaN) cache slots cannot
// reach the output; a row with no unmasked key, and every row of a unit with
// no live tile, is written as zeros.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace extkv {

namespace {

constexpr int kTile = 16;                  // keys per tile (M of the QK^T mma)
constexpr int kRows = 8;                   // query rows per unit (N of the mma)
constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits
constexpr int kMaxWork = 1024;             // work items of one slice, in shared memory
constexpr int kMaxB = 1024;                // batches (prefix table in shared memory)
constexpr int kPlanThreads = 256;
constexpr int kPlanScanBytes = 64 * 1024;  // bias rows staged in shared memory by the plan

template <int D>
struct DecodeCfg;  // SPW: shared-memory stages of the single warp
template <>
struct DecodeCfg<64> {
  static constexpr int SPW = 8;
};
template <>
struct DecodeCfg<128> {
  static constexpr int SPW = 5;
};
template <>
struct DecodeCfg<256> {
  static constexpr int SPW = 3;
};
template <>
struct DecodeCfg<512> {
  static constexpr int SPW = 2;
};

// ---- workspace ----------------------------------------------------------------

struct WsLayout {
  size_t count, tiles, counters, part, total;
};

WsLayout ws_layout(int64_t B, int64_t units, int64_t max_tiles, int64_t G, int64_t D) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  WsLayout l;
  size_t o = 0;
  l.count = o;  // int32 live tiles per batch
  o = al(o + static_cast<size_t>(B) * 4);
  l.tiles = o;  // uint16 live tile list per batch
  o = al(o + static_cast<size_t>(B * max_tiles) * 2);
  l.counters = o;  // int32 merge tickets per unit
  o = al(o + static_cast<size_t>(units) * 4);
  l.part = o;  // per CTA, two partials: m[8], l[8], O[8][D] fp32
  o = al(o + static_cast<size_t>(G) * 2 * (2 * kRows + kRows * D) * 4);
  l.total = o;
  return l;
}

struct DecodeParams {
  __nv_bfloat16* y;
  const __nv_bfloat16* bias;  // materialised bias or nullptr
  BiasSpec spec;
  int fused;
  int tile_term;  // 1: TMA brings a per-tile bias / extra-term block
  const int64_t* nonpad;
  float scale;
  int B, Hq, Hkv, S_q, g, R, D;
  int64_t max_seq, max_tiles;
  int G;
  int32_t* count;
  uint16_t* tiles;
  int32_t* counters;
  float* part;
  int32_t* status;
};

__device__ __forceinline__ float exp2_scaled(float x) { return exp2f(x * kLog2e); }

// Allowed-key hull [lo, hi) of a unit's query rows under the fused spec.
__device__ __forceinline__ void fused_hull(const DecodeParams& p, int b, int64_t np, int64_t qs,
                                           int64_t& lo, int64_t& hi) {
  lo = INT64_MAX;
  hi = INT64_MIN;
  for (int i = 0; i < p.S_q; ++i) {
    const RowWindow w = row_window(p.spec, b, qs + i, np);
    lo = min(lo, w.lo());
    hi = max(hi, w.hi());
  }
}

// ---- plan: live tiles of one batch ---------------------------------------------

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int T = kPlanThreads;
  uint8_t* flags = smem;  // [max_tiles]
  uint8_t* rows = smem + ((p.max_tiles + 127) / 128) * 128;
  uint64_t* bar = reinterpret_cast<uint64_t*>(rows + kPlanScanBytes);
  __shared__ int warp_tot[T / 32];
  const float lowest = Elem<__nv_bfloat16>::lowest();

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  const int64_t max_seq = p.max_seq;
  const int64_t np = p.nonpad[b];
  const bool bad = bad_nonpad(np, max_seq);
  if (bad && tid == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);
  const int64_t qs = bad ? 0 : query_start(p.spec.q_start, b, np, p.S_q);
  int64_t jlo = 0, jhi = bad ? 0 : np;
  if (p.fused && !bad) fused_hull(p, b, np, qs, jlo, jhi);
  const int64_t t_begin = jlo >= jhi ? 0 : jlo / kTile;
  const int64_t t_end = jlo >= jhi ? 0 : (jhi + kTile - 1) / kTile;
  const int n_range = static_cast<int>(t_end - t_begin);

  if (p.bias && n_range > 0) {
    const int64_t k_lo = t_begin * kTile, k_hi = min(t_end * kTile, max_seq);
    const uint32_t row_bytes = static_cast<uint32_t>((k_hi - k_lo) * 2);
    const uint32_t pitch = (row_bytes + 127u) & ~127u;
    if (static_cast<int64_t>(pitch) * p.S_q <= kPlanScanBytes) {
      if (tid == 0) {
        ptx::mbar_arrive_expect_tx(bar, row_bytes * p.S_q);
        for (int i = 0; i < p.S_q; ++i)
          ptx::bulk_load(rows + i * pitch, p.bias + (static_cast<int64_t>(b) * p.S_q + i) * max_seq + k_lo,
                         row_bytes, bar);
      }
      const bool ok = ptx::mbar_wait_bounded(bar, 0, kWaitPolls);
      if (!ok) report(p.status, EXTKV_DEV_TIMEOUT);
      for (int t = tid; t < n_range; t += T) {
        bool live = false;
        for (int i = 0; i < p.S_q && ok; ++i) {
          const uint4* r = reinterpret_cast<const uint4*>(rows + i * pitch + t * 32);
          const int64_t j0 = k_lo + t * kTile;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (j0 + 8 * h >= k_hi) break;  // beyond the copied row (max_seq % 16 == 8)
            const uint4 v = r[h];
            const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
            for (int q = 0; q < 8; ++q) live = live || (j0 + 8 * h + q < np && bf16_bits_to_float(e[q]) > lowest);
          }
        }
        flags[t] = live;
      }
    } else {
      for (int t = tid; t < n_range; t += T) {
        bool live = false;
        for (int i = 0; i < p.S_q; ++i) {
          const __nv_bfloat16* r = p.bias + (static_cast<int64_t>(b) * p.S_q + i) * max_seq;
          for (int q = 0; q < kTile; ++q) {
            const int64_t j = (t_begin + t) * kTile + q;
            live = live || (j < np && Elem<__nv_bfloat16>::load(r, j) > lowest);
          }
        }
        flags[t] = live;
      }
    }
  } else {
    for (int t = tid; t < n_range; t += T) {
      bool live = true;  // only nonpad masks: every tile below it
      if (p.fused) {
        const int64_t k0 = (t_begin + t) * kTile;
        live = false;
        for (int i = 0; i < p.S_q && !live; ++i) {
          const RowWindow w = row_window(p.spec, b, qs + i, np);
          const int64_t a0 = max(k0, max(w.band_lo, int64_t(0))), a1 = min(k0 + kTile, min(w.band_hi, np));
          const int64_t s0 = max(k0, max(w.span_lo, int64_t(0))), s1 = min(k0 + kTile, min(w.span_hi, np));
          live = a0 < a1 || s0 < s1;
        }
      }
      flags[t] = live;
    }
  }
  __syncthreads();
  // compaction into the batch's tile list
  const int seg = (n_range + T - 1) / T;
  const int my_lo = min(n_range, tid * seg), my_hi = min(n_range, my_lo + seg);
  int cnt = 0;
  for (int t = my_lo; t < my_hi; ++t) cnt += flags[t];
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
  for (int w2 = 0; w2 < T / 32; ++w2) {
    if (w2 < warp) base += warp_tot[w2];
    total += warp_tot[w2];
  }
  int pos = base + incl - cnt;
  uint16_t* list = p.tiles + static_cast<int64_t>(b) * p.max_tiles;
  for (int t = my_lo; t < my_hi; ++t)
    if (flags[t]) list[pos++] = static_cast<uint16_t>(t_begin + t);
  if (tid == 0) p.count[b] = total;
  for (int h = tid; h < p.Hkv; h += T) p.counters[static_cast<int64_t>(b) * p.Hkv + h] = 0;
  if (total == 0) {
    // no live tile: every row of the batch's units is an exact zero row
    uint4* dst = reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(b) * p.Hq * p.S_q * p.D);
    const int64_t nvec = static_cast<int64_t>(p.Hq) * p.S_q * p.D / 8;
    for (int64_t i = tid; i < nvec; i += T) dst[i] = make_uint4(0, 0, 0, 0);
  }
}

// ---- decode: one warp streams its slice of the work sequence ----------------------

template <int D, int SPW>
struct Smem {
  static constexpr int kBoxes = D / 64;                    // 64-column TMA boxes
  static constexpr int kTileBytes = kBoxes * kTile * 128;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;       // K then V
  static constexpr int kQBytes = kBoxes * 1024;            // 8 rows x D bf16
  static constexpr int kQ = SPW * kStageBytes;             // two Q slots
  static constexpr int kTerm = kQ + 2 * kQBytes;           // per stage: 8 rows x 16 keys bf16
  static constexpr int kBars = kTerm + SPW * 256;          // SPW stages + 2 Q slots
  static constexpr int kPrefix = kBars + (SPW + 2) * 8;    // int32 [kMaxB + 1]
  static constexpr int kNonpad = kPrefix + (kMaxB + 1) * 4 + 12;  // int32 [kMaxB]
  static constexpr int kWork = kNonpad + kMaxB * 4;        // uint32 [kMaxWork]
  static constexpr int kEnd = kWork + kMaxWork * 4;
  static constexpr size_t bytes() { return 1024 + kEnd; }
};

template <int D, int SPW>
__global__ void __launch_bounds__(32) attn_decode_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap tmap,
    const DecodeParams p) {
  using S = Smem<D, SPW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars);  // stages, Q slots
  uint64_t* qbars = bars + SPW;
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + S::kPrefix);
  int32_t* np_s = reinterpret_cast<int32_t*>(smem + S::kNonpad);
  uint32_t* work = reinterpret_cast<uint32_t*>(smem + S::kWork);
  const int lane = threadIdx.x;
  const int c = blockIdx.x;
  const float lowest = Elem<__nv_bfloat16>::lowest();

  if (lane == 0) {
    for (int s = 0; s < SPW + 2; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&kmap);
    ptx::prefetch_tensormap(&vmap);
    ptx::prefetch_tensormap(&qmap);
  }
  __syncwarp();
  // Nothing above reads an input; everything below may read what the plan
  // (and the kernels before it) wrote.
  ptx::grid_dependency_wait();

  // prefix[b] = first work item of batch b (Hkv units of count[b] tiles each)
  int run = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int v = 0;
    if (b < p.B) {
      v = p.count[b] * p.Hkv;
      np_s[b] = static_cast<int32_t>(p.nonpad[b]);  // batches with tiles have 0 <= nonpad <= max_seq
    }
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (b < p.B) prefix[b] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) prefix[p.B] = run;
  __syncwarp();
  const int64_t T = run;
  // Slice over min(G, T) CTAs so that every slice holds at least one item and
  // the CTAs covering a unit are exactly a contiguous run of non-empty slices.
  const int G = static_cast<int>(T < p.G ? T : static_cast<int64_t>(p.G));
  if (c >= G) return;
  const int64_t x0 = (static_cast<int64_t>(c) * T) / G, x1 = (static_cast<int64_t>(c + 1) * T) / G;
  const int n = static_cast<int>(x1 - x0);

  // batch of work item x: last b with prefix[b] <= x and a non-empty range
  auto batch_of = [&](int64_t x) {
    int lo = 0, hi = p.B;  // prefix[lo] <= x < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= x) lo = mid;
      else hi = mid;
    }
    return lo;
  };
  // CTA whose slice holds item x
  auto cta_of = [&](int64_t x) {
    int64_t cc = (x * G) / (T > 0 ? T : 1);
    while (cc + 1 < G && ((cc + 1) * T) / G <= x) ++cc;
    while (cc > 0 && (cc * T) / G > x) --cc;
    return static_cast<int>(cc);
  };
  // work items of the slice: (unit << 16) | tile
  for (int k = lane; k < n; k += 32) {
    const int64_t x = x0 + k;
    const int b = batch_of(x);
    const int cnt = (prefix[b + 1] - prefix[b]) / p.Hkv;
    const int r = static_cast<int>(x - prefix[b]);
    const int kvh = r / cnt, kk = r % cnt;
    const uint32_t tile = p.tiles[static_cast<int64_t>(b) * p.max_tiles + kk];
    work[k] = (static_cast<uint32_t>(b * p.Hkv + kvh) << 16) | tile;
  }
  __syncwarp();

  // ---- producer (lane 0 issues TMA; cursors are warp-uniform) ----
  int pk = 0;            // next item to issue
  int p_unit = -1, p_seg = -1;
  int c_seg = 0;         // segment the consumer is in
  const uint32_t stage_tx = S::kStageBytes + (p.tile_term ? 32u * p.S_q : 0u);
  auto unit_of = [&](int k) { return static_cast<int>(work[k] >> 16); };
  auto fill = [&](int consumed) {
    while (pk < n && pk < consumed + SPW) {
      const int u = unit_of(pk);
      const int b = u / p.Hkv, kvh = u % p.Hkv;
      if (u != p_unit) {
        if (p_seg + 1 > c_seg + 1) break;  // the Q slot of segment p_seg+1 is still in use
        ++p_seg;
        p_unit = u;
        if (lane == 0) {
          const int slot = p_seg & 1;
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_expect_tx(&qbars[slot], S::kQBytes);
          const int64_t row0 = (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(kvh) * p.g) * p.S_q;
          for (int cb = 0; cb < S::kBoxes; ++cb)
            ptx::tma_load_2d(smem + S::kQ + slot * S::kQBytes + cb * 1024, &qmap, &qbars[slot], cb * 64,
                             static_cast<int32_t>(row0));
        }
      }
      if (lane == 0) {
        const int st = pk % SPW;
        const int32_t key0 = static_cast<int32_t>(work[pk] & 0xFFFFu) * kTile;
        const int32_t bh = b * p.Hkv + kvh;
        uint8_t* dst = smem + st * S::kStageBytes;
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(&bars[st], stage_tx);
#pragma unroll
        for (int cb = 0; cb < S::kBoxes; ++cb) {
          ptx::tma_load_3d(dst + cb * kTile * 128, &kmap, &bars[st], cb * 64, key0, bh);
          ptx::tma_load_3d(dst + S::kTileBytes + cb * kTile * 128, &vmap, &bars[st], cb * 64, key0, bh);
        }
        if (p.tile_term) ptx::tma_load_2d(smem + S::kTerm + st * 256, &tmap, &bars[st], key0, b * p.S_q);
      }
      ++pk;
    }
  };
  fill(0);

  // ---- consumer ----
  constexpr bool kQReg = D <= 256;
  constexpr int kKSteps = D / 16;
  constexpr int kAcc = kKSteps >= 16 ? 4 : 2;  // independent QK^T accumulator chains
  uint32_t qf[kQReg ? kKSteps : 1][2];
  const int r_lane[2] = {2 * (lane & 3), 2 * (lane & 3) + 1};
  const bool row_ok[2] = {r_lane[0] < p.R, r_lane[1] < p.R};
  const int i_row[2] = {r_lane[0] % p.S_q, r_lane[1] % p.S_q};
  float o[D / 16][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  RowWindow win[2];
  int64_t np = 0;
  int cur_unit = -1, seg_start = 0;
  bool failed = false;
  uint32_t q_s = 0;

  auto q_frag = [&](int kp, uint32_t* f4) {  // k-steps 2kp and 2kp+1
    const int cb = kp >> 1, jb = (kp & 1) * 4 + (lane >> 3), r = lane & 7;
    ptx::ldmatrix_x4(f4[0], f4[1], f4[2], f4[3], q_s + cb * 1024 + r * 128 + ((jb ^ r) << 4));
  };

  // Finishes the segment of unit `u` (items [seg_start, k_end) of the slice).
  auto finish = [&](int u, int k_end) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
      l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
      l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
    }
    const int b = u / p.Hkv, kvh = u % p.Hkv;
    const int cnt = (prefix[b + 1] - prefix[b]) / p.Hkv;
    const int64_t ub = prefix[b] + static_cast<int64_t>(kvh) * cnt;  // unit's first item
    const int c_first = cta_of(ub), c_last = cta_of(ub + cnt - 1);
    const int64_t row0 = (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(kvh) * p.g) * p.S_q;
    if (c_first == c_last) {
      // the whole unit is in this slice: normalised output (zero rows by selection)
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        const int d = mt * 16 + (lane >> 2);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (!row_ok[e]) continue;
          const bool live = l_run[e] > 0.f && !failed;
          const float inv = live ? 1.f / l_run[e] : 0.f;
          __nv_bfloat16* yr = p.y + (row0 + r_lane[e]) * D;
          yr[d] = __float2bfloat16_rn(live ? o[mt][e] * inv : 0.f);
          yr[d + 8] = __float2bfloat16_rn(live ? o[mt][2 + e] * inv : 0.f);
        }
      }
      return;
    }
    // split unit: leave a partial; the last slice to finish merges
    const int slot = seg_start == 0 ? 0 : 1;
    constexpr int PS = 2 * kRows + kRows * D;
    float* part = p.part + (static_cast<int64_t>(c) * 2 + slot) * PS;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int d = mt * 16 + (lane >> 2);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        part[2 * kRows + r_lane[e] * D + d] = o[mt][e];
        part[2 * kRows + r_lane[e] * D + d + 8] = o[mt][2 + e];
      }
    }
    if (lane < 4) {
      part[r_lane[0]] = failed ? -INFINITY : m_run[0];
      part[r_lane[1]] = failed ? -INFINITY : m_run[1];
      part[kRows + r_lane[0]] = failed ? 0.f : l_run[0];
      part[kRows + r_lane[1]] = failed ? 0.f : l_run[1];
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&p.counters[u], 1) == c_last - c_first;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    // merge the partials of CTAs c_first..c_last; slot 0 where the unit is
    // that slice's first segment, slot 1 where it is its last
    const int nseg = c_last - c_first + 1;
    for (int r = 0; r < p.R; ++r) {
      float M = -INFINITY;
      for (int s0 = 0; s0 < nseg; s0 += 32) {
        const int cc = c_first + s0 + lane;
        if (s0 + lane < nseg) {
          const int sl = (static_cast<int64_t>(cc) * T) / G >= ub ? 0 : 1;
          M = fmaxf(M, __ldcg(p.part + (static_cast<int64_t>(cc) * 2 + sl) * PS + r));
        }
      }
      for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
      const float ref = M == -INFINITY ? 0.f : M;
      float L = 0.f;
      for (int s0 = 0; s0 < nseg; s0 += 32) {
        const int cc = c_first + s0 + lane;
        if (s0 + lane < nseg) {
          const int sl = (static_cast<int64_t>(cc) * T) / G >= ub ? 0 : 1;
          const float* pp = p.part + (static_cast<int64_t>(cc) * 2 + sl) * PS;
          L += __ldcg(pp + kRows + r) * exp2_scaled(__ldcg(pp + r) - ref);
        }
      }
      for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int d4 = lane * 4; d4 < D; d4 += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < nseg; ++s) {
          const int cc = c_first + s;
          const int sl = (static_cast<int64_t>(cc) * T) / G >= ub ? 0 : 1;
          const float* pp = p.part + (static_cast<int64_t>(cc) * 2 + sl) * PS;
          const float wgt = exp2_scaled(__ldcg(pp + r) - ref);
          const float4 v = __ldcg(reinterpret_cast<const float4*>(pp + 2 * kRows + r * D + d4));
          acc.x = fmaf(v.x, wgt, acc.x);
          acc.y = fmaf(v.y, wgt, acc.y);
          acc.z = fmaf(v.z, wgt, acc.z);
          acc.w = fmaf(v.w, wgt, acc.w);
        }
        __nv_bfloat16* yr = p.y + (row0 + r) * D + d4;
        const bool live = L > 0.f;
        yr[0] = __float2bfloat16_rn(live ? acc.x * inv : 0.f);
        yr[1] = __float2bfloat16_rn(live ? acc.y * inv : 0.f);
        yr[2] = __float2bfloat16_rn(live ? acc.z * inv : 0.f);
        yr[3] = __float2bfloat16_rn(live ? acc.w * inv : 0.f);
      }
    }
  };

  for (int k = 0; k < n; ++k) {
    const int u = unit_of(k);
    if (u != cur_unit) {
      if (cur_unit >= 0) {
        finish(cur_unit, k);
        ++c_seg;
        fill(k);  // the finished segment's Q slot is free again
      }
      cur_unit = u;
      seg_start = k;
      const int b = u / p.Hkv;
      np = np_s[b];
      if (p.fused) {
        const int64_t qs = query_start(p.spec.q_start, b, np, p.S_q);
        for (int e = 0; e < 2; ++e) win[e] = row_window(p.spec, b, qs + i_row[e], np);
      }
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
      const int slot = c_seg & 1;
      q_s = ptx::smem_u32(smem + S::kQ + slot * S::kQBytes);
      failed = failed || __any_sync(0xffffffffu, !ptx::mbar_wait_bounded(&qbars[slot], (c_seg >> 1) & 1, kWaitPolls));
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
    }
    if (failed) break;
    const int st = k % SPW;
    if (__any_sync(0xffffffffu, !ptx::mbar_wait_bounded(&bars[st], (k / SPW) & 1, kWaitPolls))) {
      failed = true;
      break;
    }
    uint8_t* kst = smem + st * S::kStageBytes;
    const uint32_t k_s = ptx::smem_u32(kst), v_s = k_s + S::kTileBytes;
    const uint16_t* term = reinterpret_cast<const uint16_t*>(smem + S::kTerm + st * 256);
    const int64_t key0 = static_cast<int64_t>(work[k] & 0xFFFFu) * kTile;

    // S^T (16 keys x 8 rows) = K (16 x D) Q^T (D x 8), kAcc interleaved chains
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

    // scale + bias + mask; s[e]: key = lane/4 (+8 for e >= 2), row r_lane[e & 1]
    bool dead[2];  // key (lane/4, +8) masked for both of this lane's rows
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int kl = (lane >> 2) + 8 * kk;
      const int64_t j = key0 + kl;
      dead[kk] = true;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float& sv = s[2 * kk + e];
        bool live = row_ok[e] && j < np;
        float bv = 0.f;
        if (live) {
          if (p.bias) {
            bv = bf16_bits_to_float(term[i_row[e] * kTile + kl]);
            live = bv > lowest;
          } else if (p.fused) {
            live = win[e].allowed(j);
            if (live && p.tile_term) {
              bv = bf16_bits_to_float(term[i_row[e] * kTile + kl]);
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
      uint8_t* vt = kst + S::kTileBytes;  // each key owns kBoxes lines of 128 B
      for (int w = lane; w < kTile * S::kBoxes * 8; w += 32) {
        const int key = w / (S::kBoxes * 8), rem = w % (S::kBoxes * 8);
        if ((dead_keys >> key) & 1) {
          const int cb = rem >> 3, ch = rem & 7;
          *reinterpret_cast<uint4*>(vt + cb * (kTile * 128) + key * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
    }

    // online softmax, rows r_lane[0], r_lane[1]
    float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
    }
    float pr[4], corr[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float m_new = fmaxf(m_run[e], mx[e]);
      const float ref = m_new == -INFINITY ? 0.f : m_new;  // never -inf - -inf
      corr[e] = exp2_scaled(m_run[e] - ref);
      pr[e] = exp2_scaled(s[e] - ref);
      pr[2 + e] = exp2_scaled(s[2 + e] - ref);
      l_run[e] = fmaf(l_run[e], corr[e], pr[e] + pr[2 + e]);
      m_run[e] = m_new;
    }
    if (!__all_sync(0xffffffffu, corr[0] == 1.f && corr[1] == 1.f)) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[mt][0] *= corr[0];
        o[mt][1] *= corr[1];
        o[mt][2] *= corr[0];
        o[mt][3] *= corr[1];
      }
    }
    // P^T as the B operand: transpose the two 8x8 blocks (keys 0-7, 8-15)
    const uint32_t pb0 = ptx::movmatrix_trans(ptx::pack_bf16x2(pr[0], pr[1]));
    const uint32_t pb1 = ptx::movmatrix_trans(ptx::pack_bf16x2(pr[2], pr[3]));

    // O^T (D x 8) += V^T (D x 16) P^T (16 x 8)
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int cb = mt >> 2, j0 = (mt & 3) * 2;
      const int key = (lane & 7) + (lane >> 4) * 8, j = j0 + ((lane >> 3) & 1);
      uint32_t a0, a1, a2, a3;
      ptx::ldmatrix_x4_trans(a0, a1, a2, a3, v_s + cb * (kTile * 128) + key * 128 + ((j ^ (key & 7)) << 4));
      ptx::mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    fill(k + 1);  // refill the stage just consumed
  }
  if (failed && lane == 0) report(p.status, EXTKV_DEV_TIMEOUT);
  // Partials of a failed slice carry max -inf and sum 0, so the other slices'
  // merges stay finite; the affected units' output is stale (flagged).
  if (cur_unit >= 0) finish(cur_unit, n);
  if (failed) {
    // wait (bounded) for every load still in flight before the CTA exits
    for (int j = 0; j < pk; ++j) ptx::mbar_wait_bounded(&bars[j % SPW], (j / SPW) & 1, kWaitPolls);
    for (int sg = 0; sg <= p_seg; ++sg) ptx::mbar_wait_bounded(&qbars[sg & 1], (sg >> 1) & 1, kWaitPolls);
  }
}

// ---- host ---------------------------------------------------------------------------

template <int D>
int persistent_grid(int64_t units, int64_t max_tiles) {
  using Cfg = DecodeCfg<D>;
  using S = Smem<D, Cfg::SPW>;
  static std::mutex mu;
  static int cached_dev = -1, cached_occ = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  int occ;
  {
    std::lock_guard<std::mutex> g(mu);
    if (cached_dev != dev) {
      auto kern = attn_decode_kernel<D, Cfg::SPW>;
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(S::bytes()));
      int o = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, 32, S::bytes()) != cudaSuccess || o <= 0) {
        (void)cudaGetLastError();
        o = 1;
      }
      cached_occ = o;
      cached_dev = dev;
    }
    occ = cached_occ;
  }
  const int64_t g = static_cast<int64_t>(occ) * num_sms();
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g, units * max_tiles)));
}

int grid_for(int64_t D, int64_t units, int64_t max_tiles) {
  switch (D) {
    case 64: return persistent_grid<64>(units, max_tiles);
    case 128: return persistent_grid<128>(units, max_tiles);
    case 256: return persistent_grid<256>(units, max_tiles);
    default: return persistent_grid<512>(units, max_tiles);
  }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const char** name) {
  using Cfg = DecodeCfg<D>;
  constexpr int SPW = Cfg::SPW;
  using S = Smem<D, SPW>;
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  const int64_t units = a.B * a.Hkv;
  const int G = persistent_grid<D>(units, max_tiles);
  const WsLayout ws = ws_layout(a.B, units, max_tiles, G, D);
  if (!a.workspace || a.ws_bytes < ws.total) return cudaErrorInvalidValue;
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);

  CUtensorMap kmap, vmap, qmap, tmap;
  const uint64_t kv_dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(units)};
  const uint64_t kv_strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.max_seq) * D * 2};
  const uint32_t kv_box[3] = {64, kTile, 1};
  const uint64_t q_dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.B * a.Hq * a.S_q)};
  const uint64_t q_strides[1] = {static_cast<uint64_t>(D) * 2};
  const uint32_t q_box[2] = {64, kRows};
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 3, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 3, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&qmap, a.q, 2, q_dims, q_strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // per-tile bias or extra-term block: rows (b, i) of B*S_q, 16 keys x S_q rows
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
  prm.y = static_cast<__nv_bfloat16*>(a.y);
  prm.bias = static_cast<const __nv_bfloat16*>(a.bias);
  prm.spec = BiasSpec{a.causal, a.window, a.span_offsets, a.spans, a.extra, a.q_start};
  prm.fused = a.fused;
  prm.tile_term = term != nullptr;
  prm.nonpad = a.nonpad;
  prm.scale = a.scale;
  prm.B = static_cast<int>(a.B);
  prm.Hq = static_cast<int>(a.Hq);
  prm.Hkv = static_cast<int>(a.Hkv);
  prm.S_q = static_cast<int>(a.S_q);
  prm.g = static_cast<int>(a.Hq / a.Hkv);
  prm.R = static_cast<int>(a.Hq / a.Hkv * a.S_q);
  prm.D = D;
  prm.max_seq = a.max_seq;
  prm.max_tiles = max_tiles;
  prm.G = G;
  prm.count = reinterpret_cast<int32_t*>(wsb + ws.count);
  prm.tiles = reinterpret_cast<uint16_t*>(wsb + ws.tiles);
  prm.counters = reinterpret_cast<int32_t*>(wsb + ws.counters);
  prm.part = reinterpret_cast<float*>(wsb + ws.part);
  prm.status = a.status;

  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;

  // plan
  const size_t plan_smem = 128 + ((max_tiles + 127) / 128) * 128 + kPlanScanBytes + 16;
  cudaError_t e = cudaFuncSetAttribute(decode_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan_smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B));
  cfg.blockDim = dim3(kPlanThreads);
  cfg.dynamicSmemBytes = plan_smem;
  cfg.stream = a.stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_plan_kernel, prm);
  if (e != cudaSuccess) return e;

  // decode
  auto kern = attn_decode_kernel<D, SPW>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(S::bytes()));
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = S::bytes();
  e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, qmap, tmap, prm);
  if (e != cudaSuccess) return e;
  *name = "attn_decode_streamk_mma";
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t D) {
  (void)Hq;
  (void)S_q;
  const int64_t max_tiles = (max_seq + kTile - 1) / kTile;
  const int64_t units = B * Hkv;
  return ws_layout(B, units, max_tiles, grid_for(D, units, max_tiles), D).total;
}

bool decode_supported(const AttnArgs& a) {
  if (a.dtype != EXTKV_BF16) return false;
  if (a.D != 64 && a.D != 128 && a.D != 256 && a.D != 512) return false;
  if ((a.Hq / a.Hkv) * a.S_q > kRows) return false;
  // 16-byte rows for the bias / extra-term block copies
  if ((a.bias || (a.fused && a.extra)) && a.max_seq % 8) return false;
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  const int64_t units = a.B * a.Hkv;
  if (a.B > kMaxB || units >= 65536 || max_tiles > 65535) return false;
  if (a.B * a.Hq * a.S_q > 0x7fffffff || units * max_tiles > 0x7fffffff) return false;
  // one slice of the work sequence must fit the CTA's work table
  const int64_t G = grid_for(a.D, units, max_tiles);
  if ((units * max_tiles + G - 1) / G > kMaxWork) return false;
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
