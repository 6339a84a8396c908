// attn_decode.cuh -- stream-K split-KV decode attention over the external
// static cache.
//
// Work unit: one (batch b, KV head, row group): up to 8 of the KV head's
// R = (Hq/Hkv) * S_q query rows (R <= 64, in at most 8 groups), which share
// every K/V row they read ("ONNX Domain Attention (Opset 23/24) CUDA
// Patterns", section 1: GQA by reshaping Q, no KV replication).  Decode is HBM-bound ("Skill: Attention Optimization": decode
// is memory-bandwidth bound regardless of kernel), so the aim is to stream
// every live K/V row exactly once with every SM busy to the end.  Q and K
// carry DK columns, V and Y DV (equal, or a pair of 128/256/512: the
// head_size != v_head_size case of "Skill: Attention Optimization", "ORT CUDA
// Attention Kernel Dispatch").
//
//   Live tiles: 16-key tiles holding at least one key some query row may
//     attend.  Without a bias they are the tiles below nonpad; with the fused
//     specification they follow from the rows' allowed intervals in closed
//     form (computed inside the decode kernel); with a materialised bias, a
//     plan kernel (one CTA per batch) bulk-copies the bias rows into shared
//     memory and lists the live tiles.  Tiles at or beyond nonpad, or fully
//     masked, are never loaded.
//   Decode kernel (persistent, one warp per CTA): the live tiles of all units
//     form one sequence of T items (unit-major); CTA c takes the slice
//     [c*T/G, (c+1)*T/G) -- equal work per CTA whatever the lengths
//     (stream-K).  Lane 0 streams the slice through SPW shared-memory stages
//     with TMA (one request each for the K and V tiles, 128-byte swizzle per
//     64 columns, plus the tile's bias or extra-term block), running ahead across units; Q
//     tiles are double-buffered per unit.  Per tile, on the tensor cores
//     (mma.sync m16n8k16 bf16, fp32 accumulation): S^T = K Q^T with the 16
//     keys on M and the <= 8 query rows on N; scale, bias, mask; online
//     softmax in fp32 (scores in natural units, the row maximum subtracted
//     before the base-2 scaling and exponentiation);
//     P^T moved into the B-operand layout with movmatrix; O^T += V^T P^T.
//     A unit wholly inside the slice is written directly; a unit split
//     across slices leaves an fp32 (max, sum, output) partial.
//   Merge kernel (one CTA per unit and group of output columns): combines a
//     split unit's partials, and writes the zero rows of units without a live tile.
//
// Masking and zero rows follow section 6 of the ORT page: a key is masked iff
// j >= nonpad[b] or bias <= lowest(T); masked scores become -inf by
// selection; V rows of keys no row of the unit attends are zeroed in shared
// memory before the PV product, so poisoned (even NaN) cache slots cannot
// reach the output; a row with no unmasked key is written as zeros.
#pragma once

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace extkv {

// A decode call's grid (G CTAs, occ resident per SM), the batches its shared
// tables hold (tb), the items its work list holds (wc), its longest slice and
// its dynamic shared memory.
struct DecodeShape {
  int G, tb, wc, occ;
  int64_t slice;
  size_t bytes;
};

namespace {

constexpr int kTile = 16;                  // keys per tile (M of the QK^T mma)
constexpr int kRows = 8;                   // query rows per unit (N of the mma)
constexpr int kMaxRowGroups = 8;           // units of 8 rows per KV head (g * S_q <= 64; S_q <= 8)
constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits
constexpr int kMaxWork = 512;              // items of one slice the default tables hold (plan mode)
constexpr int kMaxB = 256;                 // batches the default tables hold (shared memory)
constexpr int kMaxBatches = 1024;          // batches the decode kernel takes (larger tables)
constexpr int kWorkCap = 16384;            // items of one slice it takes
constexpr int kPlanThreads = 256;
constexpr int kPlanScanBytes = 64 * 1024;  // bias rows staged by the plan
constexpr int kMergeThreads = 256;

enum Mode { kNone = 0, kBias = 1, kFused = 2, kFusedExtra = 3 };

template <int D>
struct DecodeCfg;  // SPW: shared-memory stages of the warp
template <>
struct DecodeCfg<64> {
  static constexpr int SPW = 4;
};
template <>
struct DecodeCfg<128> {
  static constexpr int SPW = 3;
};
template <>
struct DecodeCfg<256> {
  static constexpr int SPW = 2;
};
template <>
struct DecodeCfg<512> {
  static constexpr int SPW = 2;
};

// ---- workspace ----------------------------------------------------------------

struct WsLayout {
  size_t count, tiles, info, part, total;
};

// floats of one partial: max[8], sum[8], then the unit's R rows of Dv
inline int64_t part_floats(int64_t R, int64_t Dv) { return 2 * kRows + R * Dv; }

// A KV head's gr = (Hq / Hkv) * S_q query rows as units of at most 8 rows
inline int64_t row_groups(int64_t gr) { return (gr + kRows - 1) / kRows; }

WsLayout ws_layout(int64_t B, int64_t Hkv, int64_t max_tiles, int64_t G, int64_t R, int64_t Dv) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  WsLayout l;
  size_t o = 0;
  l.count = o;  // int32 live tiles per batch (plan mode)
  o = al(o + static_cast<size_t>(B) * 4);
  l.tiles = o;  // uint16 live tile list per batch (plan mode)
  o = al(o + static_cast<size_t>(B * max_tiles) * 2);
  l.info = o;  // int4 per unit: first CTA, slices, slot in the first CTA (Hkv: units of a batch)
  o = al(o + static_cast<size_t>(B * Hkv) * 16);
  l.part = o;  // per CTA, two partials: m[8], l[8], O[R][Dv] fp32
  o = al(o + static_cast<size_t>(G) * 2 * part_floats(R, Dv) * 4);
  l.total = o;
  return l;
}

struct DecodeParams {
  __nv_bfloat16* y;
  const __nv_bfloat16* q;
  const __nv_bfloat16* bias;  // materialised bias or nullptr
  BiasSpec spec;
  const int64_t* nonpad;
  float scale;
  float softcap;  // > 0: scores capped before the bias
  int B, Hq, Hkv, S_q, g, R, D;  // D: the value head size (columns of Y and of the partials)
  // R: query rows of a unit (at most 8); a KV head's GR = g * S_q rows form n_rg
  // units of up to 8 rows (row groups) that read the same K/V tiles
  int GR, n_rg;
  int max_seq, max_tiles;
  int G;     // CTAs of the decode grid
  int tb;    // batches the shared-memory tables hold (>= B, a multiple of 32)
  int PS;    // floats of one partial (part_floats(R, D))
  int plan;  // 1: live tiles come from the plan kernel
  int32_t* count;
  uint16_t* tiles;
  int4* info;  // per unit: {first CTA, number of slices, slot in the first CTA, 0}; slices 0: no live tile
  uint32_t polls;  // limit of the pipeline's barrier waits
  float* part;
  int32_t* status;
  // fused scatter (k_new == nullptr: none): the new rows (B, Hkv, S_new, D) go
  // to slots [write_idx[b], write_idx[b] + S_new) of the caches
  __nv_bfloat16* kc_w;
  __nv_bfloat16* vc_w;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int64_t* write_idx;
  int S_new;
};

// Allowed keys of one query position, as int32 bounds clipped to
// [-1, max_seq + 1] (membership of every slot in [0, max_seq) is unchanged).
struct Win32 {
  int np, blo, bhi, slo, shi;
  __device__ __forceinline__ bool allowed(int j) const {
    return j < np && ((j >= blo && j < bhi) || (j >= slo && j < shi));
  }
};

__device__ __forceinline__ int clip32(int64_t v, int64_t hi) {
  return static_cast<int>(v < -1 ? -1 : (v > hi ? hi : v));
}

__device__ __forceinline__ Win32 win32(const BiasSpec& spec, int b, int64_t p, int np, int max_seq) {
  const RowWindow w = row_window(spec, b, p, np);
  Win32 r;
  r.np = np;
  r.blo = clip32(w.band_lo, max_seq + 1);
  r.bhi = clip32(w.band_hi, max_seq + 1);
  r.slo = clip32(w.span_lo, max_seq + 1);
  r.shi = clip32(w.span_hi, max_seq + 1);
  if (w.span_lo >= w.span_hi) r.slo = r.shi = 0;
  return r;
}

// Live-tile ranges of a batch without a plan: at most two runs of tiles,
// [a1, a1+n1) then [a2, a2+n2).  Used for no bias (tiles below nonpad), and for
// the fused spec with one query row (band and span intervals) or without spans
// (consecutive rows' band intervals overlap into one interval).
struct Runs {
  int a1, n1, a2, n2;
  __device__ __forceinline__ int count() const { return n1 + n2; }
  __device__ __forceinline__ int tile(int k) const { return k < n1 ? a1 + k : a2 + (k - n1); }
};

__device__ __forceinline__ void add_interval(int lo, int hi, int& a, int& e, int& a2, int& e2) {
  // keys [lo, hi) -> tiles [lo/16, ceil(hi/16)); merged with what is there
  if (lo >= hi) return;
  const int t0 = lo / kTile, t1 = (hi + kTile - 1) / kTile;
  if (a >= e) {
    a = t0;
    e = t1;
  } else if (t0 <= e && t1 >= a) {
    a = min(a, t0);
    e = max(e, t1);
  } else if (t1 < a) {
    a2 = a;
    e2 = e;
    a = t0;
    e = t1;
  } else {
    a2 = t0;
    e2 = t1;
  }
}

template <int MODE>
__device__ __forceinline__ Runs batch_runs(const DecodeParams& p, int b, int64_t np64) {
  Runs r{0, 0, 0, 0};
  if (bad_nonpad(np64, p.max_seq)) return r;
  const int np = static_cast<int>(np64);
  if (MODE == kNone || MODE == kBias) {
    r.n1 = (np + kTile - 1) / kTile;
    return r;
  }
  const int64_t qs = query_start(p.spec.q_start, b, np64, p.S_q);
  int a = 0, e = 0, a2 = 0, e2 = 0;
  if (p.S_q == 1) {
    const Win32 w = win32(p.spec, b, qs, np, p.max_seq);
    add_interval(max(w.blo, 0), min(w.bhi, np), a, e, a2, e2);
    add_interval(max(w.slo, 0), min(w.shi, np), a, e, a2, e2);
  } else {  // no spans: one interval over the rows' bands
    const Win32 w0 = win32(p.spec, b, qs, np, p.max_seq);
    const Win32 w1 = win32(p.spec, b, qs + p.S_q - 1, np, p.max_seq);
    add_interval(max(w0.blo, 0), min(max(w0.bhi, w1.bhi), np), a, e, a2, e2);
  }
  r.a1 = a;
  r.n1 = e - a;
  r.a2 = a2;
  r.n2 = e2 - a2;
  return r;
}

// ---- plan: live tiles of one batch (materialised bias, or several rows with spans)

template <int MODE>
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
  const int max_seq = p.max_seq;
  const uint32_t row_bytes = static_cast<uint32_t>(max_seq) * 2;
  const uint32_t pitch = (row_bytes + 127u) & ~127u;
  const bool staged = MODE == kBias && static_cast<int64_t>(pitch) * p.S_q <= kPlanScanBytes;

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  // The whole bias rows are copied before nonpad is known: one round trip.
  if (staged && tid == 0) {
    ptx::mbar_arrive_expect_tx(bar, row_bytes * p.S_q);
    for (int i = 0; i < p.S_q; ++i)
      if (EXTKV_IN((static_cast<int64_t>(b) * p.S_q + i) * max_seq, max_seq,
                   static_cast<int64_t>(p.B) * p.S_q * max_seq, p.status))
        ptx::bulk_load(rows + i * pitch, p.bias + (static_cast<int64_t>(b) * p.S_q + i) * max_seq, row_bytes, bar);
  }
  const int64_t np64 = p.nonpad[b];
  const bool bad = bad_nonpad(np64, max_seq);
  if (bad && tid == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int n_range = (np + kTile - 1) / kTile;
  bool ok = true;
  if (staged) {
    ok = ptx::mbar_wait_bounded(bar, 0, kWaitPolls);
    if (!ok) report(p.status, EXTKV_DEV_TIMEOUT);
  }
  const int64_t qs = bad ? 0 : query_start(p.spec.q_start, b, np64, p.S_q);
  for (int t = tid; t < n_range; t += T) {
    bool live = false;
    const int j0 = t * kTile;
    if (MODE == kBias) {
      for (int i = 0; i < p.S_q && ok && !live; ++i) {
        if (staged) {
          const uint4* r = reinterpret_cast<const uint4*>(rows + i * pitch + t * 32);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (j0 + 8 * h >= max_seq) break;
            const uint4 v = r[h];
            const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
            for (int q = 0; q < 8; ++q) live = live || (j0 + 8 * h + q < np && bf16_bits_to_float(e[q]) > lowest);
          }
        } else {
          const __nv_bfloat16* r = p.bias + (static_cast<int64_t>(b) * p.S_q + i) * max_seq;
          for (int q = 0; q < kTile && j0 + q < np; ++q) live = live || Elem<__nv_bfloat16>::load(r, j0 + q) > lowest;
        }
      }
    } else {  // fused spec, several rows: some row's allowed set meets the tile
      for (int i = 0; i < p.S_q && !live; ++i) {
        const Win32 w = win32(p.spec, b, qs + i, np, max_seq);
        const int lo = max(j0, 0), hi = min(j0 + kTile, np);
        live = (max(lo, w.blo) < min(hi, w.bhi)) || (max(lo, w.slo) < min(hi, w.shi));
      }
    }
    flags[t] = live;
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
    if (flags[t]) {
      if (EXTKV_IN(static_cast<int64_t>(b) * p.max_tiles + pos, 1, static_cast<int64_t>(p.B) * p.max_tiles, p.status))
        list[pos] = static_cast<uint16_t>(t);
      ++pos;
    }
  if (tid == 0 && EXTKV_IN(b, 1, p.B, p.status)) p.count[b] = total;
}

// ---- per-batch tables shared by the decode and merge kernels --------------------

// Fills np_s[b] and (without a plan) runs_s[b], then prefix_s[b] = first item
// of batch b (Hkv * n_rg units of cnt[b] items each), prefix_s[B] = T.  One warp.
template <int MODE>
__device__ __forceinline__ int64_t batch_tables(const DecodeParams& p, int lane, int32_t* prefix_s,
                                                int32_t* np_s, Runs* runs_s, int32_t* wi_s) {
  int run = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int v = 0;
    if (b < p.B) {
      const int64_t np64 = p.nonpad[b];
      np_s[b] = bad_nonpad(np64, p.max_seq) ? 0 : static_cast<int>(np64);
      if (p.k_new) {  // first new slot of the fused scatter; -1: none or out of range (skipped)
        const int64_t w = p.write_idx[b];
        wi_s[b] = (w < 0 || w + p.S_new > p.max_seq) ? -1 : static_cast<int>(w);
      }
      int cnt;
      if (p.plan) {
        cnt = p.count[b];
        if (!EXTKV_IN(0, cnt, p.max_tiles, p.status)) cnt = 0;  // a count past the batch's tiles
      } else {
        const Runs r = batch_runs<MODE>(p, b, np64);
        runs_s[b] = r;
        cnt = r.count();
      }
      v = cnt * p.Hkv * p.n_rg;
    }
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (b < p.B) prefix_s[b] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) prefix_s[p.B] = run;
  __syncwarp();
  return run;
}

// last b with prefix[b] <= x (x < prefix[B])
__device__ __forceinline__ int batch_of(const int32_t* prefix, int B, int64_t x) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid;
    else hi = mid;
  }
  return lo;
}

// ---- decode: one warp streams its slice of the item sequence ---------------------

template <int DK, int DV, int SPW>
struct Smem {
  static constexpr int kKBoxes = DK / 64;                   // 64-column TMA boxes of a K tile
  static constexpr int kVBoxes = DV / 64;                   // and of a V tile
  static constexpr int kKTileBytes = kKBoxes * kTile * 128;
  static constexpr int kVTileBytes = kVBoxes * kTile * 128;
  static constexpr int kStageBytes = kKTileBytes + kVTileBytes;  // K then V
  static constexpr int kQBytes = kKBoxes * 1024;            // 8 rows x DK bf16
  // Q kept in registers, not in shared memory, where the output accumulator leaves room
  static constexpr bool kQReg = DK <= 256 && DK + DV <= 640;
  static constexpr int kQ = SPW * kStageBytes;             // two Q slots (DK = 512)
  static constexpr int kTerm = kQ + (kQReg ? 0 : 2 * kQBytes);  // per stage: 8 rows x 16 keys bf16
  static constexpr int kBars = kTerm + SPW * 256;          // SPW stages + 2 Q slots
  static constexpr int kPrefix = kBars + (SPW + 2) * 8;    // int32 [kMaxB + 1]
  static constexpr int kNp = kPrefix + (kMaxB + 1) * 4 + 12;  // int32 [kMaxB]
  static constexpr int kWi = kNp + kMaxB * 4;              // int32 [kMaxB]: write_idx (fused scatter)
  static constexpr int kRuns = kWi + kMaxB * 4;            // Runs [kMaxB] (no plan)
  static constexpr int kWork = kRuns;                      // uint16 [kMaxWork] (plan)
  static constexpr int kEnd = kRuns + kMaxB * 16;
  static_assert(kMaxWork * 2 <= kMaxB * 16, "the work table shares the runs table");
  // D = 256: four CTAs per SM, not the five the tables and stages would fit
  // (measured faster: 19.5 MB of requests in flight at start-up instead of
  // 24 MB, so the first tiles land sooner and the slices end closer together)
  static constexpr int kPad = (DK == 256 && DV == 256 && SPW == 2) ? 12 * 1024 : 0;
  static constexpr size_t bytes() { return 1024 + kEnd + kPad; }
};

// Position in the item sequence: unit (b, kvh, row group rg), tile index kk of cnt.
struct Cursor {
  int b, kvh, rg, kk, cnt;
};

// CAP: the scores are softcapped (a separate instantiation, so that the
// uncapped kernel is compiled as if the cap did not exist).
template <int DK, int DV, int SPW, int MODE, bool CAP>
__global__ void __launch_bounds__(32) attn_decode_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap tmap,
    const DecodeParams p) {
  using S = Smem<DK, DV, SPW>;
  constexpr bool kOneSize = DK == DV;  // the fused scatter takes one head size
  constexpr bool kTerm = MODE == kBias || MODE == kFusedExtra;  // per-tile bias block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars);  // stages, Q slots
  uint64_t* qbars = bars + SPW;
  // per-batch tables for p.tb batches, then the slice's work list over the runs table
  // (the default layout of Smem when p.tb = kMaxB)
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + S::kPrefix);
  int32_t* np_s = prefix + p.tb + 4;  // (tb + 1) entries and 12 bytes
  int32_t* wi_s = np_s + p.tb;
  Runs* runs_s = reinterpret_cast<Runs*>(wi_s + p.tb);
  uint16_t* work = reinterpret_cast<uint16_t*>(runs_s);
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
  // Nothing above reads an input; everything below may read what the
  // previous kernel in the stream wrote.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  const int64_t T = batch_tables<MODE>(p, lane, prefix, np_s, runs_s, wi_s);
  if (c == 0) {
    // units without a live tile (the merge kernel writes their zero rows)
    for (int b = lane; b < p.B; b += 32) {
      if (prefix[b + 1] != prefix[b]) continue;
      if (!p.plan && bad_nonpad(p.nonpad[b], p.max_seq)) report(p.status, EXTKV_DEV_BAD_NONPAD);
      for (int u = 0; u < p.Hkv * p.n_rg; ++u) p.info[b * p.Hkv * p.n_rg + u] = make_int4(-1, 0, 0, 0);
    }
  }
  // Slice over min(G, T) CTAs: every slice holds at least one item.
  const int G = static_cast<int>(T < p.G ? T : static_cast<int64_t>(p.G));
  // The fused scatter, this CTA's share (all CTAs together write every new
  // row into the caches).  Loads of other CTAs may see a row before or after
  // it is written; a tile that holds new rows is patched from k_new / v_new
  // in shared memory below.
  auto scatter_share = [&]() {
    if (!kOneSize || !p.k_new) return;
    constexpr int D = DK;
    const int vpr = D / 8;  // 16-byte vectors per row
    const int64_t total = static_cast<int64_t>(p.B) * p.Hkv * p.S_new * vpr;
    for (int64_t i = static_cast<int64_t>(c) * 32 + lane; i < total; i += static_cast<int64_t>(gridDim.x) * 32) {
      const int64_t row = i / vpr;  // over (b, kv head, s)
      const int v = static_cast<int>(i % vpr);
      const int sn = static_cast<int>(row % p.S_new);
      const int64_t bh = row / p.S_new;
      const int b = static_cast<int>(bh / p.Hkv);
      const int64_t w = p.write_idx[b];
      if (w < 0 || w + p.S_new > p.max_seq) {
        if (sn == 0 && v == 0 && bh % p.Hkv == 0) report(p.status, EXTKV_DEV_BAD_WRITE_IDX);
        continue;
      }
      const int64_t dst = (bh * p.max_seq + w + sn) * D + v * 8, src = row * D + v * 8;
      const int64_t n_bh = static_cast<int64_t>(p.B) * p.Hkv;
      if (!EXTKV_IN(dst, 8, n_bh * p.max_seq * D, p.status) || !EXTKV_IN(src, 8, n_bh * p.S_new * D, p.status))
        continue;
      *reinterpret_cast<uint4*>(p.kc_w + dst) = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
      *reinterpret_cast<uint4*>(p.vc_w + dst) = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
    }
  };
  if (c >= G) {
    scatter_share();
    return;
  }
  const int64_t x0 = (static_cast<int64_t>(c) * T) / G, x1 = (static_cast<int64_t>(c + 1) * T) / G;
  const int n = static_cast<int>(x1 - x0);

  const int upb = p.Hkv * p.n_rg;  // units of a batch
  auto cursor_at = [&](int64_t x) {
    Cursor q;
    q.b = batch_of(prefix, p.B, x);
    q.cnt = (prefix[q.b + 1] - prefix[q.b]) / upb;
    const int r = static_cast<int>(x - prefix[q.b]);
    const int u = r / q.cnt;
    q.kvh = u / p.n_rg;
    q.rg = u - q.kvh * p.n_rg;
    q.kk = r - u * q.cnt;
    return q;
  };
  auto advance = [&](Cursor& q) {
    if (++q.kk < q.cnt) return;
    q.kk = 0;
    if (++q.rg < p.n_rg) return;
    q.rg = 0;
    if (++q.kvh < p.Hkv) return;
    q.kvh = 0;
    do {
      ++q.b;
    } while (q.b < p.B && prefix[q.b + 1] == prefix[q.b]);
    if (q.b < p.B) q.cnt = (prefix[q.b + 1] - prefix[q.b]) / upb;
  };
  if (p.plan) {
    // the slice's tile numbers, from the plan's per-batch lists
    for (int k = lane; k < n; k += 32) {
      const Cursor q = cursor_at(x0 + k);
      const int64_t at = static_cast<int64_t>(q.b) * p.max_tiles + q.kk;
      work[k] = EXTKV_IN(at, 1, static_cast<int64_t>(p.B) * p.max_tiles, p.status) ? p.tiles[at] : 0;
    }
    __syncwarp();
  }
  auto tile_of = [&](const Cursor& q, int k) -> int {
    return p.plan ? static_cast<int>(work[k]) : runs_s[q.b].tile(q.kk);
  };

  // ---- producer: lane 0 issues TMA; the cursor is warp-uniform ----
  // Q of a unit: for DK <= 256 every lane loads its mma B fragments straight
  // into registers (a "next" set, copied to the current set when the consumer
  // starts the unit); for DK = 512 TMA fills one of two shared-memory slots.
  // Either way the producer may enter unit s+1 only once the consumer has
  // started unit s (p_seg <= c_seg + 1).
  constexpr bool kQReg = S::kQReg;
  constexpr int kKSteps = DK / 16;
  uint32_t qn[kQReg ? kKSteps : 1][2];
  Cursor pc = cursor_at(x0);
  int pk = 0, p_seg = -1, c_seg = -1;
  const uint32_t stage_tx = S::kStageBytes + (kTerm ? 32u * p.S_q : 0u);
  int p_row0 = 0, p_bh = 0, p_nr = 0;
  auto fill = [&](int consumed) {
    while (pk < n && pk < consumed + SPW) {
      bool q_regs = false;
      if (pk == 0 || pc.kk == 0) {  // first item of a unit: its Q rows
        if (p_seg + 1 > c_seg + 1) break;  // both Q slots busy
        ++p_seg;
        p_bh = pc.b * p.Hkv + pc.kvh;
        p_row0 = (pc.b * p.Hq + pc.kvh * p.g) * p.S_q + pc.rg * kRows;
        p_nr = min(kRows, p.GR - pc.rg * kRows);
        if constexpr (kQReg) {
          q_regs = true;  // loaded once this stage's requests are out
        } else if (lane == 0) {
          const int slot = p_seg & 1;
          ptx::mbar_arrive_expect_tx(&qbars[slot], S::kQBytes);
          ptx::tma_load_3d(smem + S::kQ + slot * S::kQBytes, &qmap, &qbars[slot], 0, p_row0, 0);
        }
      }
      {
        // the stage's requests from three lanes side by side (a request costs its
        // issuing thread a fixed time), after lane 0 has armed the barrier
        const int st = pk % SPW;
        const int key0 = tile_of(pc, pk) * kTile;
        uint8_t* dst = smem + st * S::kStageBytes;
        if (lane == 0) ptx::mbar_arrive_expect_tx(&bars[st], stage_tx);
        __syncwarp();
        if (lane == 0) ptx::tma_load_4d(dst, &kmap, &bars[st], 0, key0, 0, p_bh);
        else if (lane == 1) ptx::tma_load_4d(dst + S::kKTileBytes, &vmap, &bars[st], 0, key0, 0, p_bh);
        else if (kTerm && lane == 2) ptx::tma_load_2d(smem + S::kTerm + st * 256, &tmap, &bars[st], key0, pc.b * p.S_q);
      }
      if constexpr (kQReg) {
        if (q_regs) {
          // B fragment of k-step ks: the bf16 pair at (row lane/4, d = 16 ks + 2 (lane%4)), and d + 8
          const int row = lane >> 2;
          const bool qok =
              row < p_nr && EXTKV_IN(p_row0 + row, 1, static_cast<int64_t>(p.B) * p.Hq * p.S_q, p.status);
          const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + static_cast<int64_t>(p_row0 + row) * DK) + (lane & 3);
#pragma unroll
          for (int ks = 0; ks < kKSteps; ++ks) {
            qn[ks][0] = qok ? __ldg(qrow + 8 * ks) : 0u;
            qn[ks][1] = qok ? __ldg(qrow + 8 * ks + 4) : 0u;
          }
        }
      }
      ++pk;
      advance(pc);
    }
  };
  fill(0);
  scatter_share();  // this CTA's share, while its first loads are in flight

  // ---- consumer ----
  constexpr int kAcc = kKSteps >= 16 ? 4 : 2;  // independent QK^T accumulator chains
  uint32_t qf[kQReg ? kKSteps : 1][2];
  const int r0 = 2 * (lane & 3), r1 = r0 + 1;
  // this lane's two rows of the current unit: real or not, and their query positions
  bool ok0 = false, ok1 = false;
  int i0 = 0, i1 = 0;
  float o[DV / 16][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  Win32 w0{}, w1{};
  int np = 0;
  int w_new = -1;  // first new slot of the current unit's batch (fused scatter), -1: none
  bool failed = false;
  uint32_t q_s = 0;
  Cursor cc = cursor_at(x0);
  Cursor cur_unit = cc;
  int64_t ub = 0;  // first item of the current unit

  auto q_frag = [&](int kp, uint32_t* f4) {  // k-steps 2kp and 2kp+1
    const int cb = kp >> 1, jb = (kp & 1) * 4 + (lane >> 3), r = lane & 7;
    ptx::ldmatrix_x4(f4[0], f4[1], f4[2], f4[3], q_s + cb * 1024 + r * 128 + ((jb ^ r) << 4));
  };

  // Ends the current unit (this slice's items of it are done): direct output
  // when the whole unit was in the slice, else a partial for the merge.
  auto finish = [&]() {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
    const Cursor& u = cur_unit;
    const int64_t row0 =
        (static_cast<int64_t>(u.b) * p.Hq + static_cast<int64_t>(u.kvh) * p.g) * p.S_q + u.rg * kRows;
    if (ub >= x0 && ub + u.cnt <= x1) {
      const bool live0 = l0 > 0.f && !failed, live1 = l1 > 0.f && !failed;
      const float inv0 = live0 ? 1.f / l0 : 0.f, inv1 = live1 ? 1.f / l1 : 0.f;
      __nv_bfloat16* y0 = p.y + (row0 + r0) * DV;
      __nv_bfloat16* y1 = p.y + (row0 + r1) * DV;
      const int64_t n_y = static_cast<int64_t>(p.B) * p.Hq * p.S_q * DV;
      const bool yok0 = ok0 && EXTKV_IN((row0 + r0) * DV, DV, n_y, p.status);
      const bool yok1 = ok1 && EXTKV_IN((row0 + r1) * DV, DV, n_y, p.status);
#pragma unroll
      for (int mt = 0; mt < DV / 16; ++mt) {
        const int d = mt * 16 + (lane >> 2);
        if (yok0) {
          y0[d] = __float2bfloat16_rn(o[mt][0] * inv0);
          y0[d + 8] = __float2bfloat16_rn(o[mt][2] * inv0);
        }
        if (yok1) {
          y1[d] = __float2bfloat16_rn(o[mt][1] * inv1);
          y1[d + 8] = __float2bfloat16_rn(o[mt][3] * inv1);
        }
      }
      return;
    }
    // slot 0: the slice's first unit (it began at or before x0); slot 1: its last
    const int slot = ub <= x0 ? 0 : 1;
    if (!EXTKV_IN((static_cast<int64_t>(c) * 2 + slot) * p.PS, p.PS, static_cast<int64_t>(p.G) * 2 * p.PS, p.status))
      return;
    float* part = p.part + (static_cast<int64_t>(c) * 2 + slot) * p.PS;
    float* o0 = part + 2 * kRows + r0 * DV;
    float* o1 = part + 2 * kRows + r1 * DV;
#pragma unroll
    for (int mt = 0; mt < DV / 16; ++mt) {
      const int d = mt * 16 + (lane >> 2);
      if (ok0) {
        o0[d] = o[mt][0];
        o0[d + 8] = o[mt][2];
      }
      if (ok1) {
        o1[d] = o[mt][1];
        o1[d + 8] = o[mt][3];
      }
    }
    if (lane < 4) {
      part[r0] = failed ? -INFINITY : m0;
      part[r1] = failed ? -INFINITY : m1;
      part[kRows + r0] = failed ? 0.f : l0;
      part[kRows + r1] = failed ? 0.f : l1;
    }
  };

  for (int k = 0; k < n; ++k) {
    if (k == 0 || cc.kk == 0) {
      // a new unit starts at item k
      if (k > 0) finish();
      ++c_seg;
      if constexpr (kQReg) {
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
          qf[ks][0] = qn[ks][0];
          qf[ks][1] = qn[ks][1];
        }
      }
      fill(k);  // the producer may now enter the next unit
      cur_unit = cc;
      ub = x0 + k - cc.kk;
      {
        const int nr = min(kRows, p.GR - cc.rg * kRows);  // rows of this unit
        ok0 = r0 < nr;
        ok1 = r1 < nr;
        i0 = (cc.rg * kRows + r0) % p.S_q;
        i1 = (cc.rg * kRows + r1) % p.S_q;
      }
      if (cc.kk == 0 && lane == 0) {
        // this slice holds the unit's first item: record where its partials live
        const int64_t last = ub + cc.cnt - 1;
        const int c_last = static_cast<int>(((last + 1) * G - 1) / T);  // slice holding `last`
        const int64_t at = (static_cast<int64_t>(cc.b) * p.Hkv + cc.kvh) * p.n_rg + cc.rg;
        if (EXTKV_IN(at, 1, static_cast<int64_t>(p.B) * p.Hkv * p.n_rg, p.status))
          p.info[at] = make_int4(c, c_last - c + 1, ub <= x0 ? 0 : 1, 0);
      }
      np = np_s[cc.b];
      if (p.k_new) w_new = wi_s[cc.b];  // -1: the scatter skipped this batch, no patch
      if (MODE == kFused || MODE == kFusedExtra) {
        const int64_t qs = query_start(p.spec.q_start, cc.b, np, p.S_q);
        w0 = win32(p.spec, cc.b, qs + i0, np, p.max_seq);
        w1 = win32(p.spec, cc.b, qs + i1, np, p.max_seq);
      }
#pragma unroll
      for (int mt = 0; mt < DV / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      if constexpr (!kQReg) {
        const int slot = c_seg & 1;
        q_s = ptx::smem_u32(smem + S::kQ + slot * S::kQBytes);
        if (__any_sync(0xffffffffu, !ptx::mbar_wait_bounded(&qbars[slot], (c_seg >> 1) & 1, p.polls))) {
          failed = true;
          break;
        }
      }
    }
    const int st = k % SPW;
    if (__any_sync(0xffffffffu, !ptx::mbar_wait_bounded(&bars[st], (k / SPW) & 1, p.polls))) {
      failed = true;
      break;
    }
    uint8_t* kst = smem + st * S::kStageBytes;
    const uint32_t k_s = ptx::smem_u32(kst), v_s = k_s + S::kKTileBytes;
    const uint16_t* term = reinterpret_cast<const uint16_t*>(smem + S::kTerm + st * 256);
    const int key0 = tile_of(cc, k) * kTile;
    if (kOneSize && w_new >= 0 && key0 < w_new + p.S_new && key0 + kTile > w_new) {
      // new rows of this tile straight from k_new / v_new (what the cache
      // holds after the scatter), into the 128-byte-swizzled stage layout
      const int lo = max(key0, w_new), hi = min(key0 + kTile, w_new + p.S_new);
      constexpr int D = DK;
      constexpr int vpr = D / 8;
      const int64_t nb = static_cast<int64_t>(cc.b * p.Hkv + cc.kvh) * p.S_new;
      for (int idx = lane; idx < (hi - lo) * vpr; idx += 32) {
        const int key = lo + idx / vpr;
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

    // mask + bias in natural units: s = scale*qk + bias.  The base-2 scaling
    // comes only after the row maximum is subtracted, so an extreme finite
    // bias (beyond about 2.4e38 in magnitude) never overflows into a mask.
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
    // key q of a half is dead when its four lanes (4q..4q+3) all say so
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
    advance(cc);
    fill(k + 1);  // refill the stage just consumed
  }
  if (failed && lane == 0) report(p.status, EXTKV_DEV_TIMEOUT);
  // Partials of a failed slice carry max -inf and sum 0, so merges stay
  // finite; the affected units' output is stale (and flagged).
  finish();
  if (failed) {
    // wait (bounded, at the full limit) for every load still in flight before
    // the CTA exits: the newest request of each stage (items pk - SPW .. pk - 1;
    // a stage is refilled only after its previous item was consumed, so older
    // phases are complete) and the Q slots of the newest two units
    for (int j = pk > SPW ? pk - SPW : 0; j < pk; ++j)
      ptx::mbar_wait_bounded(&bars[j % SPW], (j / SPW) & 1, kWaitPolls);
    if (!kQReg)
      for (int sg = p_seg > 0 ? p_seg - 1 : 0; sg <= p_seg; ++sg)
        ptx::mbar_wait_bounded(&qbars[sg & 1], (sg >> 1) & 1, kWaitPolls);
  }
}

// ---- merge: split units' partials, and the zero rows of empty units -------------

// One CTA per (unit, group of output columns): thread (r, c) holds row r's
// float4 c of the group.  Each thread loads, for up to kPre slices at once,
// the slice's maximum and sum for its row and its partial float4, then forms
// the weights exp(max_s - M) in registers (maxima in natural units); slices
// are summed in slice order, so the result does not depend on timing.
template <int MODE>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p, int n_cg) {
  constexpr int kPre = 16;  // slices whose loads are in flight together
  const int u = blockIdx.x / n_cg, cg = blockIdx.x % n_cg;
  const int b = u / (p.Hkv * p.n_rg), kvh = (u / p.n_rg) % p.Hkv, rg = u % p.n_rg;
  const int D = p.D, R = min(kRows, p.GR - rg * kRows);  // rows of this unit
  const int cols = D / 4 / n_cg;  // float4 per row in this group
  const int i = threadIdx.x;
  const int r = i / cols, d4 = (cg * cols + i % cols) * 4;
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  const int4 info = p.info[u];
  const int64_t row0 = (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(kvh) * p.g) * p.S_q + rg * kRows;
  if (i >= R * cols) return;
  auto store = [&](const float4& acc) {
    if (!EXTKV_IN((row0 + r) * D + d4, 4, static_cast<int64_t>(p.B) * p.Hq * p.S_q * D, p.status)) return;
    __nv_bfloat16* yr = p.y + (row0 + r) * D + d4;
    uint2 pk;
    pk.x = ptx::pack_bf16x2(acc.x, acc.y);
    pk.y = ptx::pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(yr) = pk;
  };
  if (info.y == 0) {  // no live tile: an exact zero row
    store(make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const int ns = info.y;
  if (ns == 1) return;  // written by the decode kernel
  // the slices' partials, recorded by the decode kernel: inside the partial slots
  if (!EXTKV_IN(static_cast<int64_t>(info.x) * 2 * p.PS, static_cast<int64_t>(ns) * 2 * p.PS,
                static_cast<int64_t>(p.G) * 2 * p.PS, p.status) ||
      !EXTKV_IN(info.z, 1, 2, p.status))
    return;
  constexpr int PS = 2 * kRows;  // header floats of a partial
  const int stride = p.PS;
  // slice s of the unit: CTA info.x + s; the unit is the first unit of every
  // slice after the first, whose slot the decode kernel recorded
  auto part_of = [&](int sg) {
    const int slot = sg == 0 ? info.z : 0;
    return p.part + (static_cast<int64_t>(info.x + sg) * 2 + slot) * stride;
  };
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += kPre) {
    float m[kPre], l[kPre];
    float4 o[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      if (s0 + k < ns) {
        const float* pp = part_of(s0 + k);
        m[k] = __ldcg(pp + r);
        l[k] = __ldcg(pp + kRows + r);
        o[k] = __ldcg(reinterpret_cast<const float4*>(pp + PS + r * D + d4));
      } else {
        m[k] = -INFINITY;
        l[k] = 0.f;
        o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // a new maximum rescales what has been summed so far
    float mc = M;
#pragma unroll
    for (int k = 0; k < kPre; ++k) mc = fmaxf(mc, m[k]);
    if (mc != -INFINITY && mc != M) {
      const float c = M == -INFINITY ? 0.f : ptx::ex2((M - mc) * kLog2e);
      L *= c;
      acc.x *= c;
      acc.y *= c;
      acc.z *= c;
      acc.w *= c;
      M = mc;
    }
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const float w = m[k] == -INFINITY ? 0.f : ptx::ex2((m[k] - M) * kLog2e);
      L = fmaf(w, l[k], L);
      acc.x = fmaf(o[k].x, w, acc.x);
      acc.y = fmaf(o[k].y, w, acc.y);
      acc.z = fmaf(o[k].z, w, acc.z);
      acc.w = fmaf(o[k].w, w, acc.w);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;  // no unmasked key: zero row
  store(make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
}

// Column groups of the merge: enough CTAs that each holds about 64 threads.
int merge_groups(int R, int D) {
  const int per_row = D / 4;
  int n = 1;
  while (n * 2 <= per_row && R * per_row / (n * 2) >= 64) n *= 2;
  return n;
}

// ---- host ---------------------------------------------------------------------------

// Stages per warp for a pair of head sizes: as for the larger one.
template <int DK, int DV>
struct PairCfg {
  static constexpr int SPW = DecodeCfg<(DK > DV ? DK : DV)>::SPW;
};

// Shared memory of a decode CTA whose tables hold tb batches and a work list
// of wc items: the default layout (with its occupancy pad) at least.
template <int DK, int DV>
size_t decode_smem(int tb, int wc) {
  using S = Smem<DK, DV, PairCfg<DK, DV>::SPW>;
  const size_t tables = static_cast<size_t>(tb + 1) * 4 + 12 + static_cast<size_t>(tb) * 8 +
                        std::max<size_t>(static_cast<size_t>(tb) * 16, static_cast<size_t>(wc) * 2);
  return std::max<size_t>(S::bytes(), 1024 + S::kPrefix + tables);
}

// Resident decode CTAs per SM at `bytes` of shared memory (per device and size).
template <int DK, int DV>
int decode_occupancy(size_t bytes) {
  static std::mutex mu;
  struct Entry {
    int dev;
    size_t bytes;
    int occ;
  };
  static Entry entries[32];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> g(mu);
  for (int i = 0; i < n; ++i)
    if (entries[i].dev == dev && entries[i].bytes == bytes) return entries[i].occ;
  auto kern = attn_decode_kernel<DK, DV, PairCfg<DK, DV>::SPW, kBias, false>;
  int o = 0;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), bytes) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, 32, bytes) != cudaSuccess || o <= 0) {
    (void)cudaGetLastError();
    o = 0;
  }
  if (n < 32) entries[n++] = Entry{dev, bytes, o};
  return o;
}

// Grid and shared-memory tables of a call over B batches and at most
// items_max work items: the tables hold max(B, 256) batches and the longest
// slice; the slice follows from the grid, the grid from the shared memory the
// tables take (a few rounds settle it).  occ 0: the tables do not fit.
template <int DK, int DV>
DecodeShape decode_shape(int64_t B, int64_t items_max) {
  DecodeShape d;
  d.tb = static_cast<int>((std::max<int64_t>(B, kMaxB) + 31) / 32 * 32);
  d.wc = kMaxWork;
  for (int round = 0; round < 4; ++round) {
    d.bytes = decode_smem<DK, DV>(d.tb, d.wc);
    d.occ = decode_occupancy<DK, DV>(d.bytes);
    const int64_t g = static_cast<int64_t>(std::max(d.occ, 1)) * num_sms();
    d.G = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g, items_max)));
    d.slice = (items_max + d.G - 1) / d.G;
    if (d.slice <= d.wc || d.slice > kWorkCap) break;
    d.wc = static_cast<int>((d.slice + 63) / 64 * 64);
  }
  return d;
}

inline bool needs_plan(const AttnArgs& a) {
  if (a.bias) return true;
  if (!a.fused) return false;
  return a.S_q > 1 && a.spans != nullptr;
}

inline int mode_of(const AttnArgs& a) {
  if (a.bias) return kBias;
  if (!a.fused) return kNone;
  return a.extra ? kFusedExtra : kFused;
}

template <int DK, int DV, int MODE, bool CAP>
cudaError_t launch_dm(const AttnArgs& a, const DecodeParams& prm, const CUtensorMap& kmap,
                      const CUtensorMap& vmap, const CUtensorMap& qmap, const CUtensorMap& tmap,
                      int64_t max_tiles, size_t smem) {
  constexpr int SPW = PairCfg<DK, DV>::SPW;
  using S = Smem<DK, DV, SPW>;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = a.stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (prm.plan) {
    const size_t plan_smem = 128 + ((max_tiles + 127) / 128) * 128 + kPlanScanBytes + 16;
    auto pk = decode_plan_kernel<MODE == kBias ? kBias : kFused>;
    e = set_max_dynamic_smem(reinterpret_cast<const void*>(pk), plan_smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(a.B));
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = plan_smem;
    e = cudaLaunchKernelEx(&cfg, pk, prm);
    if (e != cudaSuccess) return e;
  }
  auto kern = attn_decode_kernel<DK, DV, SPW, MODE, CAP>;
  e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(prm.G));
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = smem;
  e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, qmap, tmap, prm);
  if (e != cudaSuccess) return e;
  const int n_cg = merge_groups(prm.R, DV);
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.Hkv * prm.n_rg * n_cg));
  cfg.blockDim = dim3(static_cast<unsigned>((prm.R * (DV / 4 / n_cg) + 31) / 32 * 32));
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<MODE>, prm, n_cg);
  if (e == cudaSuccess) note_launches(prm.plan ? 3 : 2);
  return e;
}

template <int DK, int DV, int MODE>
cudaError_t launch_dmc(const AttnArgs& a, const DecodeParams& prm, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& qmap, const CUtensorMap& tmap, int64_t max_tiles, size_t smem) {
  if constexpr (DK == DV) {
    return a.softcap > 0.f ? launch_dm<DK, DV, MODE, true>(a, prm, kmap, vmap, qmap, tmap, max_tiles, smem)
                           : launch_dm<DK, DV, MODE, false>(a, prm, kmap, vmap, qmap, tmap, max_tiles, smem);
  } else {  // two head sizes: no softcap instantiation (the prefill kernel takes that case)
    if (a.softcap > 0.f) return cudaErrorInvalidValue;
    return launch_dm<DK, DV, MODE, false>(a, prm, kmap, vmap, qmap, tmap, max_tiles, smem);
  }
}

template <int DK, int DV>
cudaError_t launch_d(const AttnArgs& a, const char** name) {
  const int64_t max_tiles = (a.max_seq + kTile - 1) / kTile;
  const int64_t units = a.B * a.Hkv;  // K/V heads (the views' last dimension)
  const int64_t gr = a.Hq / a.Hkv * a.S_q, n_rg = row_groups(gr);
  const DecodeShape shape = decode_shape<DK, DV>(a.B, units * n_rg * max_tiles);
  if (shape.occ <= 0 || shape.slice > shape.wc) return cudaErrorInvalidValue;
  const int G = shape.G;
  const WsLayout ws = ws_layout(a.B, a.Hkv * n_rg, max_tiles, G, std::min<int64_t>(gr, kRows), DV);
  if (!a.workspace || a.ws_bytes < ws.total) return cudaErrorInvalidValue;
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);

  // K/V and Q are read through views (d % 64, row, d / 64[, unit]) whose second
  // and third strides are not increasing: one TMA box then brings a whole tile
  // laid out as D/64 blocks of (rows x 128 B), each with the 128-byte swizzle --
  // the same shared-memory image as one box per 64 columns, in one request.
  CUtensorMap kmap, vmap, qmap, tmap;
  const uint64_t k_dims[4] = {64, static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(DK / 64),
                              static_cast<uint64_t>(units)};
  const uint64_t k_strides[3] = {static_cast<uint64_t>(DK) * 2, 128, static_cast<uint64_t>(a.max_seq) * DK * 2};
  const uint32_t k_box[4] = {64, kTile, static_cast<uint32_t>(DK / 64), 1};
  const uint64_t v_dims[4] = {64, static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(DV / 64),
                              static_cast<uint64_t>(units)};
  const uint64_t v_strides[3] = {static_cast<uint64_t>(DV) * 2, 128, static_cast<uint64_t>(a.max_seq) * DV * 2};
  const uint32_t v_box[4] = {64, kTile, static_cast<uint32_t>(DV / 64), 1};
  const uint64_t q_dims[3] = {64, static_cast<uint64_t>(a.B * a.Hq * a.S_q), static_cast<uint64_t>(DK / 64)};
  const uint64_t q_strides[2] = {static_cast<uint64_t>(DK) * 2, 128};
  const uint32_t q_box[3] = {64, kRows, static_cast<uint32_t>(DK / 64)};
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 4, k_dims, k_strides, k_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 4, v_dims, v_strides, v_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&qmap, a.q, 3, q_dims, q_strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B))
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
  prm.GR = static_cast<int>(gr);
  prm.n_rg = static_cast<int>(n_rg);
  prm.R = static_cast<int>(std::min<int64_t>(gr, kRows));
  prm.D = DV;
  prm.max_seq = static_cast<int>(a.max_seq);
  prm.max_tiles = static_cast<int>(max_tiles);
  prm.G = G;
  prm.tb = shape.tb;
  prm.PS = static_cast<int>(part_floats(prm.R, DV));
  prm.plan = needs_plan(a);
  prm.count = reinterpret_cast<int32_t*>(wsb + ws.count);
  prm.tiles = reinterpret_cast<uint16_t*>(wsb + ws.tiles);
  prm.info = reinterpret_cast<int4*>(wsb + ws.info);
  prm.part = reinterpret_cast<float*>(wsb + ws.part);
  prm.status = a.status;
  prm.polls = wait_limit(a.wait_limit_plus1, kWaitPolls);
  prm.kc_w = static_cast<__nv_bfloat16*>(a.kc_w);
  prm.vc_w = static_cast<__nv_bfloat16*>(a.vc_w);
  prm.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  prm.write_idx = a.write_idx;
  prm.S_new = static_cast<int>(a.S_new);

  cudaError_t e;
  switch (mode_of(a)) {
    case kNone: e = launch_dmc<DK, DV, kNone>(a, prm, kmap, vmap, qmap, tmap, max_tiles, shape.bytes); break;
    case kBias: e = launch_dmc<DK, DV, kBias>(a, prm, kmap, vmap, qmap, tmap, max_tiles, shape.bytes); break;
    case kFused: e = launch_dmc<DK, DV, kFused>(a, prm, kmap, vmap, qmap, tmap, max_tiles, shape.bytes); break;
    default: e = launch_dmc<DK, DV, kFusedExtra>(a, prm, kmap, vmap, qmap, tmap, max_tiles, shape.bytes); break;
  }
  if (e != cudaSuccess) return e;
  *name = prm.k_new ? "attn_decode_streamk_mma_scatter" : "attn_decode_streamk_mma";
  return cudaGetLastError();
}

}  // namespace

// Launchers for the head-size pairs of each translation unit.
cudaError_t launch_attn_decode_mixed(const AttnArgs& a, const char** name);  // Dk != Dv
DecodeShape decode_shape_mixed(int64_t Dk, int64_t Dv, int64_t B, int64_t items_max);

}  // namespace extkv
