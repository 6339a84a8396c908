// attn_prefill.cuh -- prefill attention over the external static cache on the
// 5th-generation tensor cores (tcgen05 MMAs, accumulators in tensor memory,
// operands staged by TMA).
//
// Work unit: one CTA per (batch b, query head h, tile of 128 query rows[,
// 256-column chunk of Y when the value head size is 512][, key split]).
// Scores and outputs are dense contractions ("ONNX Domain Attention (Opset
// 23/24) CUDA Patterns", section 1: S = Q K^T, softmax, O = P V; GQA maps
// query head h to KV head h / (Hq/Hkv)), so both run as tcgen05 MMAs with
// M = 128 query rows, for a query-key head size DK and DV output columns:
//   S_j = Q K_j^T   M=128, N=128 keys, K=DK   (A = Q in tensor or shared memory; B = K tile, K-major)
//   O  += P_j V_j   M=128, N=DV,       K=128  (A = P in tensor memory; B = V tile, MN-major)
// Q sits in tensor memory where there is room for it (with A in shared
// memory the tensor cores re-read Q for every key tile), else in shared
// memory, loaded once.  The value head size may differ from DK
// ("Skill: Attention Optimization", "ORT CUDA Attention Kernel Dispatch":
// head_size != v_head_size); a value head size of 512 is covered by two CTAs
// that share the scores' work and write 256 columns each, because S_0, S_1
// and O must fit the 512 tensor-memory columns.
// The CTA is warp-specialised (192 threads; 320 with the split softmax):
//   warp 0   TMA producer: K_0, K_1, V_0, K_2, V_1, ... through a ring of
//            shared-memory slots (one request per load unit via a permuted
//            4-D view that lands the 128-byte-swizzled per-64-column layout),
//            plus the 128 x 128 bias or extra-term block of each tile.
//   warp 1   MMA issuer (one thread): S_{j+1} while the softmax works on S_j,
//            then O += P_j V_j; completion is signalled through tcgen05.commit
//            on mbarriers.  S is double-buffered in tensor memory.
//   warps 2-5  softmax, one thread per query row (= tensor-memory lane): scale,
//            bias or in-register mask, online softmax on scores in natural
//            units, the running maximum subtracted before the base-2 scaling
//            and exponentiation (an extreme finite bias never overflows into
//            a mask); the output accumulator is rescaled in tensor memory
//            only when a row's maximum grows by more than 8 ln 2 (otherwise
//            the stale maximum keeps every term below 2^8, exact after the
//            final division); P is written as bf16 over the first half of
//            its own S buffer.  They
//            also copy the Q tile into tensor memory at the start.
//            Epilogue: O / l from tensor memory to Y (bf16), zero rows where no
//            key is unmasked.
//   warps 2-9  (head sizes up to 128) the same with two warps per query row,
//            one per 64-key half of each tile; the pair exchanges its half
//            maxima once per tile and its sums at the end.
// Tensor memory: S_0, S_1 (128 columns each), O (DV columns), Q (DK/2
// columns) when held there.
//
// Live key range of a tile: without a bias, [0, nonpad); with the fused
// specification, the union of the rows' allowed intervals (each holds the
// row's own position, so the union over consecutive rows is one interval);
// with a materialised bias or the fused specification's extra term, a plan
// kernel scans the term once per (batch, query tile) -- shared by all heads --
// and records, per 64-key tile, which keys some row may attend.
//
// Masking and zero rows follow section 6 of the ORT page: a key is masked iff
// j >= nonpad[b] or bias <= lowest(T); masked scores become -inf by selection;
// V rows of keys that no row of the CTA attends (known in closed form from the
// live range, or from the plan's column masks) are zeroed in shared memory
// before the PV product, so poisoned (even NaN) cache slots cannot reach the
// output; a row with no unmasked key is written as zeros.
#pragma once

#include <climits>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace extkv {

namespace {

constexpr int kBM = 128;                   // query rows per CTA (M, tensor-memory lanes)
constexpr int kBN = 128;                   // keys per KV tile (N of S = Q K^T)
constexpr int kPlanKeys = 256;             // keys per block of the extra-term plan (8 per lane)
constexpr int kPlanThreads = 256;
constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits
constexpr int kMaxUnits = 8;
constexpr int kMaxSplit = 8;               // key splits of a query tile (small grids)

enum Mode { kNone = 0, kBias = 1, kFused = 2, kFusedExtra = 3 };

// A CTA contracts Q and K over DK (the query-key head size) and produces DV
// output columns (the whole value head size, or one of its 256-column chunks
// when it is larger: tensor memory holds S_0, S_1 and O, 256 + DV columns).
// K/V tiles (128 keys) stream through a ring of load units of at most 32 KB:
// a K tile is DK/128 units split by 128-column slices of the head dim (each
// feeds its share of the K steps of Q K^T) when DK > 128, else one unit; a V
// tile is two units split by key halves (each feeds half of the K steps of
// P V) when DV > 128, else one unit.
template <int DK, int DV, int MODE>
struct Cfg {
  static constexpr bool kTerm = MODE == kBias || MODE == kFusedExtra;  // a 128 x 128 block per tile
  // Softmax warps: with DV <= 128 a tile's tensor work (~1.2 k cycles) is
  // shorter than one thread's softmax of a 128-key row, so two warps share
  // each tensor-memory lane quadrant, one per 64-key half of the tile.
  static constexpr bool kSplit = DV <= 128 && DK <= 128;
  static constexpr int kSoftWarps = kSplit ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kSoftWarps;
  // Q as a shared-memory A operand where tensor memory has no room for it
  static constexpr bool kQSmem = 256 + DV + DK / 2 > 512;
  static constexpr int kKP = DK > 128 ? DK / 128 : 1;  // load units of a K tile
  static constexpr int kVP = DV > 128 ? 2 : 1;         // load units of a V tile
  static constexpr int kKBytes = kBN * DK * 2 / kKP;
  static constexpr int kVBytes = kBN * DV * 2 / kVP;
  static constexpr int kUnitBytes = kKBytes > kVBytes ? kKBytes : kVBytes;
  static constexpr int kKChunks = DK / 64 / kKP;  // 64-column chunks in a K unit
  static constexpr int kVKeys = kBN / kVP;        // keys in a V unit
  static constexpr int kQBytes = kQSmem ? kBM * DK * 2 : 0;
  static constexpr int kTermBytes = kTerm ? kBM * kBN * 2 : 0;
  static constexpr int kTermBufs = kTerm ? (kQSmem ? 1 : 2) : 0;
  static constexpr int kTB = kTermBufs > 0 ? kTermBufs : 1;  // divisor for buffer indexing
  static constexpr int kXchBytes = kSplit ? 2 * 2 * kBM * 4 : 0;  // [tile parity][half][row] floats
  static constexpr int kBudget = 232448 - 1024 - 512 - kXchBytes;  // opt-in maximum, alignment, barriers, exchange
  static constexpr int kFit = (kBudget - kQBytes - kTermBufs * kTermBytes) / kUnitBytes;
  static constexpr int kNU = kFit > kMaxUnits ? kMaxUnits : kFit;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffT = kOffKV + kNU * kUnitBytes;
  static_assert(kNU * kUnitBytes >= 4 * (DV / 64) * 4096, "the epilogue stages 128 rows x DV in the K/V ring");
  static constexpr int kOffBar = kOffT + kTermBufs * kTermBytes;
  static constexpr int kOffXch = kOffBar + 512;
  static constexpr int kSmem = kOffXch + kXchBytes + 1024;
  // tensor memory: S_0, S_1 at columns 0 and 128 (P_j, bf16, over the first 64
  // columns of S_j), O at 256, Q (when held there) after O
  static constexpr uint32_t kOCol = 256;
  static constexpr uint32_t kQCol = kOCol + DV;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, 0, 0);
  static constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, DV, 0, 1);
  static_assert(kNU >= 2, "shared memory holds fewer than two load units");
  static_assert(kOCol + DV + (kQSmem ? 0 : DK / 2) <= kTmemCols, "tensor memory columns");
  static_assert(DV <= 256 && DV % 64 == 0 && DK % 64 == 0 && DK <= 512, "head sizes of one CTA");
};


struct Bars {
  uint64_t q_full;
  uint64_t u_full[kMaxUnits], u_empty[kMaxUnits];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t v_ready[2];  // V_j has landed (MMA thread): dead V rows may be zeroed
  uint64_t xch[4][2];   // split softmax: both warps of lane quadrant q wrote slot [parity]
  uint64_t t_full[2], t_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int range_lo, range_hi;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct PrefillParams {
  __nv_bfloat16* y;
  const __nv_bfloat16* q;
  const int64_t* nonpad;
  const uint64_t* colmask;  // bias / extra-term modes: per (b, query tile, 64-key tile) live columns
  // materialised bias: per (b, query tile, row, 128-key tile) the row's live keys (16 bytes), and per
  // (b, query tile, 128-key tile) whether the bias holds values other than 0 and the sentinel there
  const uint8_t* rowmask;
  const uint8_t* impure;
  int rm_stride, n_kt;
  BiasSpec spec;
  float scale;
  float softcap;     // > 0: scores capped to softcap * tanh(score / softcap) before the bias
  int B, Hq, Hkv, S_q, max_seq, n_pt, n_tiles;  // n_tiles: 64-key words per colmask row
  int Dv;    // value head size (columns of Y)
  int n_vc;  // column chunks of Y per (b, h, query tile): Dv / DV
  int32_t* status;
  // Key splits of a query tile (small grids): CTA split s takes its share of
  // the tile's KV tiles and writes an fp32 partial row per query row,
  // part[((b*Hq + h)*n_split + s)*S_q + i][part_stride(Dv)] = O[Dv], max, sum
  // (max in natural units; O and sum relative to it); a merge kernel combines
  // them.  n_split == 1: the output rows are written directly.
  int n_split;
  float* part;
  uint32_t polls;  // limit of the pipeline's barrier waits
  // Packed query rows (all positions of a query fit one tile, S_q <= 128, and
  // a KV head serves several query heads): a tile holds the rows (head, s) of
  // the group's heads one after the other, n_pk tiles per KV head, so each
  // KV tile is read once for the whole group.
  int packed, n_pk;
};

// floats per partial row: O, then max and sum, rounded to 16 bytes
__host__ __device__ constexpr int part_stride(int D) { return D + 4; }

// Bounded wait (at most `limit` polls) that also gives up once another role
// has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 127u) == 127u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Bounded wait polling with test_wait (no suspension): for short hand-offs
// between warps that are usually already complete.
__device__ __forceinline__ bool spin_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ptx::mbar_test_wait(bar, parity)) return true;
    if ((i & 127u) == 127u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Bounded wait for up to three barrier phases at once: the polls are issued
// back to back so their shared-memory round trips overlap (n = 1 .. 3).
__device__ __forceinline__ bool wait3_or_abort(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                               uint32_t p2, int n, volatile int* abort, uint32_t limit) {
  bool d0 = false, d1 = n < 2, d2 = n < 3;
  for (uint32_t i = 0; i < limit; ++i) {
    const bool r0 = d0 || ptx::mbar_try_wait(b0, p0);
    const bool r1 = d1 || ptx::mbar_try_wait(b1, p1);
    const bool r2 = d2 || ptx::mbar_try_wait(b2, p2);
    d0 = r0;
    d1 = r1;
    d2 = r2;
    if (d0 && d1 && d2) return true;
    if ((i & 127u) == 127u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Bits [lo, hi) of a 64-bit word, both ends clamped to [0, 64].
__device__ __forceinline__ uint64_t bit_range(int lo, int hi) {
  lo = lo < 0 ? 0 : (lo > 64 ? 64 : lo);
  hi = hi < 0 ? 0 : (hi > 64 ? 64 : hi);
  if (lo >= hi) return 0;
  const uint64_t upto_hi = hi >= 64 ? ~0ull : ((1ull << hi) - 1);
  const uint64_t below_lo = (1ull << lo) - 1;  // lo < 64 here
  return upto_hi & ~below_lo;
}

// Tile-level load order K_0, K_1, V_0, K_2, V_1, ..., K_{T-1}, V_{T-2}, V_{T-1}:
// the position of K_j and V_j in it.
__device__ __forceinline__ int k_index(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_index(int j, int T) { return j == T - 1 ? 2 * T - 1 : 2 * j + 2; }

// First load unit of K_j and of V_j in the order K_0, K_1, V_0, K_2, V_1, ...
// (K tiles of KP units, V tiles of VP units).
template <int KP, int VP>
__device__ __forceinline__ int k_unit(int j) {
  return j * KP + (k_index(j) - j) * VP;
}
template <int KP, int VP>
__device__ __forceinline__ int v_unit(int j, int T) {
  return (v_index(j, T) - j) * KP + j * VP;
}

// ---- plan: which keys some row of a query tile may attend -------------------------

// Bit k of word (b, pt, t) of the table says whether some query row of tile
// pt of batch b may attend key 64 t + k: key < nonpad[b] and term > lowest,
// and, for the fused specification's extra term, key inside the row's
// allowed intervals.  Keys outside the allowed intervals are never read.
// One block per (256-key chunk, query tile, batch), shared by all heads; each
// lane owns 8 keys and keeps the loads of all its rows in flight at once.
template <bool FUSED>
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const __nv_bfloat16* __restrict__ term,
                                                                   const int64_t* __restrict__ nonpad,
                                                                   const BiasSpec spec,
                                                                   uint64_t* __restrict__ colmask, int S_q,
                                                                   int max_seq, int n_pt, int n_words) {
  constexpr int kRowsPerWarp = kBM / (kPlanThreads / 32);
  const int ch = blockIdx.x, pt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ uint32_t words[kPlanKeys / 32];
  __shared__ int4 win_s[FUSED ? kBM : 1];  // per row: band [x, y) and span [z, w), clipped to [-1, max_seq + 1]
  if (tid < kPlanKeys / 32) words[tid] = 0;
  ptx::grid_launch_dependents();  // the attention kernel may start its prologue
  const int64_t np64 = nonpad[b];
  const bool bad = bad_nonpad(np64, max_seq);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int64_t qs = bad ? 0 : query_start(spec.q_start, b, np64, S_q);
  const int q0 = pt * kBM;
  const int rows = min(kBM, S_q - q0);
  if (FUSED) {
    // each row's allowed intervals once per block (one thread per row)
    auto clip = [&](int64_t v) { return static_cast<int>(v < -1 ? -1 : (v > max_seq + 1 ? max_seq + 1 : v)); };
    for (int r = tid; r < rows; r += kPlanThreads) {
      const RowWindow w = row_window(spec, b, qs + q0 + r, np);
      int4 v = make_int4(clip(w.band_lo), clip(w.band_hi), clip(w.span_lo), clip(w.span_hi));
      if (w.band_lo >= w.band_hi) v.x = v.y = 0;
      if (w.span_lo >= w.span_hi) v.z = v.w = 0;
      win_s[r] = v;
    }
  }
  __syncthreads();
  const float lowest = Elem<__nv_bfloat16>::lowest();
  const int kl = ch * kPlanKeys + 8 * lane;  // this lane's 8 keys
  uint32_t acc = 0;
  if (kl < np) {
    const uint32_t valid = np - kl >= 8 ? 0xFFu : ((1u << (np - kl)) - 1);
    const uint16_t* base = reinterpret_cast<const uint16_t*>(term) +
                           (static_cast<int64_t>(b) * S_q + q0) * max_seq + kl;
    uint32_t want[kRowsPerWarp];
    uint4 v[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int r = warp + (kPlanThreads / 32) * i;
      uint32_t m = r < rows ? valid : 0u;
      if (FUSED && m) {
        // this lane's 8 keys [kl, kl + 8) against the row's two intervals
        const int4 wv = win_s[r];
        const int bl = min(max(wv.x - kl, 0), 8), bh = min(max(wv.y - kl, 0), 8);
        const int sl = min(max(wv.z - kl, 0), 8), sh = min(max(wv.w - kl, 0), 8);
        const uint32_t a = (bl < bh ? ((1u << bh) - 1) & ~((1u << bl) - 1) : 0u) |
                           (sl < sh ? ((1u << sh) - 1) & ~((1u << sl) - 1) : 0u);
        m &= a;
      }
      want[i] = m;
      // in bounds whenever some key of the vector is below nonpad (max_seq % 8 == 0)
      v[i] = make_uint4(0, 0, 0, 0);
      if (m) {
        const uint16_t* src = base + static_cast<int64_t>(r) * max_seq;
        asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w)
                     : "l"(src));
      }
    }
    asm volatile("" ::: "memory");  // every row's load is issued before any is consumed
    const __nv_bfloat162 lowest2 = __bfloat162bfloat162(__float2bfloat16_rn(lowest));
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t m = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // 0xFFFF in each half whose value is above the sentinel (false for NaN)
        const uint32_t live = __hgt2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w4[q]), lowest2);
        m |= ((live & 1u) | ((live >> 15) & 2u)) << (2 * q);
      }
      acc |= m & want[i];
    }
  }
  // lanes 4i .. 4i+3 share word i (32 keys)
  if (acc) atomicOr(&words[lane >> 2], acc << (8 * (lane & 3)));
  __syncthreads();
  if (tid < kPlanKeys / 64) {
    const int t = ch * (kPlanKeys / 64) + tid;
    if (t < n_words)
      colmask[(static_cast<int64_t>(b) * n_pt + pt) * n_words + t] =
          static_cast<uint64_t>(words[2 * tid]) | (static_cast<uint64_t>(words[2 * tid + 1]) << 32);
  }
}

// The same table for a materialised bias: each block stages the 128 x 128
// bias block of one key tile in shared memory (32 KB, so seven blocks fit an
// SM and a whole query tile's row of blocks is in flight at once) with one
// tiled TMA copy (one request: with a copy per row, the 128 requests of each
// of an SM's seven blocks queued behind one another), then thread (g, k) ORs
// rows g, g + 16, ... of keys 8k .. 8k + 7.  It also writes, per query row and
// 128-key tile, the bits of the keys the row may attend (rowmask: 16 bytes
// per row and tile, rm_stride bytes per row), and per (query tile, 128-key
// tile) whether the bias holds a value other than 0 and the sentinel inside
// the live keys (impure).  Where it does not, the attention kernel needs only
// the bits: adding a bias of 0 changes no score.
constexpr int kPlanSmem = kBM * kBN * 2 + 64;

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_bias_kernel(const __grid_constant__ CUtensorMap bmap,
                                                                        const int64_t* __restrict__ nonpad,
                                                                        uint64_t* __restrict__ colmask, int S_q,
                                                                        int max_seq, int n_pt, int n_words,
                                                                        uint8_t* __restrict__ rowmask, int rm_stride,
                                                                        uint8_t* __restrict__ impure, int n_kt,
                                                                        int32_t* status) {
  constexpr int kGroups = kPlanThreads / (kBN / 8);  // row groups (16): thread = (group, 8-key column)
  extern __shared__ __align__(128) uint8_t plan_smem[];
  uint16_t* rows_s = reinterpret_cast<uint16_t*>(plan_smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(plan_smem + kBM * kBN * 2);
  __shared__ uint32_t words[kBN / 32];
  __shared__ int impure_s;
  const int kt = blockIdx.x, pt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, kc = tid % (kBN / 8), grp = tid / (kBN / 8);
  if (tid == 0) ptx::prefetch_tensormap(&bmap);
  ptx::grid_dependency_wait();    // the bias and nonpad as the preceding kernels left them
  ptx::grid_launch_dependents();  // the attention kernel may start its prologue
  const int64_t np64 = nonpad[b];
  const int np = bad_nonpad(np64, max_seq) ? 0 : static_cast<int>(np64);
  const int k_begin = kt * kBN;
  const int keys = min(kBN, np - k_begin);  // <= 0: nothing live in this tile
  const int q0 = pt * kBM;
  const int rows = min(kBM, S_q - q0);
  if (tid < kBN / 32) words[tid] = 0;
  if (tid == 0) {
    impure_s = 0;
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int kl = 8 * kc;  // this thread's 8 keys of the tile
  uint8_t* rm = rowmask + (static_cast<int64_t>(b) * n_pt + pt) * kBM * rm_stride + kt * 16 + kc;
  uint32_t mrow[kBM / kGroups / 4] = {0, 0};  // this thread's byte of its 8 rows
  if (keys > 0) {
    // the (rows x 128 keys) block as one box of the (B*S_q, max_seq) view:
    // rows past S_q or keys past max_seq arrive as zeros and are not read
    if (tid == 0) {
      ptx::mbar_arrive_expect_tx(bar, kBM * kBN * 2);
      ptx::tma_load_2d(rows_s, &bmap, bar, k_begin, b * S_q + q0);
    }
    const bool ok = ptx::mbar_wait_bounded(bar, 0, kWaitPolls);
    if (!ok && tid == 0) report(status, EXTKV_DEV_TIMEOUT);
    const uint32_t valid = keys - kl >= 8 ? 0xFFu : (keys - kl > 0 ? ((1u << (keys - kl)) - 1) : 0u);
    const float lowest = Elem<__nv_bfloat16>::lowest();
    const __nv_bfloat162 lowest2 = __bfloat162bfloat162(__float2bfloat16_rn(lowest));
    // magnitude bits of the valid keys' values, per 32-bit word of two keys
    uint32_t vmask[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      vmask[q] = (((valid >> (2 * q)) & 1) ? 0x7FFFu : 0u) | (((valid >> (2 * q + 1)) & 1) ? 0x7FFF0000u : 0u);
    uint32_t acc = 0, nz = ok ? 0u : 1u;  // a failed copy leaves the tile to the general path
#pragma unroll
    for (int i = 0; i < kBM / kGroups; ++i) {
      const int r = grp + kGroups * i;
      uint32_t m = 0;
      if (ok && valid && r < rows) {
        const uint4 v = *reinterpret_cast<const uint4*>(rows_s + r * kBN + kl);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // 0xFFFF in each half whose value is above the sentinel (false for NaN)
          const uint32_t live = __hgt2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w4[q]), lowest2);
          m |= ((live & 1u) | ((live >> 15) & 2u)) << (2 * q);
          // a live value other than +-0 needs the bias itself
          nz |= w4[q] & vmask[q] & live;
        }
        m &= valid;
      }
      acc |= m;
      mrow[i >> 2] |= m << (8 * (i & 3));
    }
    if (acc) atomicOr(&words[kc >> 2], acc << (8 * (kc & 3)));
    if (nz) impure_s = 1;
  }
  __syncthreads();
  // the row bits, where the attention kernel reads them: tiles that hold a
  // live key and whose bias is 0 or the sentinel throughout
  if (keys > 0 && !impure_s) {
    const int64_t rm0 = (static_cast<int64_t>(b) * n_pt + pt) * kBM * rm_stride + kt * 16 + kc;
    const int64_t n_rm = static_cast<int64_t>(gridDim.z) * n_pt * kBM * rm_stride;
#pragma unroll
    for (int i = 0; i < kBM / kGroups; ++i)
      if (EXTKV_IN(rm0 + static_cast<int64_t>(grp + kGroups * i) * rm_stride, 1, n_rm, status))
        rm[static_cast<int64_t>(grp + kGroups * i) * rm_stride] = static_cast<uint8_t>(mrow[i >> 2] >> (8 * (i & 3)));
  }
  if (tid == 0 && EXTKV_IN((static_cast<int64_t>(b) * n_pt + pt) * n_kt + kt, 1,
                           static_cast<int64_t>(gridDim.z) * n_pt * n_kt, status))
    impure[(static_cast<int64_t>(b) * n_pt + pt) * n_kt + kt] = static_cast<uint8_t>(impure_s);
  if (tid < kBN / 64) {
    const int t = kt * (kBN / 64) + tid;
    if (t < n_words && EXTKV_IN((static_cast<int64_t>(b) * n_pt + pt) * n_words + t, 1,
                                static_cast<int64_t>(gridDim.z) * n_pt * n_words, status))
      colmask[(static_cast<int64_t>(b) * n_pt + pt) * n_words + t] =
          static_cast<uint64_t>(words[2 * tid]) | (static_cast<uint64_t>(words[2 * tid + 1]) << 32);
  }
}

// ---- softmax helpers ------------------------------------------------------------------

// Scores of 64 keys (half H of a tile) in natural units: t = scale*s
// (+ term), -inf where the key is masked: outside the row's allowed keys
// (PARTIAL halves only; `allowed` bit c) or, with a term, term <= lowest.
template <int H, bool TERM, bool PARTIAL, int N>
__device__ __forceinline__ void half_scores(float (&t)[N], const uint32_t (&sa)[32], const uint32_t (&sb)[32],
                                            const uint32_t (&tw)[32], uint64_t allowed, float scale, float lowest) {
  const uint64_t sc2 = ptx::f2(scale, scale);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const uint32_t s0 = c < 16 ? sa[2 * c] : sb[2 * c - 32];
    const uint32_t s1 = c < 16 ? sa[2 * c + 1] : sb[2 * c - 31];
    const uint64_t sv = ptx::f2(__uint_as_float(s0), __uint_as_float(s1));
    bool ok0 = true, ok1 = true;
    uint64_t v;
    if (TERM) {
      const float b0 = __uint_as_float(tw[c] << 16), b1 = __uint_as_float(tw[c] & 0xFFFF0000u);
      v = ptx::fma2(sv, sc2, ptx::f2(b0, b1));
      ok0 = b0 > lowest;
      ok1 = b1 > lowest;
    } else {
      v = ptx::mul2(sv, sc2);
    }
    if (PARTIAL) {
      ok0 = ok0 && ((allowed >> (2 * c)) & 1);
      ok1 = ok1 && ((allowed >> (2 * c + 1)) & 1);
    }
    t[64 * H + 2 * c] = ok0 ? ptx::f2_lo(v) : -INFINITY;
    t[64 * H + 2 * c + 1] = ok1 ? ptx::f2_hi(v) : -INFINITY;
  }
}

// The same with the softcap of the ORT page's section 4 op order: the scaled
// score x = scale*s becomes cap*tanh(x/cap) before the term is added.
template <int H, bool TERM, bool PARTIAL, int N>
__device__ __forceinline__ void half_scores_capped(float (&t)[N], const uint32_t (&sa)[32], const uint32_t (&sb)[32],
                                                   const uint32_t (&tw)[32], uint64_t allowed, float scale, float cap,
                                                   float lowest) {
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    const uint32_t sv = c < 32 ? sa[c] : sb[c - 32];
    bool ok = true;
    float b = 0.f;
    if (TERM) {
      b = __uint_as_float((c & 1) ? (tw[c >> 1] & 0xFFFF0000u) : (tw[c >> 1] << 16));
      ok = b > lowest;
    }
    if (PARTIAL) ok = ok && ((allowed >> c) & 1);
    const float x = cap * tanhf(__uint_as_float(sv) * scale / cap);
    t[64 * H + c] = ok ? x + b : -INFINITY;
  }
}

// Growth of a row maximum (natural units) beyond which the output
// accumulator is rescaled: 8 ln 2, so that every weight stays below 2^8.
constexpr float kRescaleGrow = 5.5451774f;

// Weights of 32 pairs of scores t[T0 + 2c], t[T0 + 2c + 1] against the row's
// maximum m (natural units): exp(t - m) = 2^(t log2 e - m log2 e), one fused
// multiply-add per pair while m log2 e is finite; past that (|m| above about
// 2.36e38, an extreme finite bias) the difference is formed first.  P goes to
// pk as bf16 pairs, the sum into ls.
template <int T0, int N>
__device__ __forceinline__ void exp_pairs(const float (&t)[N], float m, uint32_t (&pk)[32], uint64_t (&ls)[4]) {
  const float nml = -m * kLog2e;
  const uint64_t l2e = ptx::f2(kLog2e, kLog2e);
  if (fabsf(nml) <= 3.0e38f) {
    const uint64_t nm2 = ptx::f2(nml, nml);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const uint64_t d = ptx::fma2(ptx::f2(t[T0 + 2 * c], t[T0 + 2 * c + 1]), l2e, nm2);
      const float e0 = ptx::ex2(ptx::f2_lo(d)), e1 = ptx::ex2(ptx::f2_hi(d));
      ls[c & 3] = ptx::add2(ls[c & 3], ptx::f2(e0, e1));
      pk[c] = ptx::pack_bf16x2(e0, e1);
    }
  } else {
    const uint64_t nm2 = ptx::f2(-m, -m);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const uint64_t d = ptx::mul2(ptx::add2(ptx::f2(t[T0 + 2 * c], t[T0 + 2 * c + 1]), nm2), l2e);
      const float e0 = ptx::ex2(ptx::f2_lo(d)), e1 = ptx::ex2(ptx::f2_hi(d));
      ls[c & 3] = ptx::add2(ls[c & 3], ptx::f2(e0, e1));
      pk[c] = ptx::pack_bf16x2(e0, e1);
    }
  }
}

__device__ __forceinline__ float tile_max(const float (&t)[kBN]) {
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    // the 16 values t[k + 8m], m = 0 .. 15
    acc[k] = ptx::max3(t[k], t[k + 8], t[k + 16]);
#pragma unroll
    for (int m = 3; m + 1 < kBN / 8; m += 2) acc[k] = ptx::max3(acc[k], t[k + 8 * m], t[k + 8 * m + 8]);
    acc[k] = fmaxf(acc[k], t[k + kBN - 8]);
  }
  static_assert(kBN == 128, "tile_max covers 16 values per accumulator");
  return ptx::max3(ptx::max3(acc[0], acc[1], acc[2]), ptx::max3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

// The maximum of 64 values (one half of a tile).
__device__ __forceinline__ float half_max(const float (&t)[64]) {
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    // the 8 values t[k + 8m], m = 0 .. 7
    acc[k] = ptx::max3(t[k], t[k + 8], t[k + 16]);
    acc[k] = ptx::max3(acc[k], t[k + 24], t[k + 32]);
    acc[k] = ptx::max3(acc[k], t[k + 40], t[k + 48]);
    acc[k] = fmaxf(acc[k], t[k + 56]);
  }
  return ptx::max3(ptx::max3(acc[0], acc[1], acc[2]), ptx::max3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

// The 128-byte row `row` of a 64-key block stored with the 128-byte swizzle.
__device__ __forceinline__ void load_swizzled_row(uint32_t (&w)[32], const uint8_t* blk, int row) {
  const uint8_t* r = blk + row * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 v = *reinterpret_cast<const uint4*>(r + ((u ^ (row & 7)) << 4));
    w[4 * u] = v.x;
    w[4 * u + 1] = v.y;
    w[4 * u + 2] = v.z;
    w[4 * u + 3] = v.w;
  }
}

// ---- the attention kernel ---------------------------------------------------------

// CAP: the scores are softcapped (a separate instantiation, so that the
// uncapped kernel is compiled as if the cap did not exist).
template <int DK, int DV, int MODE, bool CAP>
__global__ void __launch_bounds__(Cfg<DK, DV, MODE>::kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap tmap,
                        const __grid_constant__ CUtensorMap ymap, const PrefillParams p) {
  using C = Cfg<DK, DV, MODE>;
  constexpr int kKP = C::kKP, kVP = C::kVP;
  constexpr bool kFusedMode = MODE == kFused || MODE == kFusedExtra;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sKV = sm + C::kOffKV;
  uint8_t* sT = sm + C::kOffT;
  Bars& bar = *reinterpret_cast<Bars*>(sm + C::kOffBar);
  volatile int* abort = &bar.abort;
  const uint32_t lim = p.polls;  // pipeline waits; the drains keep the full limit

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // blockIdx.x = (hx * n_vc + vc) * n_split + sp: the tile's query head (or, with
  // packed rows, hx = hk * n_pk + packed tile), column chunk of Y, key split
  const int sp = blockIdx.x % p.n_split, hv = blockIdx.x / p.n_split, pt = blockIdx.y, b = blockIdx.z;
  const int hx = hv / p.n_vc, vc = hv % p.n_vc;
  const int g = p.Hq / p.Hkv;
  const int hk = p.packed ? hx / p.n_pk : hx / g;
  const int q0 = pt * kBM;  // position of the tile's first row (0 with packed rows)
  // the tile's rows in the (B * Hq * S_q) query-row space, and how many are real
  const int64_t row_base = p.packed ? (static_cast<int64_t>(b) * p.Hq + hk * g) * p.S_q + (hx % p.n_pk) * kBM
                                    : (static_cast<int64_t>(b) * p.Hq + hx) * p.S_q + q0;
  const int rows_here = p.packed ? min(kBM, g * p.S_q - (hx % p.n_pk) * kBM) : min(kBM, p.S_q - q0);

  if (tid == 0) {
    ptx::mbar_init(&bar.q_full, C::kQSmem ? 1 : C::kSoftWarps * 32);
    for (int s = 0; s < C::kNU; ++s) {
      ptx::mbar_init(&bar.u_full[s], 1);
      ptx::mbar_init(&bar.u_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar.s_full[s], 1);
      ptx::mbar_init(&bar.p_full[s], C::kSoftWarps * 32);
      ptx::mbar_init(&bar.pv_done[s], 1);
      ptx::mbar_init(&bar.v_ready[s], 1);
      for (int q = 0; q < 4; ++q) ptx::mbar_init(&bar.xch[q][s], 64);
      ptx::mbar_init(&bar.t_full[s], 1);
      ptx::mbar_init(&bar.t_empty[s], C::kSoftWarps);
    }
    ptx::mbar_init(&bar.drain, 1);
    bar.range_lo = INT_MAX;
    bar.range_hi = 0;
    bar.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (C::kQSmem) ptx::prefetch_tensormap(&qmap);
    ptx::prefetch_tensormap(&kmap);
    ptx::prefetch_tensormap(&vmap);
    if (C::kTerm) ptx::prefetch_tensormap(&tmap);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bar.tmem_base, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::grid_dependency_wait();  // the preceding kernels' writes (cache, bias, plan) are visible

  // a shared-memory Q tile is needed whenever any key is live: start it first
  if (C::kQSmem && warp == 0 && lane == 0) {
    ptx::mbar_arrive_expect_tx(&bar.q_full, C::kQBytes);
    ptx::tma_load_3d(sQ, &qmap, &bar.q_full, 0, static_cast<int>(row_base), 0);
  }

  const int64_t np64 = p.nonpad[b];
  const bool bad = bad_nonpad(np64, p.max_seq);
  if (bad && tid == 0 && hx == 0 && vc == 0 && pt == 0 && sp == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int64_t qs = bad ? 0 : query_start(p.spec.q_start, b, np64, p.S_q);
  const uint64_t* cmrow = C::kTerm ? p.colmask + (static_cast<int64_t>(b) * p.n_pt + pt) * p.n_tiles : nullptr;
  const int64_t imp0 = MODE == kBias ? (static_cast<int64_t>(b) * p.n_pt + pt) * p.n_kt : 0;

  // softmax threads: this thread's query row (tile row `row`: query head h at
  // position pos; prow: its row in the plan's tables and the term blocks,
  // which are laid out by position) and its allowed key intervals
  const bool is_sm = warp >= 2;
  const int row = 32 * (warp & 3) + lane;
  const bool row_valid = is_sm && row < rows_here;
  const int64_t flat = row_base + row;
  const int h = p.packed ? static_cast<int>(flat / p.S_q) - b * p.Hq : hx;
  const int pos = p.packed ? static_cast<int>(flat % p.S_q) : q0 + row;
  const int prow = p.packed ? pos : row;
  int a1 = 0, b1 = np, a2 = 0, b2 = 0;  // allowed keys: [a1, b1) U [a2, b2)
  if (kFusedMode && is_sm) {
    const RowWindow w = row_window(p.spec, b, qs + pos, np);
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
    const int lim = (np + 63) / 64;
    for (int t = lane; t < lim; t += 32)
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
  const int rlo = bar.range_lo, rhi = bar.range_hi;
  const int t_lo0 = rlo < rhi ? rlo / kBN : 0;
  const int T0 = rlo < rhi ? (rhi + kBN - 1) / kBN - t_lo0 : 0;  // KV tiles of the query tile
  // this split's whole tiles (the rows' masks are per key, so a tile range
  // needs nothing else)
  const int t_lo = t_lo0 + (T0 * sp) / p.n_split;
  const int T = (T0 * (sp + 1)) / p.n_split - (T0 * sp) / p.n_split;
  const uint32_t tbase = bar.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int unit = b * p.Hkv + hk;
      int issued = 0, t_issued = 0;
      bool ok = true;
      // term blocks of the tiles that need one, buffers taken in that order;
      // the flag of the next tile is loaded one call ahead (calls come in tile order)
      bool imp_next = MODE != kBias || (T > 0 && EXTKV_IN(imp0 + t_lo, T, static_cast<int64_t>(p.B) * p.n_pt * p.n_kt, p.status) &&
                                        p.impure[imp0 + t_lo] != 0);
      auto load_term = [&](int j) -> bool {
        const bool imp = imp_next;
        if (MODE == kBias && j + 1 < T)
          imp_next = EXTKV_IN(imp0 + t_lo + j + 1, 1, static_cast<int64_t>(p.B) * p.n_pt * p.n_kt, p.status) && p.impure[imp0 + t_lo + j + 1] != 0;
        if (!imp) return true;  // the row bits suffice
        const int tb = t_issued % C::kTB;
        if (t_issued >= C::kTB && !wait_or_abort(&bar.t_empty[tb], ((t_issued / C::kTB) - 1) & 1, abort, lim))
          return false;
        uint8_t* dst = sT + tb * C::kTermBytes;
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
        const int parts = is_v ? kVP : kKP;
        for (int part = 0; part < parts; ++part) {
          const int u = issued, slot = u % C::kNU;  // units leave in sequence order
          if (u >= C::kNU && !wait_or_abort(&bar.u_empty[slot], ((u / C::kNU) - 1) & 1, abort, lim)) {
            ok = false;
            break;
          }
          uint8_t* dst = sKV + slot * C::kUnitBytes;
          if (is_v) {
            ptx::mbar_arrive_expect_tx(&bar.u_full[slot], C::kVBytes);
            ptx::tma_load_4d(dst, &vmap, &bar.u_full[slot], 0, key0 + part * C::kVKeys, vc * (DV / 64), unit);
          } else {
            ptx::mbar_arrive_expect_tx(&bar.u_full[slot], C::kKBytes);
            ptx::tma_load_4d(dst, &kmap, &bar.u_full[slot], 0, key0, part * C::kKChunks, unit);
          }
          ++issued;
        }
        // the term block of tile j goes out once V_{j-1} (or, for tile 0, K_0) is on its way
        if (ok && C::kTerm) {
          if (idx == 0) ok = load_term(0);
          else if (is_v && j + 1 < T) ok = load_term(j + 1);
        }
      }
      // copies still in flight after an abort land before the CTA leaves
      if (*abort) {
        if (C::kQSmem) ptx::mbar_wait_bounded(&bar.q_full, 0, kWaitPolls);
        for (int u = issued > C::kNU ? issued - C::kNU : 0; u < issued; ++u)
          ptx::mbar_wait_bounded(&bar.u_full[u % C::kNU], (u / C::kNU) & 1, kWaitPolls);
        if (C::kTerm)
          for (int j = t_issued > C::kTB ? t_issued - C::kTB : 0; j < t_issued; ++j)
            ptx::mbar_wait_bounded(&bar.t_full[j % C::kTB], (j / C::kTB) & 1, kWaitPolls);
      } else if (C::kQSmem && T == 0) {
        ptx::mbar_wait_bounded(&bar.q_full, 0, kWaitPolls);  // no consumer: let it land
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      const uint32_t kv_addr = ptx::smem_u32(sKV), q_addr = ptx::smem_u32(sQ);
      // Shared-memory descriptors are built once and advanced by adding the
      // byte offset >> 4 to the start-address field (every operand lies in
      // the first 256 KB of shared memory, so the 14-bit field never carries).
      const uint64_t kdesc0 = ptx::smem_desc_sw128(kv_addr, 16, 1024);
      const uint64_t vdesc0 = ptx::smem_desc_sw128(kv_addr, C::kVKeys * 128, 1024);
      const uint64_t qdesc0 = ptx::smem_desc_sw128(q_addr, 16, 1024);
      // Readiness tests of the next batch: the issuing thread blocks while the
      // tensor pipe's queue is full, so one test placed a few MMAs before the
      // end of the current batch overlaps its shared-memory round trip with
      // queued tensor work; the blocking wait remains for what is not there.
      // A K tile of more than two units is waited for unit by unit (the ring
      // may be shorter than the tile).
      constexpr bool kBatchK = kKP <= 2;
      auto k_ready = [&](int j) -> bool {
        const int u0 = k_unit<kKP, kVP>(j);
        bool r = ptx::mbar_test_wait(&bar.u_full[u0 % C::kNU], (u0 / C::kNU) & 1);
        if (kKP > 1) r = ptx::mbar_test_wait(&bar.u_full[(u0 + 1) % C::kNU], ((u0 + 1) / C::kNU) & 1) && r;
        return r;
      };
      auto pv_ready = [&](int j) -> bool {
        const int u0 = v_unit<kKP, kVP>(j, T);
        bool r = ptx::mbar_test_wait(&bar.p_full[j & 1], (j >> 1) & 1);
        r = ptx::mbar_test_wait(&bar.u_full[u0 % C::kNU], (u0 / C::kNU) & 1) && r;
        if (kVP > 1) r = ptx::mbar_test_wait(&bar.u_full[(u0 + 1) % C::kNU], ((u0 + 1) / C::kNU) & 1) && r;
        return r;
      };
      bool k_known = false, pv_known = false;
      // Q K_j^T into S_{j & 1}; tests P_pj / V_pj on the way when pj >= 0
      auto issue_qk = [&](int j, int pj) -> bool {
        const uint32_t d = tbase + (j & 1) * kBN;
        const int u0 = k_unit<kKP, kVP>(j);
        if (kBatchK) {  // both units of K_j polled together
          const int s0 = u0 % C::kNU, s1 = (u0 + 1) % C::kNU;
          if (!k_known && !wait3_or_abort(&bar.u_full[s0], (u0 / C::kNU) & 1, &bar.u_full[s1],
                                          ((u0 + 1) / C::kNU) & 1, &bar.u_full[s0], 0, kKP, abort, lim))
            return false;
          ptx::tc_fence_after();
        }
        k_known = false;
#pragma unroll
        for (int part = 0; part < kKP; ++part) {
          const int slot = (u0 + part) % C::kNU;
          if (!kBatchK) {
            if (!wait_or_abort(&bar.u_full[slot], ((u0 + part) / C::kNU) & 1, abort, lim)) return false;
            ptx::tc_fence_after();
          }
          const uint64_t kd = kdesc0 + ((slot * C::kUnitBytes) >> 4);
#pragma unroll
          for (int k = 0; k < DK / 16 / kKP; ++k) {
            const int kk = part * (DK / 16 / kKP) + k;  // K step over the head dim
            const uint64_t bd = kd + (((k >> 2) * (kBN * 128) + (k & 3) * 32) >> 4);
            if (C::kQSmem) {
              const uint64_t ad = qdesc0 + (((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
              ptx::umma_bf16(d, ad, bd, C::kIdescQK, kk > 0);
            } else {
              ptx::umma_bf16_ts(d, tbase + C::kQCol + kk * 8, bd, C::kIdescQK, kk > 0);
            }
            if (pj >= 0 && kk == DK / 16 - 4) pv_known = pv_ready(pj);
          }
          ptx::umma_commit(&bar.u_empty[slot]);
        }
        ptx::umma_commit(&bar.s_full[j & 1]);
        return true;
      };
      bool ok = wait_or_abort(&bar.q_full, 0, abort, lim);
      if (ok) {
        ptx::tc_fence_after();
        ok = issue_qk(0, -1);
      }
      for (int j = 0; j < T && ok; ++j) {
        pv_known = false;
        if (j + 1 < T && !(ok = issue_qk(j + 1, j))) break;
        // V_j landed (both units polled together), announced to the softmax
        // warps, which zero its dead rows before they release P_j; then P_j
        const int u0 = v_unit<kKP, kVP>(j, T), s0 = u0 % C::kNU, s1 = (u0 + 1) % C::kNU;
        if (!pv_known && !(ok = wait3_or_abort(&bar.u_full[s0], (u0 / C::kNU) & 1, &bar.u_full[s1],
                                               ((u0 + 1) / C::kNU) & 1, &bar.u_full[s0], 0, kVP, abort, lim)))
          break;
        ptx::mbar_arrive(&bar.v_ready[j & 1]);
        if (!pv_known && !(ok = wait_or_abort(&bar.p_full[j & 1], (j >> 1) & 1, abort, lim))) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int part = 0; part < kVP; ++part) {
          const int slot = (u0 + part) % C::kNU;
          const uint64_t vd = vdesc0 + ((slot * C::kUnitBytes) >> 4);
#pragma unroll
          for (int k = 0; k < kBN / 16 / kVP; ++k) {
            const int ks = part * (kBN / 16 / kVP) + k;  // K step over the keys
            ptx::umma_bf16_ts(tbase + C::kOCol, tbase + (j & 1) * kBN + ks * 8, vd + ((k * 2048) >> 4),
                              C::kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
            if (kBatchK && j + 2 < T && ks == kBN / 16 - 3) k_known = k_ready(j + 2);
          }
          ptx::umma_commit(&bar.u_empty[slot]);
        }
        ptx::umma_commit(&bar.pv_done[j & 1]);
      }
      // every MMA issued has completed before tensor memory is released
      ptx::umma_commit(&bar.drain);
      if (!ptx::mbar_wait_bounded(&bar.drain, 0, kWaitPolls)) *abort = 1;
    }
  } else {
    // ---------------- softmax and epilogue (one query row per thread) ----------------
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    // split softmax: warps 2-5 score keys 0-63 of each tile, warps 6-9 keys
    // 64-127 of the same rows; each pair meets once per tile for the maximum
    const int hh = C::kSplit ? (warp - 2) >> 2 : 0;
    const int quad = warp & 3;
    float* xch = reinterpret_cast<float*>(sm + C::kOffXch);  // [parity][half][row]
    const float sc = p.scale;
    constexpr bool capped = CAP;
    const float lowest = Elem<__nv_bfloat16>::lowest();
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int t_seen = 0;  // term blocks consumed
    if (!C::kQSmem && T > 0) {
      // this row of Q into tensor memory (rows past the chunk: zeros)
      const uint4* qrow =
          reinterpret_cast<const uint4*>(p.q + (row_base + row) * DK);
#pragma unroll
      for (int c = 0; c < DK / 64; ++c) {
        if (C::kSplit && (c & 1) != hh) continue;  // the pair shares the chunks
        uint32_t r[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = row_valid ? qrow[8 * c + u] : make_uint4(0, 0, 0, 0);
          r[4 * u] = v.x;
          r[4 * u + 1] = v.y;
          r[4 * u + 2] = v.z;
          r[4 * u + 3] = v.w;
        }
        ptx::tmem_st32(tl + C::kQCol + 32 * c, r);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar.q_full);
    }
    // whether the bias of a tile holds only 0 and the sentinel: loaded one tile ahead
    bool pure_next = MODE == kBias && T > 0 && EXTKV_IN(imp0 + t_lo, T, static_cast<int64_t>(p.B) * p.n_pt * p.n_kt, p.status) &&
                     p.impure[imp0 + t_lo] == 0;
    for (int j = 0; j < T; ++j) {
      const int tile = t_lo + j, key0 = tile * kBN;
      const bool pure = pure_next;
      if (MODE == kBias && j + 1 < T)
        pure_next = EXTKV_IN(imp0 + tile + 1, 1, static_cast<int64_t>(p.B) * p.n_pt * p.n_kt, p.status) && p.impure[imp0 + tile + 1] == 0;
      // keys of the tile no row of the CTA attends (their V rows are zeroed)
      uint64_t dead0, dead1;
      if (C::kTerm) {
        dead0 = EXTKV_IN(2 * tile, 1, p.n_tiles, p.status) ? ~cmrow[2 * tile] : ~0ull;
        dead1 = 2 * tile + 1 < p.n_tiles ? ~cmrow[2 * tile + 1] : ~0ull;
      } else {
        dead0 = ~bit_range(rlo - key0, rhi - key0);
        dead1 = ~bit_range(rlo - key0 - 64, rhi - key0 - 64);
      }
      // this row's allowed keys before the term test; a tile whose bias
      // holds only 0 and the sentinel needs the plan's bits of the row alone
      uint64_t al0, al1;
      if (pure) {
        const int64_t at = ((static_cast<int64_t>(b) * p.n_pt + pt) * kBM + prow) * p.rm_stride + tile * 16;
        const bool in = EXTKV_IN(at, 16, static_cast<int64_t>(p.B) * p.n_pt * kBM * p.rm_stride, p.status);
        const uint4 rb = in ? *reinterpret_cast<const uint4*>(p.rowmask + at) : make_uint4(0, 0, 0, 0);
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
      if constexpr (C::kSplit) {
        // this warp's half of the tile: keys 64 hh .. 64 hh + 63
        const uint64_t al = hh ? al1 : al0;
        const bool part = hh ? part1 : part0;
        const bool termed = C::kTerm && !pure;
        float t[64];
        {
          uint32_t sa[32], sb[32], tw[32];
          ptx::tmem_ld32(ts + 64 * hh, sa);
          ptx::tmem_ld32(ts + 64 * hh + 32, sb);
          if (termed) {
            // term blocks arrive in the order of the tiles that need one
            const int tb = t_seen % C::kTB;
            if (!__all_sync(0xffffffffu, wait_or_abort(&bar.t_full[tb], (t_seen / C::kTB) & 1, abort, lim))) {
              ok = false;
              break;
            }
            ++t_seen;
            load_swizzled_row(tw, sT + tb * C::kTermBytes + hh * (C::kTermBytes / 2), prow);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.t_empty[tb]);
          }
          ptx::tmem_wait_ld();
          if constexpr (capped) {
            if (termed) {
              if (part) half_scores_capped<0, true, true>(t, sa, sb, tw, al, p.scale, p.softcap, lowest);
              else half_scores_capped<0, true, false>(t, sa, sb, tw, al, p.scale, p.softcap, lowest);
            } else if (part) {
              half_scores_capped<0, false, true>(t, sa, sb, tw, al, p.scale, p.softcap, lowest);
            } else {
              half_scores_capped<0, false, false>(t, sa, sb, tw, al, p.scale, p.softcap, lowest);
            }
          } else if (termed) {
            if (part) half_scores<0, true, true>(t, sa, sb, tw, al, sc, lowest);
            else half_scores<0, true, false>(t, sa, sb, tw, al, sc, lowest);
          } else if (part) {
            half_scores<0, false, true>(t, sa, sb, tw, al, sc, lowest);
          } else {
            half_scores<0, false, false>(t, sa, sb, tw, al, sc, lowest);
          }
        }
        // the tile's maximum: both halves' maxima through shared memory, the
        // pair's 64 threads meeting on the quadrant's barrier of this parity.
        // The meeting also orders the pair's tensor-memory accesses: P of keys
        // 64-127 goes over S columns 32-63, which the other warp has read by
        // the time it arrives.
        float* xm = xch + (j & 1) * 2 * kBM;
        xm[hh * kBM + row] = half_max(t);
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bar.xch[quad][j & 1]);
        if (!__all_sync(0xffffffffu, spin_or_abort(&bar.xch[quad][j & 1], (j >> 1) & 1, abort, lim))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const float mt = fmaxf(xm[row], xm[kBM + row]);  // the same in both warps
        const float m_new = fmaxf(m_run, mt);
        const bool grow = m_new > m_run + kRescaleGrow;
        const bool rescale_o = grow && m_run != -INFINITY;
        const float factor = rescale_o ? ptx::ex2((m_run - m_new) * kLog2e) : 1.f;
        if (__any_sync(0xffffffffu, rescale_o)) {
          // this warp's half of the output columns, once P_{j-1} V_{j-1} completed
          if (!__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, lim))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = hh * (DV / 64); c < (hh + 1) * (DV / 64); ++c) {
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
        uint32_t pk[32];
        exp_pairs<0>(t, m_use, pk, ls);
        ptx::tmem_st32(ts + 32 * hh, pk);  // this half's P over S_j's first half
        const uint64_t lsum = ptx::add2(ptx::add2(ls[0], ls[1]), ptx::add2(ls[2], ls[3]));
        l_run += ptx::f2_lo(lsum) + ptx::f2_hi(lsum);  // this half's share of the row sum
      } else {
        float t[kBN];
        if (pure) {
          // bits only: the fused path's scores (a bias of 0 adds nothing)
          uint32_t sa[32], sb[32], tw[32];
          ptx::tmem_ld32(ts, sa);
          ptx::tmem_ld32(ts + 32, sb);
          ptx::tmem_wait_ld();
          if constexpr (capped) {
            if (part0) half_scores_capped<0, false, true>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
            else half_scores_capped<0, false, false>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
          } else if (part0) {
            half_scores<0, false, true>(t, sa, sb, tw, al0, sc, lowest);
          } else {
            half_scores<0, false, false>(t, sa, sb, tw, al0, sc, lowest);
          }
          ptx::tmem_ld32(ts + 64, sa);
          ptx::tmem_ld32(ts + 96, sb);
          ptx::tmem_wait_ld();
          if constexpr (capped) {
            if (part1) half_scores_capped<1, false, true>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
            else half_scores_capped<1, false, false>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
          } else if (part1) {
            half_scores<1, false, true>(t, sa, sb, tw, al1, sc, lowest);
          } else {
            half_scores<1, false, false>(t, sa, sb, tw, al1, sc, lowest);
          }
        } else {
          // term blocks arrive in the order of the tiles that need one
          const int tb = t_seen % C::kTB;
          const uint8_t* tblk = sT + tb * C::kTermBytes;
          if (C::kTerm &&
              !__all_sync(0xffffffffu, wait_or_abort(&bar.t_full[tb], (t_seen / C::kTB) & 1, abort, lim))) {
            ok = false;
            break;
          }
          if (C::kTerm) ++t_seen;
          uint32_t sa[32], sb[32], tw[32];
          ptx::tmem_ld32(ts, sa);
          ptx::tmem_ld32(ts + 32, sb);
          if (C::kTerm) load_swizzled_row(tw, tblk, prow);
          ptx::tmem_wait_ld();
          if constexpr (capped) {
            if (part0)
              half_scores_capped<0, C::kTerm, true>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
            else
              half_scores_capped<0, C::kTerm, false>(t, sa, sb, tw, al0, p.scale, p.softcap, lowest);
          } else if (part0) {
            half_scores<0, C::kTerm, true>(t, sa, sb, tw, al0, sc, lowest);
          } else {
            half_scores<0, C::kTerm, false>(t, sa, sb, tw, al0, sc, lowest);
          }
          ptx::tmem_ld32(ts + 64, sa);
          ptx::tmem_ld32(ts + 96, sb);
          if (C::kTerm) {
            load_swizzled_row(tw, tblk + C::kTermBytes / 2, prow);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.t_empty[tb]);
          }
          ptx::tmem_wait_ld();
          if constexpr (capped) {
            if (part1)
              half_scores_capped<1, C::kTerm, true>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
            else
              half_scores_capped<1, C::kTerm, false>(t, sa, sb, tw, al1, p.scale, p.softcap, lowest);
          } else if (part1) {
            half_scores<1, C::kTerm, true>(t, sa, sb, tw, al1, sc, lowest);
          } else {
            half_scores<1, C::kTerm, false>(t, sa, sb, tw, al1, sc, lowest);
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
        // P_j over the first half of S_j: QK_{j+2}, the next writer of this
        // buffer, is issued after P_j V_j and the tensor pipe runs in order
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
      }
      if (dead0 | dead1) {
        // zero the V rows of dead keys once V_j has landed (the MMA thread,
        // which consumes the units in order, says so: a parity wait on the
        // units' own barriers could match a slot's previous phase)
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.v_ready[j & 1], (j >> 1) & 1, abort, lim))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int part = 0; part < kVP; ++part) {
          const int slot = (v_unit<kKP, kVP>(j, T) + part) % C::kNU;
          uint8_t* vt = sKV + slot * C::kUnitBytes;
          constexpr int kLines = C::kVKeys * (DV / 64) * 8;  // 16-byte pieces of the unit
          for (int w = tid - 64; w < kLines; w += 32 * C::kSoftWarps) {
            const int kl = w / ((DV / 64) * 8), rem = w % ((DV / 64) * 8);
            const int key = part * C::kVKeys + kl;
            const uint64_t dm = key < 64 ? dead0 : dead1;
            if ((dm >> (key & 63)) & 1)
              *reinterpret_cast<uint4*>(vt + (rem >> 3) * (C::kVKeys * 128) + kl * 128 + (rem & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
          }
        }
        ptx::fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar.p_full[j & 1]);
    }
    // epilogue: O / l, zero rows without an unmasked key
    if (ok && T > 0 &&
        !__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort, lim)))
      ok = false;
    ptx::tc_fence_after();
    if constexpr (C::kSplit) {
      // the row's sum: both halves' shares, added in the same order in both warps
      float* xl = xch + (T & 1) * 2 * kBM;
      xl[hh * kBM + row] = l_run;
      ptx::mbar_arrive(&bar.xch[quad][T & 1]);
      if (!__all_sync(0xffffffffu, spin_or_abort(&bar.xch[quad][T & 1], (T >> 1) & 1, abort, lim))) ok = false;
      l_run = xl[row] + xl[kBM + row];
    }
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    // output columns of this warp: all of them, or its half with the split softmax
    constexpr int kNB = DV / 64;  // 64-column blocks
    const int c32_lo = C::kSplit ? hh * (DV / 64) : 0, c32_hi = C::kSplit ? (hh + 1) * (DV / 64) : DV / 32;
    const int cb_lo = C::kSplit ? (kNB >= 2 ? hh * (kNB / 2) : (hh ? kNB : 0)) : 0;
    const int cb_hi = C::kSplit ? (kNB >= 2 ? (hh + 1) * (kNB / 2) : kNB) : kNB;
    // The warp's 32 rows go through shared memory (the K/V ring is idle now:
    // every MMA that read it has completed) in 32 x 64-column blocks with the
    // 128-byte swizzle, and leave as one TMA store per block; rows beyond S_q
    // fall outside the (D, S_q, B*Hq) view and are not written.
    if (p.n_split > 1) {
      // a partial row of this split: unnormalised O (this CTA's DV columns),
      // the running max and sum (the same in every column chunk)
      float* prow_out = p.part + ((static_cast<int64_t>(b * p.Hq + h) * p.n_split + sp) * p.S_q + pos) *
                                     part_stride(p.Dv);
      const bool live = ok && T > 0;
      // (only rows that are written are tested)
      const bool part_in =
          !row_valid ||
          EXTKV_IN(((static_cast<int64_t>(b * p.Hq + h) * p.n_split + sp) * p.S_q + pos) * part_stride(p.Dv),
                   part_stride(p.Dv), static_cast<int64_t>(p.B) * p.Hq * p.n_split * p.S_q * part_stride(p.Dv),
                   p.status);
#pragma unroll 1
      for (int c = c32_lo; c < c32_hi; ++c) {
        uint32_t o[32];
        if (live) {
          ptx::tmem_ld32(tl + C::kOCol + 32 * c, o);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0;
        }
        if (row_valid && part_in) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(prow_out + vc * DV + 32 * c + 4 * q) =
                make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]), __uint_as_float(o[4 * q + 2]),
                            __uint_as_float(o[4 * q + 3]));
        }
      }
      if (row_valid && part_in && vc == 0 && hh == 0) {
        prow_out[p.Dv] = live ? m_run : -INFINITY;
        prow_out[p.Dv + 1] = live ? l_run : 0.f;
      }
    } else if (p.packed) {
      // packed rows: a warp's 32 rows may belong to several query heads, so
      // each thread writes its own row (rows past the group's are not written)
      __nv_bfloat16* yrow = p.y + (row_base + row) * p.Dv + vc * DV;
      const bool y_in = !(ok && row_valid) ||
                        EXTKV_IN((row_base + row) * p.Dv + vc * DV, DV,
                                 static_cast<int64_t>(p.B) * p.Hq * p.S_q * p.Dv, p.status);
#pragma unroll 1
      for (int cb = cb_lo; cb < cb_hi; ++cb) {
        uint32_t o[64];
        if (ok && T > 0) {
          ptx::tmem_ld32(tl + C::kOCol + 64 * cb, *reinterpret_cast<uint32_t(*)[32]>(o));
          ptx::tmem_ld32(tl + C::kOCol + 64 * cb + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) o[e] = 0;
        }
        if (ok && row_valid && y_in) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv,
                                      __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
            *reinterpret_cast<uint4*>(yrow + 64 * cb + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    } else {
      uint8_t* stage = sKV + quad * kNB * 4096;
#pragma unroll 1
      for (int cb = cb_lo; cb < cb_hi; ++cb) {
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
        for (int cb = cb_lo; cb < cb_hi; ++cb)
          ptx::tma_store_3d(&ymap, stage + cb * 4096, vc * DV + cb * 64, q0 + 32 * (warp & 3), b * p.Hq + h);
        ptx::bulk_commit_group();
        ptx::bulk_wait_read_all();  // shared memory stays valid until the stores have read it
      }
      __syncwarp();
    }
  }
  ptx::grid_launch_dependents();
  if (tid == 0 && *abort) report(p.status, EXTKV_DEV_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tbase, C::kTmemCols);
}

// ---- merge of the key splits ----------------------------------------------------------

// One warp per query row: weights exp(max_s - M) of the splits (lane s holds
// split s; n_split <= kMaxSplit), then the row's columns four per lane, summed in
// split order (the result does not depend on timing).  A row whose splits
// saw no unmasked key is an exact zero row.
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillParams p, int D) {
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int ns = p.n_split, ps = part_stride(D);
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.S_q;
  const int64_t split_stride = static_cast<int64_t>(p.S_q) * ps;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); r < rows;
       r += static_cast<int64_t>(gridDim.x) * 8) {
    const int64_t bh = r / p.S_q, i = r % p.S_q;
    const float* base = p.part + (bh * ns * p.S_q + i) * ps;
    float m = -INFINITY, l = 0.f;
    if (lane < ns) {
      m = __ldcg(base + lane * split_stride + D);
      l = __ldcg(base + lane * split_stride + D + 1);
    }
    float M = m;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float ref = M == -INFINITY ? 0.f : M;
    const float w = (lane < ns && m != -INFINITY) ? ptx::ex2((m - ref) * kLog2e) : 0.f;
    float L = w * l;
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float wsv[kMaxSplit];
#pragma unroll
    for (int sg = 0; sg < kMaxSplit; ++sg) wsv[sg] = __shfl_sync(0xffffffffu, w, sg);
    for (int d = 4 * lane; d < D; d += 128) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sg = 0; sg < kMaxSplit; ++sg) {
        const float ws = wsv[sg];
        if (sg >= ns || ws == 0.f) continue;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(base + sg * split_stride + d));
        a.x = fmaf(v.x, ws, a.x);
        a.y = fmaf(v.y, ws, a.y);
        a.z = fmaf(v.z, ws, a.z);
        a.w = fmaf(v.w, ws, a.w);
      }
      uint2 pk;
      pk.x = ptx::pack_bf16x2(a.x * inv, a.y * inv);
      pk.y = ptx::pack_bf16x2(a.z * inv, a.w * inv);
      if (EXTKV_IN(r * D + d, 4, rows * D, p.status)) *reinterpret_cast<uint2*>(p.y + r * D + d) = pk;
    }
  }
}

// ---- host side ----------------------------------------------------------------------

int n_query_tiles(int64_t S_q) { return static_cast<int>((S_q + kBM - 1) / kBM); }
int n_plan_chunks(int64_t max_seq) { return static_cast<int>((max_seq + kPlanKeys - 1) / kPlanKeys); }
// the plan's column-mask table: one 64-bit word per 64 keys
int n_mask_words(int64_t max_seq) { return static_cast<int>((max_seq + 63) / 64); }

// Key splits: a grid of fewer CTAs than half the SMs has its tiles' key
// ranges split so that about one CTA per SM works.
int splits_for(int64_t ctas) {
  const int sms = num_sms();
  if (ctas <= 0 || ctas * 2 > sms) return 1;
  return static_cast<int>(std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, sms / ctas)));
}
int prefill_splits(int64_t B, int64_t Hq, int64_t S_q) { return splits_for(B * Hq * n_query_tiles(S_q)); }

// The tiles per KV head with packed rows, and whether a call packs them: all
// positions fit one tile and packing takes fewer tiles than one per query
// head (otherwise the tiles are the same and the unpacked epilogue's TMA
// stores are kept).
int packed_tiles(int64_t Hq, int64_t Hkv, int64_t S_q) {
  return static_cast<int>((Hq / Hkv * S_q + kBM - 1) / kBM);
}
bool packs_rows(int64_t Hq, int64_t Hkv, int64_t S_q) {
  return S_q <= kBM && packed_tiles(Hq, Hkv, S_q) < Hq / Hkv;
}

// Key splits of a call with n_vc column chunks of Y, packed or not.
int prefill_call_splits(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t n_vc) {
  if (packs_rows(Hq, Hkv, S_q)) return splits_for(B * Hkv * packed_tiles(Hq, Hkv, S_q) * n_vc);
  return prefill_splits(B, Hq * n_vc, S_q);
}

// bytes of the column-mask table, rounded to 256
size_t colmask_bytes(int64_t B, int64_t S_q, int64_t max_seq) {
  const size_t n = static_cast<size_t>(B) * n_query_tiles(S_q) * n_mask_words(max_seq) * sizeof(uint64_t);
  return (n + 255) & ~size_t(255);
}

// 128-key tiles of the cache, and the row bits of a materialised bias: 16
// bytes per (b, query tile, row, 128-key tile); then one byte per (b, query
// tile, 128-key tile) saying whether the tile needs the bias values
int n_key_tiles(int64_t max_seq) { return static_cast<int>((max_seq + kBN - 1) / kBN); }
size_t rowmask_bytes(int64_t B, int64_t S_q, int64_t max_seq) {
  return static_cast<size_t>(B) * n_query_tiles(S_q) * kBM * n_key_tiles(max_seq) * 16;
}
size_t impure_bytes(int64_t B, int64_t S_q, int64_t max_seq) {
  return (static_cast<size_t>(B) * n_query_tiles(S_q) * n_key_tiles(max_seq) + 255) & ~size_t(255);
}
// the tables of a bias or extra term (the partials of key splits follow them)
size_t term_tables_bytes(int64_t B, int64_t S_q, int64_t max_seq) {
  return colmask_bytes(B, S_q, max_seq) + rowmask_bytes(B, S_q, max_seq) + impure_bytes(B, S_q, max_seq);
}

// Columns of Y one CTA produces: the whole value head size up to 256, else
// 256-column chunks (one CTA each).
int64_t v_chunk(int64_t Dv) { return Dv > 256 ? 256 : Dv; }

// The kernel parameters of a prefill call with `dv_chunk` output columns per
// CTA, and the plan kernel a materialised bias or an extra term needs
// (launched here, on the call's stream, ahead of the attention kernel).
cudaError_t prefill_setup(const AttnArgs& a, int mode, int dv_chunk, PrefillParams* out) {
  PrefillParams& prm = *out;
  const int64_t Dvf = a.Dv;
  const void* term = mode == kBias ? a.bias : (mode == kFusedExtra ? a.extra : nullptr);
  prm.y = static_cast<__nv_bfloat16*>(a.y);
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.nonpad = a.nonpad;
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);
  const size_t off_rowmask = colmask_bytes(a.B, a.S_q, a.max_seq);
  const size_t off_impure = off_rowmask + rowmask_bytes(a.B, a.S_q, a.max_seq);
  prm.colmask = reinterpret_cast<const uint64_t*>(wsb);
  prm.rowmask = wsb + off_rowmask;
  prm.impure = wsb + off_impure;
  prm.n_kt = n_key_tiles(a.max_seq);
  prm.rm_stride = prm.n_kt * 16;
  prm.spec = BiasSpec{a.causal, a.window, a.span_offsets, a.spans, a.extra, a.q_start};
  prm.scale = a.scale;
  prm.softcap = a.softcap;
  prm.B = static_cast<int>(a.B);
  prm.Hq = static_cast<int>(a.Hq);
  prm.Hkv = static_cast<int>(a.Hkv);
  prm.S_q = static_cast<int>(a.S_q);
  prm.max_seq = static_cast<int>(a.max_seq);
  prm.n_pt = n_query_tiles(a.S_q);
  prm.n_tiles = n_mask_words(a.max_seq);
  prm.Dv = static_cast<int>(Dvf);
  prm.n_vc = static_cast<int>(Dvf / dv_chunk);
  prm.status = a.status;
  prm.packed = packs_rows(a.Hq, a.Hkv, a.S_q) ? 1 : 0;
  prm.n_pk = prm.packed ? packed_tiles(a.Hq, a.Hkv, a.S_q) : 0;
  prm.n_split = prefill_call_splits(a.B, a.Hq, a.Hkv, a.S_q, prm.n_vc);
  prm.polls = wait_limit(a.wait_limit_plus1, kWaitPolls);
  prm.part = reinterpret_cast<float*>(wsb + term_tables_bytes(a.B, a.S_q, a.max_seq));

  if (mode == kBias) {
    if (cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(prefill_plan_bias_kernel), kPlanSmem);
        e != cudaSuccess)
      return e;
    // the bias as a (B*S_q rows, max_seq keys) view, boxes of 128 x 128
    CUtensorMap bmap;
    const uint64_t b_dims[2] = {static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(a.B * a.S_q)};
    const uint64_t b_strides[1] = {static_cast<uint64_t>(a.max_seq) * 2};
    const uint32_t b_box[2] = {kBN, kBM};
    if (!make_tensor_map_bf16(&bmap, term, 2, b_dims, b_strides, b_box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    // a dependent launch: its blocks may be placed before the preceding kernel ends
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(prm.n_kt, prm.n_pt, prm.B);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = kPlanSmem;
    cfg.stream = a.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_plan_bias_kernel, bmap, a.nonpad,
                                       static_cast<uint64_t*>(a.workspace), prm.S_q, prm.max_seq, prm.n_pt,
                                       prm.n_tiles, wsb + off_rowmask, prm.rm_stride, wsb + off_impure,
                                       prm.n_kt, a.status);
    if (e != cudaSuccess) return e;
  } else if (mode == kFusedExtra) {
    prefill_plan_kernel<true><<<dim3(n_plan_chunks(a.max_seq), prm.n_pt, prm.B), kPlanThreads, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(term), a.nonpad, prm.spec, static_cast<uint64_t*>(a.workspace),
        prm.S_q, prm.max_seq, prm.n_pt, prm.n_tiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  return cudaSuccess;
}

template <int DK, int DV, int MODE, bool CAP>
cudaError_t launch_dm(const AttnArgs& a, const char** name) {
  using C = Cfg<DK, DV, MODE>;
  if (cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(attn_prefill_kernel<DK, DV, MODE, CAP>),
                                           C::kSmem);
      e != cudaSuccess)
    return e;
  const int64_t Dvf = a.Dv;  // the whole value head size
  if (Dvf % DV) return cudaErrorInvalidValue;

  // permuted views (64 columns, key, 64-column chunk, batch x KV head): one
  // request lands a whole unit in the 128-byte-swizzled per-chunk layout
  CUtensorMap qmap, kmap, vmap, tmap;
  const uint64_t units = static_cast<uint64_t>(a.B * a.Hkv);
  const uint64_t k_dims[4] = {64, static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(DK / 64), units};
  const uint64_t k_strides[3] = {static_cast<uint64_t>(DK) * 2, 128, static_cast<uint64_t>(a.max_seq) * DK * 2};
  const uint64_t v_dims[4] = {64, static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(Dvf / 64), units};
  const uint64_t v_strides[3] = {static_cast<uint64_t>(Dvf) * 2, 128, static_cast<uint64_t>(a.max_seq) * Dvf * 2};
  const uint32_t k_box[4] = {64, kBN, static_cast<uint32_t>(C::kKChunks), 1};
  const uint32_t v_box[4] = {64, static_cast<uint32_t>(C::kVKeys), static_cast<uint32_t>(DV / 64), 1};
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 4, k_dims, k_strides, k_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 4, v_dims, v_strides, v_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  std::memset(&qmap, 0, sizeof qmap);
  if (C::kQSmem) {
    const uint64_t q_dims[3] = {64, static_cast<uint64_t>(a.B * a.Hq * a.S_q), static_cast<uint64_t>(DK / 64)};
    const uint64_t q_strides[2] = {static_cast<uint64_t>(DK) * 2, 128};
    const uint32_t q_box[3] = {64, kBM, static_cast<uint32_t>(DK / 64)};
    if (!make_tensor_map_bf16(&qmap, a.q, 3, q_dims, q_strides, q_box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // output view (Dv, S_q, B*Hq): the epilogue's 32-row x 64-column stores
  CUtensorMap ymap;
  const uint64_t y_dims[3] = {static_cast<uint64_t>(Dvf), static_cast<uint64_t>(a.S_q),
                              static_cast<uint64_t>(a.B * a.Hq)};
  const uint64_t y_strides[2] = {static_cast<uint64_t>(Dvf) * 2, static_cast<uint64_t>(a.S_q) * Dvf * 2};
  const uint32_t y_box[3] = {64, 32, 1};
  if (!make_tensor_map_bf16(&ymap, a.y, 3, y_dims, y_strides, y_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  std::memset(&tmap, 0, sizeof tmap);
  const void* term = MODE == kBias ? a.bias : (MODE == kFusedExtra ? a.extra : nullptr);
  if (term) {
    const uint64_t t_dims[2] = {static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(a.B * a.S_q)};
    const uint64_t t_strides[1] = {static_cast<uint64_t>(a.max_seq) * 2};
    const uint32_t t_box[2] = {64, kBM};  // two requests per 128-key tile
    if (!make_tensor_map_bf16(&tmap, term, 2, t_dims, t_strides, t_box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }

  PrefillParams prm;
  if (cudaError_t e = prefill_setup(a, MODE, DV, &prm); e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  // blockIdx.x: (query head, or packed tile of a KV head) x column chunk x key split
  cfg.gridDim = dim3((prm.packed ? prm.Hkv * prm.n_pk : prm.Hq) * prm.n_vc * prm.n_split, prm.n_pt, prm.B);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, attn_prefill_kernel<DK, DV, MODE, CAP>, qmap, kmap, vmap, tmap, ymap, prm);
  if (e != cudaSuccess) return e;
  if (prm.n_split > 1) {
    const int64_t rows = static_cast<int64_t>(prm.B) * prm.Hq * prm.S_q;
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>((rows + 7) / 8, int64_t(num_sms()) * 8)));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, prefill_merge_kernel, prm, prm.Dv);
    if (e != cudaSuccess) return e;
  }
  *name = prm.packed ? "attn_prefill_tcgen05_packed" : "attn_prefill_tcgen05";
  // the plan kernel, the attention kernel, the merge of the key splits
  note_launches((C::kTerm ? 2 : 1) + (prm.n_split > 1 ? 1 : 0));
  return cudaGetLastError();
}

template <int DK, int DV, bool CAP>
cudaError_t launch_dc(const AttnArgs& a, const char** name) {
  if (a.bias) return launch_dm<DK, DV, kBias, CAP>(a, name);
  if (a.fused)
    return a.extra ? launch_dm<DK, DV, kFusedExtra, CAP>(a, name) : launch_dm<DK, DV, kFused, CAP>(a, name);
  return launch_dm<DK, DV, kNone, CAP>(a, name);
}

// The tensor-core kernel for query-key head size DK and value chunk DV.
template <int DK, int DV>
cudaError_t launch_kv(const AttnArgs& a, const char** name) {
  return a.softcap > 0.f ? launch_dc<DK, DV, true>(a, name) : launch_dc<DK, DV, false>(a, name);
}

}  // namespace

// Head-size pairs (Dk, Dv) the tensor-core kernel runs; each translation unit
// instantiates a group of them.
inline bool prefill_pair_supported(int64_t Dk, int64_t Dv) {
  if (Dk == Dv) return Dk == 64 || Dk == 128 || Dk == 256 || Dk == 512;
  auto in = [](int64_t d) { return d == 128 || d == 256 || d == 512; };
  return in(Dk) && in(Dv);
}
cudaError_t launch_attn_prefill_equal(const AttnArgs& a, const char** name);  // Dk == Dv <= 256
cudaError_t launch_attn_prefill_dk512(const AttnArgs& a, const char** name);  // Dk == 512
cudaError_t launch_attn_prefill_mixed(const AttnArgs& a, const char** name);  // Dk != Dv, Dk <= 256

}  // namespace extkv
