// attn_prefill.cu -- prefill attention over the external static cache on the
// 5th-generation tensor cores (tcgen05 MMAs, accumulators in tensor memory,
// operands staged by TMA).
//
// Work unit: one CTA per (batch b, query head h, tile of 128 query rows).
// Scores and outputs are dense contractions ("ONNX Domain Attention (Opset
// 23/24) CUDA Patterns", section 1: S = Q K^T, softmax, O = P V; GQA maps
// query head h to KV head h / (Hq/Hkv)), so both run as tcgen05 MMAs with
// M = 128 query rows:
//   S_j = Q K_j^T   M=128, N=64 keys,  K=D     (A = Q in tensor memory; B = K tile, K-major)
//   O  += P_j V_j   M=128, N=D,        K=64    (A = P in tensor memory; B = V tile, MN-major)
// Both A operands live in tensor memory, so the tensor cores read only the
// K/V tiles from shared memory: with A in shared memory, re-reading Q for every
// 64-key tile would take more shared-memory bandwidth than the MMAs' operand
// port and the TMA writes have between them.
// The CTA is warp-specialised (192 threads):
//   warp 0   TMA producer: K_0, K_1, V_0, K_2, V_1, ... through a ring of
//            shared-memory slots (one request per tile via a permuted 4-D view
//            that lands the 128-byte-swizzled per-64-column layout), plus the
//            128 x 64 bias or extra-term block of each tile.
//   warp 1   MMA issuer (one thread): S_{j+1} while the softmax works on S_j,
//            then O += P_j V_j; completion is signalled through tcgen05.commit
//            on mbarriers.  S is double-buffered in tensor memory.
//   warps 2-5  softmax, one thread per query row (= tensor-memory lane): scale,
//            bias or in-register mask, online softmax in base 2 with the
//            running maximum subtracted before exponentiation; the output
//            accumulator is rescaled in tensor memory only when a row's
//            maximum grows by more than 2^8 (otherwise the stale maximum keeps
//            every term below 2^8, exact after the final division); P is
//            written as bf16 over the first half of its own S buffer.  They
//            also copy the Q tile into tensor memory at the start.
//            Epilogue: O / l from tensor memory to Y (bf16), zero rows where no
//            key is unmasked.
// Tensor memory: S_0, S_1 (64 columns each), Q (D/2 columns), O (D columns).
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
constexpr int kBN = 64;                    // keys per KV tile
constexpr int kThreads = 192;              // producer, MMA, 4 softmax warps
constexpr int kPlanKeys = 512;             // keys per plan block
constexpr int kPlanThreads = 256;
constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits
constexpr int kMaxSlots = 8;

enum Mode { kNone = 0, kBias = 1, kFused = 2, kFusedExtra = 3 };

template <int D, int MODE>
struct Cfg {
  static constexpr bool kTerm = MODE == kBias || MODE == kFusedExtra;  // a 128 x 64 block per tile
  static constexpr int kSlotBytes = kBN * D * 2;
  static constexpr int kTermBytes = kTerm ? kBM * kBN * 2 : 0;
  static constexpr int kBudget = 232448 - 1024 - 512;  // opt-in maximum, alignment, barriers
  static constexpr int kFit = (kBudget - 2 * kTermBytes) / kSlotBytes;
  static constexpr int kNS = kFit > kMaxSlots ? kMaxSlots : kFit;
  static constexpr int kOffKV = 0;
  static constexpr int kOffT = kOffKV + kNS * kSlotBytes;
  static constexpr int kOffBar = kOffT + 2 * kTermBytes;
  static constexpr int kSmem = kOffBar + 512 + 1024;
  // tensor memory: S buffers at columns 0 and 64 (P_j over the first 32
  // columns of S_j), Q at 128, O at a multiple of its width
  static constexpr uint32_t kQCol = 128;
  static constexpr uint32_t kOCol = D == 64 ? 192 : 256;
  static constexpr uint32_t kTmemCols = D == 64 ? 256 : 512;
  static constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, 0, 0);
  static constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, D, 0, 1);
  static_assert(kNS >= 2, "shared memory holds fewer than two K/V slots");
  static_assert(kQCol + D / 2 <= kOCol && kOCol + D <= kTmemCols, "tensor memory columns");
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots];
  uint64_t s_full[2], p_full[2], pv_done[2];
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
  const uint64_t* colmask;  // bias / extra-term modes: per (b, query tile, key tile) live columns
  BiasSpec spec;
  float scale_log2;  // scale * log2(e)
  int B, Hq, Hkv, S_q, max_seq, n_pt, n_tiles;
  int32_t* status;
};

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
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

// Position of load `idx` in the producer's order K_0, K_1, V_0, K_2, V_1, ...,
// K_{T-1}, V_{T-2}, V_{T-1}.
__device__ __forceinline__ int k_index(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_index(int j, int T) { return j == T - 1 ? 2 * T - 1 : 2 * j + 2; }

// ---- plan: which keys some row of a query tile may attend -------------------------

// Bit k of word (b, pt, t) of the table says whether some query row of tile
// pt of batch b may attend key 64 t + k: key < nonpad[b] and term > lowest,
// and, for the fused specification's extra term, key inside the row's
// allowed intervals.  Keys outside the allowed intervals are never read.
// One block per (512-key chunk, query tile, batch); shared by all heads.
template <bool FUSED>
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const __nv_bfloat16* __restrict__ term,
                                                                   const int64_t* __restrict__ nonpad,
                                                                   const BiasSpec spec,
                                                                   uint64_t* __restrict__ colmask, int S_q,
                                                                   int max_seq, int n_pt, int n_tiles) {
  const int ch = blockIdx.x, pt = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ uint32_t words[kPlanKeys / 32];
  if (tid < kPlanKeys / 32) words[tid] = 0;
  __syncthreads();
  ptx::grid_launch_dependents();  // the attention kernel may start its prologue
  const int64_t np64 = nonpad[b];
  const bool bad = bad_nonpad(np64, max_seq);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int64_t qs = bad ? 0 : query_start(spec.q_start, b, np64, S_q);
  const int k_begin = ch * kPlanKeys;
  const int k_end = min(k_begin + kPlanKeys, np);
  const int q0 = pt * kBM;
  const int rows = min(kBM, S_q - q0);
  const float lowest = Elem<__nv_bfloat16>::lowest();
  const int kl = k_begin + 16 * lane;  // this lane's 16 keys
  uint32_t acc = 0;
  if (kl < k_end) {
    const uint16_t* base = reinterpret_cast<const uint16_t*>(term) +
                           (static_cast<int64_t>(b) * S_q + q0) * max_seq + kl;
    for (int r0 = warp; r0 < rows; r0 += 32) {
      uint32_t want[4];
      uint4 v[4][2];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = r0 + 8 * rr;
        // keys of this lane the row may attend (16 bits)
        uint32_t m = r < rows ? (k_end - kl >= 16 ? 0xFFFFu : ((1u << (k_end - kl)) - 1)) : 0u;
        if (FUSED && m) {
          const RowWindow w = row_window(spec, b, qs + q0 + r, np);
          uint32_t a = 0;
          if (w.band_lo < w.band_hi) {
            const int64_t lo = w.band_lo - kl, hi = w.band_hi - kl;
            const int l = lo < 0 ? 0 : (lo > 16 ? 16 : static_cast<int>(lo));
            const int h = hi < 0 ? 0 : (hi > 16 ? 16 : static_cast<int>(hi));
            if (l < h) a |= ((h >= 16 ? 0xFFFFu : ((1u << h) - 1)) & ~((1u << l) - 1));
          }
          if (w.span_lo < w.span_hi) {
            const int64_t lo = w.span_lo - kl, hi = w.span_hi - kl;
            const int l = lo < 0 ? 0 : (lo > 16 ? 16 : static_cast<int>(lo));
            const int h = hi < 0 ? 0 : (hi > 16 ? 16 : static_cast<int>(hi));
            if (l < h) a |= ((h >= 16 ? 0xFFFFu : ((1u << h) - 1)) & ~((1u << l) - 1));
          }
          m &= a;
        }
        want[rr] = m;
        const uint16_t* src = base + static_cast<int64_t>(r) * max_seq;
        const uint4 none = make_uint4(0xFF7FFF7Fu, 0xFF7FFF7Fu, 0xFF7FFF7Fu, 0xFF7FFF7Fu);
        // the second vector exists whenever one of its keys is below nonpad (max_seq % 8 == 0)
        v[rr][0] = (m & 0xFFu) ? *reinterpret_cast<const uint4*>(src) : none;
        v[rr][1] = (m & 0xFF00u) ? *reinterpret_cast<const uint4*>(src + 8) : none;
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint16_t* e = reinterpret_cast<const uint16_t*>(&v[rr][h]);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (bf16_bits_to_float(e[q]) > lowest) acc |= (1u << (8 * h + q)) & want[rr];
        }
    }
  }
  if (acc) atomicOr(&words[lane >> 1], acc << (16 * (lane & 1)));
  __syncthreads();
  if (tid < kPlanKeys / 64) {
    const int t = ch * (kPlanKeys / 64) + tid;
    if (t < n_tiles)
      colmask[(static_cast<int64_t>(b) * n_pt + pt) * n_tiles + t] =
          static_cast<uint64_t>(words[2 * tid]) | (static_cast<uint64_t>(words[2 * tid + 1]) << 32);
  }
}

// ---- softmax helpers ------------------------------------------------------------------

// Scores of one 64-key tile in base 2: t = scale*log2(e)*s (+ log2(e)*term),
// -inf where the key is masked: outside the row's allowed keys (PARTIAL
// tiles only; `allowed` bit c) or, with a term, term <= lowest.
template <bool TERM, bool PARTIAL>
__device__ __forceinline__ void tile_scores(float (&t)[kBN], const uint32_t (&sa)[32], const uint32_t (&sb)[32],
                                            const uint32_t (&tw)[32], uint64_t allowed, float sl2,
                                            float lowest) {
  const uint64_t sl2x2 = ptx::f2(sl2, sl2);
  const uint64_t l2e = ptx::f2(kLog2e, kLog2e);
#pragma unroll
  for (int c = 0; c < kBN / 2; ++c) {
    const uint32_t s0 = c < 16 ? sa[2 * c] : sb[2 * c - 32];
    const uint32_t s1 = c < 16 ? sa[2 * c + 1] : sb[2 * c - 31];
    const uint64_t sv = ptx::f2(__uint_as_float(s0), __uint_as_float(s1));
    bool ok0 = true, ok1 = true;
    uint64_t v;
    if (TERM) {
      const float b0 = __uint_as_float(tw[c] << 16), b1 = __uint_as_float(tw[c] & 0xFFFF0000u);
      v = ptx::fma2(sv, sl2x2, ptx::mul2(ptx::f2(b0, b1), l2e));
      ok0 = b0 > lowest;
      ok1 = b1 > lowest;
    } else {
      v = ptx::mul2(sv, sl2x2);
    }
    if (PARTIAL) {
      ok0 = ok0 && ((allowed >> (2 * c)) & 1);
      ok1 = ok1 && ((allowed >> (2 * c + 1)) & 1);
    }
    t[2 * c] = ok0 ? ptx::f2_lo(v) : -INFINITY;
    t[2 * c + 1] = ok1 ? ptx::f2_hi(v) : -INFINITY;
  }
}

__device__ __forceinline__ float tile_max(const float (&t)[kBN]) {
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    acc[k] = ptx::max3(t[k], t[k + 8], t[k + 16]);
    acc[k] = ptx::max3(acc[k], t[k + 24], t[k + 32]);
    acc[k] = ptx::max3(acc[k], t[k + 40], t[k + 48]);
    acc[k] = fmaxf(acc[k], t[k + 56]);
  }
  return ptx::max3(ptx::max3(acc[0], acc[1], acc[2]), ptx::max3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

// ---- the attention kernel ---------------------------------------------------------

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap tmap, const PrefillParams p) {
  using C = Cfg<D, MODE>;
  constexpr bool kFusedMode = MODE == kFused || MODE == kFusedExtra;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKV = sm + C::kOffKV;
  uint8_t* sT = sm + C::kOffT;
  Bars& bar = *reinterpret_cast<Bars*>(sm + C::kOffBar);
  volatile int* abort = &bar.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, pt = blockIdx.y, b = blockIdx.z;
  const int g = p.Hq / p.Hkv;
  const int hk = h / g;
  const int q0 = pt * kBM;

  if (tid == 0) {
    ptx::mbar_init(&bar.q_full, 4 * 32);
    for (int s = 0; s < C::kNS; ++s) {
      ptx::mbar_init(&bar.kv_full[s], 1);
      ptx::mbar_init(&bar.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar.s_full[s], 1);
      ptx::mbar_init(&bar.p_full[s], 4 * 32);
      ptx::mbar_init(&bar.pv_done[s], 1);
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

  const int64_t np64 = p.nonpad[b];
  const bool bad = bad_nonpad(np64, p.max_seq);
  if (bad && tid == 0 && h == 0 && pt == 0) report(p.status, EXTKV_DEV_BAD_NONPAD);
  const int np = bad ? 0 : static_cast<int>(np64);
  const int64_t qs = bad ? 0 : query_start(p.spec.q_start, b, np64, p.S_q);
  const uint64_t* cmrow = C::kTerm ? p.colmask + (static_cast<int64_t>(b) * p.n_pt + pt) * p.n_tiles : nullptr;

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
    // first and last tile with a live key in the plan's column masks
    int lo = INT_MAX, hi = 0;
    const int lim = (np + kBN - 1) / kBN;
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
      bar.range_lo = lo * kBN;
      bar.range_hi = hi * kBN;
    }
  }
  __syncthreads();
  const int rlo = bar.range_lo, rhi = bar.range_hi;
  const int t_lo = rlo < rhi ? rlo / kBN : 0;
  const int T = rlo < rhi ? (rhi + kBN - 1) / kBN - t_lo : 0;  // KV tiles
  const uint32_t tbase = bar.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int unit = b * p.Hkv + hk;
      int issued = 0, t_issued = 0;
      for (int idx = 0; idx < 2 * T; ++idx) {
        const bool is_v = idx == 2 * T - 1 ? true : (idx == 0 ? false : (idx & 1) == 0);
        const int j = idx == 2 * T - 1 ? T - 1 : (is_v ? idx / 2 - 1 : (idx + 1) / 2);
        const int slot = idx % C::kNS;
        if (idx >= C::kNS && !wait_or_abort(&bar.kv_empty[slot], ((idx / C::kNS) - 1) & 1, abort)) break;
        const int key0 = (t_lo + j) * kBN;
        ptx::mbar_arrive_expect_tx(&bar.kv_full[slot], C::kSlotBytes);
        ptx::tma_load_4d(sKV + slot * C::kSlotBytes, is_v ? &vmap : &kmap, &bar.kv_full[slot], 0, key0, 0, unit);
        ++issued;
        if (C::kTerm && !is_v) {
          const int ts = j & 1;
          if (j >= 2 && !wait_or_abort(&bar.t_empty[ts], ((j >> 1) - 1) & 1, abort)) break;
          ptx::mbar_arrive_expect_tx(&bar.t_full[ts], C::kTermBytes);
          ptx::tma_load_2d(sT + ts * C::kTermBytes, &tmap, &bar.t_full[ts], key0, b * p.S_q + q0);
          ++t_issued;
        }
      }
      // copies still in flight after an abort land before the CTA leaves
      if (*abort) {
        for (int idx = issued > C::kNS ? issued - C::kNS : 0; idx < issued; ++idx)
          ptx::mbar_wait_bounded(&bar.kv_full[idx % C::kNS], (idx / C::kNS) & 1, kWaitPolls);
        for (int j = t_issued > 2 ? t_issued - 2 : 0; j < t_issued; ++j)
          ptx::mbar_wait_bounded(&bar.t_full[j & 1], (j >> 1) & 1, kWaitPolls);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      const uint32_t kv_addr = ptx::smem_u32(sKV);
      auto issue_qk = [&](int j) -> bool {
        const int idx = k_index(j), slot = idx % C::kNS;
        if (!wait_or_abort(&bar.kv_full[slot], (idx / C::kNS) & 1, abort)) return false;
        ptx::tc_fence_after();
        const uint32_t d = tbase + (j & 1) * kBN;
        const uint32_t kb = kv_addr + slot * C::kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bd = ptx::smem_desc_sw128(kb + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
          ptx::umma_bf16_ts(d, tbase + C::kQCol + kk * 8, bd, C::kIdescQK, kk > 0);
        }
        ptx::umma_commit(&bar.s_full[j & 1]);
        ptx::umma_commit(&bar.kv_empty[slot]);
        return true;
      };
      bool ok = wait_or_abort(&bar.q_full, 0, abort);
      if (ok) {
        ptx::tc_fence_after();
        ok = issue_qk(0);
      }
      for (int j = 0; j < T && ok; ++j) {
        if (j + 1 < T && !(ok = issue_qk(j + 1))) break;
        if (!(ok = wait_or_abort(&bar.p_full[j & 1], (j >> 1) & 1, abort))) break;
        ptx::tc_fence_after();
        const int idx = v_index(j, T), slot = idx % C::kNS;
        if (!(ok = wait_or_abort(&bar.kv_full[slot], (idx / C::kNS) & 1, abort))) break;
        ptx::tc_fence_after();
        const uint32_t vb = kv_addr + slot * C::kSlotBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t bd = ptx::smem_desc_sw128(vb + ks * 2048, kBN * 128, 1024);
          ptx::umma_bf16_ts(tbase + C::kOCol, tbase + (j & 1) * kBN + ks * 8, bd, C::kIdescPV,
                            (j > 0 || ks > 0) ? 1u : 0u);
        }
        ptx::umma_commit(&bar.pv_done[j & 1]);
        ptx::umma_commit(&bar.kv_empty[slot]);
      }
      // every MMA issued has completed before tensor memory is released
      ptx::umma_commit(&bar.drain);
      if (!ptx::mbar_wait_bounded(&bar.drain, 0, kWaitPolls)) *abort = 1;
    }
  } else {
    // ---------------- softmax and epilogue (one query row per thread) ----------------
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const float sl2 = p.scale_log2;
    const float lowest = Elem<__nv_bfloat16>::lowest();
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    if (T > 0) {
      // this row of Q into tensor memory (rows past the chunk: zeros)
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((static_cast<int64_t>(b) * p.Hq + h) * p.S_q + q0 + row) * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
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
    for (int j = 0; j < T; ++j) {
      const int tile = t_lo + j, key0 = tile * kBN;
      // keys of the tile no row of the CTA attends (their V rows are zeroed)
      const uint64_t dead = C::kTerm ? ~cmrow[tile] : ~bit_range(rlo - key0, rhi - key0);
      // this row's allowed keys before the term test
      const uint64_t allowed = kFusedMode ? (bit_range(a1 - key0, b1 - key0) | bit_range(a2 - key0, b2 - key0))
                                          : bit_range(-key0, np - key0);
      const bool partial = !__all_sync(0xffffffffu, allowed == ~0ull);
      if (!__all_sync(0xffffffffu, wait_or_abort(&bar.s_full[j & 1], (j >> 1) & 1, abort))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t sa[32], sb[32], tw[32];
      ptx::tmem_ld32(tl + (j & 1) * kBN, sa);
      ptx::tmem_ld32(tl + (j & 1) * kBN + 32, sb);
      if (C::kTerm) {
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.t_full[j & 1], (j >> 1) & 1, abort))) {
          ok = false;
          break;
        }
        const uint8_t* trow = sT + (j & 1) * C::kTermBytes + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4*>(trow + ((u ^ (row & 7)) << 4));
          tw[4 * u] = v.x;
          tw[4 * u + 1] = v.y;
          tw[4 * u + 2] = v.z;
          tw[4 * u + 3] = v.w;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar.t_empty[j & 1]);
      }
      ptx::tmem_wait_ld();
      float t[kBN];
      if (partial)
        tile_scores<C::kTerm, true>(t, sa, sb, tw, allowed, sl2, lowest);
      else
        tile_scores<C::kTerm, false>(t, sa, sb, tw, allowed, sl2, lowest);
      const float mt = tile_max(t);
      // lazy rescale: only when the running maximum grows by more than 2^8
      const float m_new = fmaxf(m_run, mt);
      const bool grow = m_new > m_run + 8.f;  // false while the row has no unmasked key
      const bool rescale_o = grow && m_run != -INFINITY;
      const float factor = rescale_o ? ptx::ex2(m_run - m_new) : 1.f;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // the output accumulator holds P_{j-1} V_{j-1} once that product completes
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
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
      const uint64_t nm = ptx::f2(-m_use, -m_use);
      uint64_t ls[4] = {0, 0, 0, 0};
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN / 2; ++c) {
        const uint64_t d = ptx::add2(ptx::f2(t[2 * c], t[2 * c + 1]), nm);
        const float e0 = ptx::ex2(ptx::f2_lo(d)), e1 = ptx::ex2(ptx::f2_hi(d));
        ls[c & 3] = ptx::add2(ls[c & 3], ptx::f2(e0, e1));
        pk[c] = ptx::pack_bf16x2(e0, e1);
      }
      const uint64_t l01 = ptx::add2(ls[0], ls[1]), l23 = ptx::add2(ls[2], ls[3]);
      const uint64_t lsum = ptx::add2(l01, l23);
      l_run += ptx::f2_lo(lsum) + ptx::f2_hi(lsum);
      // P_j over the first half of S_j: QK_{j+2}, the next writer of this
      // buffer, is issued after P_j V_j and the tensor pipe runs in order
      ptx::tmem_st32(tl + (j & 1) * kBN, pk);
      if (dead) {
        const int idx = v_index(j, T), slot = idx % C::kNS;
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.kv_full[slot], (idx / C::kNS) & 1, abort))) {
          ok = false;
          break;
        }
        uint8_t* vt = sKV + slot * C::kSlotBytes;
        for (int w = tid - 64; w < kBN * (D / 64) * 8; w += 128) {
          const int key = w / ((D / 64) * 8), rem = w % ((D / 64) * 8);
          if ((dead >> key) & 1)
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kBN * 128) + key * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
      }
      ptx::tmem_wait_st();
      if (dead) ptx::fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar.p_full[j & 1]);
    }
    // epilogue: O / l, zero rows without an unmasked key
    if (ok && T > 0 &&
        !__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort)))
      ok = false;
    ptx::tc_fence_after();
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    __nv_bfloat16* yrow = p.y + ((static_cast<int64_t>(b) * p.Hq + h) * p.S_q + q0 + row) * D;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (ok && T > 0) {
        ptx::tmem_ld32(tl + C::kOCol + 32 * c, o);
        ptx::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0;
      }
      if (row_valid && ok) {
        uint4* dst = reinterpret_cast<uint4*>(yrow + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv,
                                    __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
          dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  ptx::grid_launch_dependents();
  if (tid == 0 && *abort) report(p.status, EXTKV_DEV_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tbase, C::kTmemCols);
}

// ---- host side ----------------------------------------------------------------------

int n_query_tiles(int64_t S_q) { return static_cast<int>((S_q + kBM - 1) / kBM); }
int n_plan_chunks(int64_t max_seq) { return static_cast<int>((max_seq + kPlanKeys - 1) / kPlanKeys); }
int n_key_tiles(int64_t max_seq) { return static_cast<int>((max_seq + kBN - 1) / kBN); }

template <int D, int MODE>
cudaError_t launch_dm(const AttnArgs& a, const char** name) {
  using C = Cfg<D, MODE>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_prefill_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;

  CUtensorMap kmap, vmap, tmap;
  const uint64_t kv_dims[4] = {64, static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(D / 64),
                               static_cast<uint64_t>(a.B * a.Hkv)};
  const uint64_t kv_strides[3] = {static_cast<uint64_t>(D) * 2, 128, static_cast<uint64_t>(a.max_seq) * D * 2};
  const uint32_t kv_box[4] = {64, kBN, static_cast<uint32_t>(D / 64), 1};
  if (!make_tensor_map_bf16(&kmap, a.k_cache, 4, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_bf16(&vmap, a.v_cache, 4, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  std::memset(&tmap, 0, sizeof tmap);
  const void* term = MODE == kBias ? a.bias : (MODE == kFusedExtra ? a.extra : nullptr);
  if (term) {
    const uint64_t t_dims[2] = {static_cast<uint64_t>(a.max_seq), static_cast<uint64_t>(a.B * a.S_q)};
    const uint64_t t_strides[1] = {static_cast<uint64_t>(a.max_seq) * 2};
    const uint32_t t_box[2] = {kBN, kBM};
    if (!make_tensor_map_bf16(&tmap, term, 2, t_dims, t_strides, t_box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }

  PrefillParams prm;
  prm.y = static_cast<__nv_bfloat16*>(a.y);
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.nonpad = a.nonpad;
  prm.colmask = static_cast<const uint64_t*>(a.workspace);
  prm.spec = BiasSpec{a.causal, a.window, a.span_offsets, a.spans, a.extra, a.q_start};
  prm.scale_log2 = a.scale * kLog2e;
  prm.B = static_cast<int>(a.B);
  prm.Hq = static_cast<int>(a.Hq);
  prm.Hkv = static_cast<int>(a.Hkv);
  prm.S_q = static_cast<int>(a.S_q);
  prm.max_seq = static_cast<int>(a.max_seq);
  prm.n_pt = n_query_tiles(a.S_q);
  prm.n_tiles = n_key_tiles(a.max_seq);
  prm.status = a.status;

  if (C::kTerm) {
    prefill_plan_kernel<MODE == kFusedExtra><<<dim3(n_plan_chunks(a.max_seq), prm.n_pt, prm.B), kPlanThreads, 0,
                                                a.stream>>>(static_cast<const __nv_bfloat16*>(term), a.nonpad,
                                                            prm.spec, static_cast<uint64_t*>(a.workspace),
                                                            prm.S_q, prm.max_seq, prm.n_pt, prm.n_tiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.Hq, prm.n_pt, prm.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_prefill_kernel<D, MODE>, kmap, vmap, tmap, prm);
  if (e != cudaSuccess) return e;
  *name = "attn_prefill_tcgen05";
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const char** name) {
  if (a.bias) return launch_dm<D, kBias>(a, name);
  if (a.fused) return a.extra ? launch_dm<D, kFusedExtra>(a, name) : launch_dm<D, kFused>(a, name);
  return launch_dm<D, kNone>(a, name);
}

}  // namespace

size_t prefill_workspace_bytes(int64_t B, int64_t S_q, int64_t max_seq) {
  return static_cast<size_t>(B) * n_query_tiles(S_q) * n_key_tiles(max_seq) * sizeof(uint64_t);
}

bool prefill_supported(const AttnArgs& a) {
  if (a.dtype != EXTKV_BF16) return false;
  if (a.D != 64 && a.D != 128 && a.D != 256) return false;
  // 16-byte rows for the bias / extra-term copies
  if ((a.bias || (a.fused && a.extra)) && a.max_seq % 8) return false;
  if (a.B * a.Hq * a.S_q > 0x7fffffff || a.B * a.S_q > 0x7fffffff) return false;
  if (a.max_seq > 0x7fffffff - 2 * kPlanKeys || a.B > 65535 || n_query_tiles(a.S_q) > 65535) return false;
  return true;
}

cudaError_t launch_attn_prefill(const AttnArgs& a, const char** name) {
  switch (a.D) {
    case 64: return launch_d<64>(a, name);
    case 128: return launch_d<128>(a, name);
    case 256: return launch_d<256>(a, name);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace extkv
