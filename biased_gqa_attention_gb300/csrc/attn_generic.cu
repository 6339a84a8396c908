// attn_generic.cu -- exact-fp32 SIMT attention over the external cache.
//
// One warp per query row (b, h, i).  This is the path for fp32 inputs (the
// tensor-core paths cannot multiply fp32 exactly) and for any supported shape
// the specialised kernels do not take.  Lane l holds elements d = l + 32 t of
// q (Dk of them) and of its running output (Dv); a key's score is a
// warp-wide dot product, then an online-softmax update (running max m,
// running sum l, rescaled output).  Dk and Dv may differ (head_size !=
// v_head_size, "Skill: Attention Optimization", "ORT CUDA Attention Kernel
// Dispatch").
//
// Semantics ("ONNX Domain Attention (Opset 23/24) CUDA Patterns"): section 4
// op order scale*QK^T + bias -> softmax -> @V; section 6 masking (a key is
// unmasked iff j < nonpad and bias > lowest(T)) and exact-zero rows; section 1
// reshape-Q GQA (query head h reads KV head h / (Hq/Hkv)).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace extkv {

namespace {

constexpr int kWarps = 4;

template <typename T, int DPL>
__global__ void __launch_bounds__(32 * kWarps) attn_generic_kernel(
    T* __restrict__ y, const T* __restrict__ q, const T* __restrict__ k_cache,
    const T* __restrict__ v_cache, const T* __restrict__ bias, BiasSpec spec, int fused,
    const int64_t* __restrict__ nonpad, float scale, float softcap, int64_t Hq, int64_t Hkv, int64_t S_q,
    int64_t max_seq, int Dk, int Dv, int64_t rows, int32_t* status) {
  using E = Elem<T>;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const float lowest = E::lowest();
  const T* extra = static_cast<const T*>(spec.extra);

  for (int64_t row = warp0; row < rows; row += nwarps) {
    const int64_t i = row % S_q;
    const int64_t bh = row / S_q;
    const int64_t h = bh % Hq;
    const int64_t b = bh / Hq;
    const int64_t kvh = h / (Hq / Hkv);
    const int64_t np = nonpad[b];
    T* yrow = y + row * Dv;
    if (bad_nonpad(np, max_seq)) {
      if (lane == 0 && h == 0 && i == 0) report(status, EXTKV_DEV_BAD_NONPAD);
      for (int d = lane; d < Dv; d += 32) yrow[d] = E::from_float(0.0f);
      continue;
    }
    float qr[DPL], acc[DPL];
#pragma unroll
    for (int t = 0; t < DPL; ++t) {
      const int d = lane + 32 * t;
      qr[t] = d < Dk ? E::load(q, row * Dk + d) : 0.0f;
      acc[t] = 0.0f;
    }
    const T* kbase = k_cache + (b * Hkv + kvh) * max_seq * Dk;
    const T* vbase = v_cache + (b * Hkv + kvh) * max_seq * Dv;
    const T* brow = bias ? bias + (b * S_q + i) * max_seq : nullptr;
    const T* erow = extra ? extra + (b * S_q + i) * max_seq : nullptr;

    // Keys that can be unmasked lie in [jlo, jhi).
    int64_t jlo = 0, jhi = np;
    RowWindow win{};
    if (fused) {
      const int64_t p = query_start(spec.q_start, b, np, S_q) + i;
      win = row_window(spec, b, p, np);
      jlo = win.lo();
      jhi = win.hi();
    }
    // the keys the row reads, inside the cache rows and the bias row
    if (jhi > jlo && !EXTKV_IN(jlo, jhi - jlo, max_seq, status)) jhi = jlo;
    float m = -INFINITY, l = 0.0f;
    for (int64_t j0 = jlo; j0 < jhi; j0 += 32) {
      // Each lane decides one key of this group of 32; the warp then walks
      // the unmasked ones.
      const int64_t jm = j0 + lane;
      bool live = jm < jhi;
      float bj = 0.0f;
      if (live) {
        if (brow) {
          bj = E::load(brow, jm);
          live = bj > lowest;
        } else if (fused) {
          live = win.allowed(jm);
          if (live && erow) {
            bj = E::load(erow, jm);
            live = bj > lowest;
          }
        }
      }
      unsigned mask = __ballot_sync(0xffffffffu, live);
      while (mask) {
        const int src = __ffs(mask) - 1;
        mask &= mask - 1;
        const int64_t j = j0 + src;
        const float bb = __shfl_sync(0xffffffffu, bj, src);
        const T* kr = kbase + j * Dk;
        const T* vr = vbase + j * Dv;
        float part = 0.0f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
          const int d = lane + 32 * t;
          if (d < Dk) part = fmaf(qr[t], E::load(kr, d), part);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        // softcap (if > 0) on the scaled score, before the bias (section 4 op order)
        const float s = softcap > 0.f ? fmaf(softcap, tanhf(scale * part / softcap), bb) : fmaf(scale, part, bb);
        const float m_new = fmaxf(m, s);
        // Differences are formed before any scaling, so an extreme finite
        // score can never overflow to -inf and be mistaken for a mask.
        const float corr = expf(m - m_new);
        const float pj = expf(s - m_new);
        l = fmaf(l, corr, pj);
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
          const int d = lane + 32 * t;
          const float vv = d < Dv ? E::load(vr, d) : 0.0f;
          acc[t] = fmaf(pj, vv, acc[t] * corr);
        }
        m = m_new;
      }
    }
    // No unmasked key: exact zero row (select, not multiply).
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) {
      const int d = lane + 32 * t;
      if (d < Dv) yrow[d] = E::from_float(l > 0.0f ? acc[t] * inv : 0.0f);
    }
  }
}

template <typename T, int DPL>
void launch_dpl(const AttnArgs& a, int blocks, const BiasSpec& spec, int64_t rows) {
  attn_generic_kernel<T, DPL><<<blocks, 32 * kWarps, 0, a.stream>>>(
      static_cast<T*>(a.y), static_cast<const T*>(a.q), static_cast<const T*>(a.k_cache),
      static_cast<const T*>(a.v_cache), static_cast<const T*>(a.bias), spec, a.fused, a.nonpad,
      a.scale, a.softcap, a.Hq, a.Hkv, a.S_q, a.max_seq, static_cast<int>(a.D), static_cast<int>(a.Dv), rows,
      a.status);
}

template <typename T>
cudaError_t launch_typed(const AttnArgs& a) {
  const int64_t rows = a.B * a.Hq * a.S_q;
  const int64_t want = (rows + kWarps - 1) / kWarps;
  const int blocks = static_cast<int>(std::min<int64_t>(want, int64_t(num_sms()) * 16));
  BiasSpec spec{a.causal, a.window, a.span_offsets, a.spans, a.extra, a.q_start};
  const int64_t dpl = (std::max(a.D, a.Dv) + 31) / 32;  // elements per lane, Dk, Dv <= 512
  if (dpl <= 1) launch_dpl<T, 1>(a, blocks, spec, rows);
  else if (dpl <= 2) launch_dpl<T, 2>(a, blocks, spec, rows);
  else if (dpl <= 4) launch_dpl<T, 4>(a, blocks, spec, rows);
  else if (dpl <= 8) launch_dpl<T, 8>(a, blocks, spec, rows);
  else launch_dpl<T, 16>(a, blocks, spec, rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_generic(const AttnArgs& a, const char** name) {
  *name = a.dtype == EXTKV_F32 ? "attn_generic_f32" : "attn_generic_bf16";
  if (a.B * a.Hq * a.S_q == 0) return cudaSuccess;
  note_launches(1);
  return a.dtype == EXTKV_F32 ? launch_typed<float>(a) : launch_typed<__nv_bfloat16>(a);
}

}  // namespace extkv
