// scatter_bias.cu -- the TensorScatter write into the static cache and the
// static-cache bias builder.  Both are pure HBM streams: 16-byte vector loads
// and stores, grid-stride loops over a grid sized to the SM count.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace extkv {

namespace {

cudaLaunchConfig_t pdl_config(int blocks, int threads, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  return cfg;
}

// Programmatic dependent launch: the kernel may be scheduled while the
// previous kernel in the stream drains; it waits (griddepcontrol.wait)
// before touching global memory.
void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

}  // namespace

// ---- TensorScatter ----------------------------------------------------------
// "Skill: Attention Optimization", "In-place KV for ONNX Attention via
// TensorScatter (static cache)": new rows go to slot write_idx[b] + s of the
// preallocated (B,Hkv,max_seq,D) buffer; nothing is concatenated.
//
// One 16-byte vector per loop trip, for K and for V.  Row r of the update
// (b,h,s) is contiguous, as is its destination row, so consecutive threads
// touch consecutive vectors on both sides.
__global__ void __launch_bounds__(256) scatter_kernel(uint4* __restrict__ k_cache,
                                                      uint4* __restrict__ v_cache,
                                                      const uint4* __restrict__ k_new,
                                                      const uint4* __restrict__ v_new,
                                                      const int64_t* __restrict__ write_idx,
                                                      int64_t Hkv, int64_t S_new, int64_t max_seq,
                                                      int64_t row_vecs, int64_t total,
                                                      int32_t* status) {
  // Launched as a programmatic dependent: wait for the previous grid's memory
  // (the previous step may still read these cache rows), then let the next
  // kernel start its prologue.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int64_t v = idx % row_vecs;
    const int64_t r = idx / row_vecs;  // (b*Hkv + h)*S_new + s
    const int64_t s = r % S_new;
    const int64_t bh = r / S_new;
    const int64_t b = bh / Hkv;
    const int64_t n_bh = total / (S_new * row_vecs);  // batches x KV heads
    if (!EXTKV_IN(b, 1, n_bh / Hkv, status)) continue;
    const int64_t w = write_idx[b];
    if (w < 0 || w > max_seq - S_new) {
      if (v == 0 && s == 0 && bh % Hkv == 0) report(status, EXTKV_DEV_BAD_WRITE_IDX);
      continue;
    }
    const int64_t dst = (bh * max_seq + w + s) * row_vecs + v;
    if (!EXTKV_IN(dst, 1, n_bh * max_seq * row_vecs, status)) continue;
    const uint4 kx = __ldg(k_new + idx);
    const uint4 vx = __ldg(v_new + idx);
    k_cache[dst] = kx;
    v_cache[dst] = vx;
  }
}

cudaError_t launch_scatter(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                           const int64_t* write_idx, int64_t B, int64_t Hkv, int64_t S_new,
                           int64_t max_seq, int64_t D, int dtype, int32_t* status,
                           cudaStream_t stream) {
  const int64_t es = dtype == EXTKV_F32 ? 4 : 2;
  const int64_t row_vecs = D * es / 16;
  const int64_t total = B * Hkv * S_new * row_vecs;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(std::min<int64_t>(want, int64_t(num_sms()) * 8));
  cudaLaunchConfig_t cfg = pdl_config(blocks, threads, stream);
  cudaLaunchAttribute attr[1];
  pdl_attr(cfg, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, scatter_kernel, static_cast<uint4*>(k_cache),
                                     static_cast<uint4*>(v_cache), static_cast<const uint4*>(k_new),
                                     static_cast<const uint4*>(v_new), write_idx, Hkv, S_new,
                                     max_seq, row_vecs, total, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- static-cache bias ------------------------------------------------------
// mobius issue #366, deliverable: the (B,1,S_q,max_seq) additive bias keyed on
// absolute query positions (causal + sliding + block overlay + padding, valid
// only where slot < nonpad).  One block per row (grid-stride over rows): the
// row's allowed keys are two intervals, computed once; the block's threads
// then stream the row's 16-byte vectors (coalesced stores; with an extra term
// each vector is a select between it and the sentinel).
template <typename T>
__global__ void __launch_bounds__(256) bias_kernel(uint4* __restrict__ bias, BiasSpec spec,
                                                   const int64_t* __restrict__ nonpad, int64_t S_q,
                                                   int64_t max_seq, int64_t row_vecs, int64_t rows,
                                                   int32_t* status) {
  constexpr int kVec = 16 / sizeof(T);
  using E = Elem<T>;
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  const uint4* extra = static_cast<const uint4*>(spec.extra);
  union Vec {
    uint4 u;
    T e[kVec];
  };
  Vec low, zero;
#pragma unroll
  for (int e = 0; e < kVec; ++e) {
    low.e[e] = E::from_float(E::lowest());
    zero.e[e] = E::from_float(0.0f);
  }
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {  // r = b*S_q + i
    const int64_t i = r % S_q;
    const int64_t b = r / S_q;
    if (!EXTKV_IN(b, 1, rows / S_q, status)) continue;
    const int64_t np = nonpad[b];
    uint4* out = bias + r * row_vecs;
    const uint4* ext = extra ? extra + r * row_vecs : nullptr;
    if (bad_nonpad(np, max_seq)) {
      if (i == 0 && threadIdx.x == 0) report(status, EXTKV_DEV_BAD_NONPAD);
      continue;
    }
    const int64_t p = query_start(spec.q_start, b, np, S_q) + i;
    const RowWindow w = row_window(spec, b, p, np);
    // allowed keys: [a1, b1) U [a2, b2), both inside [0, nonpad)
    const int64_t bl = w.band_lo < 0 ? 0 : w.band_lo, bh = w.band_hi < np ? w.band_hi : np;
    const int64_t sl = w.span_lo < 0 ? 0 : w.span_lo, sh = w.span_hi < np ? w.span_hi : np;
    const int a1 = static_cast<int>(bl < bh ? bl : 0), b1 = static_cast<int>(bl < bh ? bh : 0);
    const int a2 = static_cast<int>(sl < sh ? sl : 0), b2 = static_cast<int>(sl < sh ? sh : 0);
    for (int64_t jv = threadIdx.x; jv < row_vecs; jv += blockDim.x) {
      const int j0 = static_cast<int>(jv * kVec);
      const bool all_in = (j0 >= a1 && j0 + kVec <= b1) || (j0 >= a2 && j0 + kVec <= b2);
      const bool all_out = (j0 + kVec <= a1 || j0 >= b1) && (j0 + kVec <= a2 || j0 >= b2);
      Vec v;
      if (all_out) {
        v = low;
      } else if (all_in) {
        v.u = ext ? __ldg(ext + jv) : zero.u;
      } else {
        Vec x;
        x.u = ext ? __ldg(ext + jv) : zero.u;
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          const int j = j0 + e;
          const bool ok = (j >= a1 && j < b1) || (j >= a2 && j < b2);
          v.e[e] = ok ? x.e[e] : low.e[e];
        }
      }
      if (EXTKV_IN(r * row_vecs + jv, 1, rows * row_vecs, status)) out[jv] = v.u;
    }
  }
}

cudaError_t launch_bias(void* bias, const extkv_bias_spec& s, const int64_t* nonpad, int64_t B,
                        int64_t S_q, int64_t max_seq, int dtype, int32_t* status,
                        cudaStream_t stream) {
  const int64_t es = dtype == EXTKV_F32 ? 4 : 2;
  const int64_t row_vecs = max_seq * es / 16;
  const int64_t rows = B * S_q;
  if (rows == 0) return cudaSuccess;
  BiasSpec spec{s.causal, s.window, s.span_offsets, s.spans, s.extra, s.q_start};
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>(rows, int64_t(num_sms()) * 8));
  cudaLaunchConfig_t cfg = pdl_config(blocks, threads, stream);
  cudaLaunchAttribute attr[1];
  pdl_attr(cfg, attr);
  cudaError_t e =
      dtype == EXTKV_F32
          ? cudaLaunchKernelEx(&cfg, bias_kernel<float>, static_cast<uint4*>(bias), spec, nonpad,
                               S_q, max_seq, row_vecs, rows, status)
          : cudaLaunchKernelEx(&cfg, bias_kernel<__nv_bfloat16>, static_cast<uint4*>(bias), spec,
                               nonpad, S_q, max_seq, row_vecs, rows, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- a boolean attention mask as the additive bias ------------------------
// "ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 6 (additive-bias
// path: a bool mask is converted to a bias) and the attention-mask skill ("Bool
// mask vs float additive bias"): an attended slot (mask byte != 0) gets 0, a
// masked slot lowest(T), the same sentinel the bias builder writes.  16 mask
// bytes per step (one 16-byte load) become 16 elements (two or four 16-byte
// stores); a ragged tail of fewer than 16 elements is done element by element.
template <typename T>
__global__ void __launch_bounds__(256) mask_bias_kernel(T* __restrict__ bias, const uint8_t* __restrict__ mask,
                                                        int64_t n) {
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  const T low = Elem<T>::from_float(Elem<T>::lowest());
  const T zero = Elem<T>::from_float(0.f);
  const int64_t nv = n / 16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nv; v += stride) {
    const uint4 m = __ldg(reinterpret_cast<const uint4*>(mask) + v);
    const uint8_t* mb = reinterpret_cast<const uint8_t*>(&m);
    constexpr int kPerVec = 16 / sizeof(T);  // elements per 16-byte store
    uint4* out = reinterpret_cast<uint4*>(bias + v * 16);
#pragma unroll
    for (int q = 0; q < 16 / kPerVec; ++q) {
      union {
        uint4 u;
        T e[kPerVec];
      } w;
#pragma unroll
      for (int e = 0; e < kPerVec; ++e) w.e[e] = mb[q * kPerVec + e] ? zero : low;
      out[q] = w.u;
    }
  }
  for (int64_t i = nv * 16 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    bias[i] = mask[i] ? zero : low;
}

cudaError_t launch_mask_bias(void* bias, const uint8_t* mask, int64_t n, int dtype, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (n / 16 + threads - 1) / threads;
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(num_sms()) * 8)));
  cudaLaunchConfig_t cfg = pdl_config(blocks, threads, stream);
  cudaLaunchAttribute attr[1];
  pdl_attr(cfg, attr);
  cudaError_t e = dtype == EXTKV_F32
                      ? cudaLaunchKernelEx(&cfg, mask_bias_kernel<float>, static_cast<float*>(bias), mask, n)
                      : cudaLaunchKernelEx(&cfg, mask_bias_kernel<__nv_bfloat16>,
                                           static_cast<__nv_bfloat16*>(bias), mask, n);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace extkv
