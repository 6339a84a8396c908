// common.cuh -- device helpers shared by the extkv kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "extkv.h"

namespace extkv {

// ---- element types --------------------------------------------------------

// Exact widening of a bf16 bit pattern.
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  using storage = float;
  // numeric_limits<float>::lowest(): the CPU reference's mask value.
  static constexpr uint32_t kLowestBits = 0xFF7FFFFFu;
  __device__ __forceinline__ static float load(const float* p, int64_t i) { return p[i]; }
  __device__ __forceinline__ static float to_float(float v) { return v; }
  __device__ __forceinline__ static float from_float(float v) { return v; }
  __device__ __forceinline__ static float lowest() { return __uint_as_float(kLowestBits); }
};

template <>
struct Elem<__nv_bfloat16> {
  using storage = __nv_bfloat16;
  static constexpr uint16_t kLowestBits = 0xFF7Fu;
  __device__ __forceinline__ static float load(const __nv_bfloat16* p, int64_t i) {
    return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p)[i]);
  }
  __device__ __forceinline__ static float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_float(float v) { return __float2bfloat16_rn(v); }
  __device__ __forceinline__ static float lowest() { return bf16_bits_to_float(kLowestBits); }
};

// ---- device status word ---------------------------------------------------

__device__ __forceinline__ void report(int32_t* status, int32_t flag) {
  if (status) {
    atomicOr(status, flag);
    atomicAdd(status + 1, 1);
  }
}

// ---- checked builds ----------------------------------------------------------
// Built with EXTKV_CHECKED, the kernels test every plain global load or store
// whose index they compute: elements [first, first + count) must lie in a
// buffer of n elements, else the access is skipped and EXTKV_DEV_BOUNDS is
// flagged in the status word (a bounds check in place of a sanitizer: no trap,
// no fault).  Otherwise the test is the constant true and its arguments are
// not evaluated.
#ifdef EXTKV_CHECKED
__device__ __forceinline__ bool in_bounds(int64_t first, int64_t count, int64_t n, int32_t* status) {
  if (first >= 0 && count >= 0 && first + count <= n) return true;
  report(status, EXTKV_DEV_BOUNDS);
  return false;
}
#define EXTKV_IN(first, count, n, status) ::extkv::in_bounds((first), (count), (n), (status))
#else
#define EXTKV_IN(first, count, n, status) true
#endif

// ---- the bias specification, evaluated on the device -----------------------

// Kernel-parameter copy of extkv_bias_spec.
struct BiasSpec {
  int32_t causal;
  int32_t window;
  const int64_t* span_offsets;
  const int64_t* spans;
  const void* extra;
  const int64_t* q_start;
};

// For one query position p the allowed keys form the union of two intervals
// cut by the padding frontier:
//   band  = [p-W+1, p+1)  (lower end open without a window, upper end open
//                          without causal masking)
//   span  = union of the image spans holding p; spans holding a common point
//           overlap, so their union is one interval [span_lo, span_hi)
//   allowed(j) = j < nonpad && (band_lo <= j < band_hi || span_lo <= j < span_hi)
struct RowWindow {
  int64_t band_lo, band_hi, span_lo, span_hi, nonpad;
  __device__ __forceinline__ bool allowed(int64_t j) const {
    return j < nonpad && ((j >= band_lo && j < band_hi) || (j >= span_lo && j < span_hi));
  }
  // Smallest interval holding every allowed key.
  __device__ __forceinline__ int64_t lo() const {
    int64_t l = band_lo < band_hi ? band_lo : INT64_MAX;
    if (span_lo < span_hi && span_lo < l) l = span_lo;
    return l < 0 ? 0 : l;
  }
  __device__ __forceinline__ int64_t hi() const {
    int64_t h = band_lo < band_hi ? band_hi : INT64_MIN;
    if (span_lo < span_hi && span_hi > h) h = span_hi;
    return h > nonpad ? nonpad : h;
  }
};

// Position of query row 0 of batch b: q_start[b] when given, else the
// bottom-right alignment of an external cache, max(nonpad - S_q, 0)
// ("ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 11).
__device__ __forceinline__ int64_t query_start(const int64_t* q_start, int64_t b, int64_t nonpad,
                                               int64_t S_q) {
  if (q_start) return q_start[b];
  int64_t off = nonpad - S_q;  // signed: may be negative
  return off > 0 ? off : 0;
}

__device__ __forceinline__ RowWindow row_window(const BiasSpec& s, int64_t b, int64_t p,
                                                int64_t nonpad) {
  RowWindow w;
  w.nonpad = nonpad;
  w.band_lo = s.window > 0 ? p - s.window + 1 : INT64_MIN / 2;
  w.band_hi = s.causal ? p + 1 : INT64_MAX / 2;
  w.span_lo = 0;
  w.span_hi = 0;
  if (s.span_offsets && s.spans) {
    int64_t e = s.span_offsets[b + 1];
    for (int64_t k = s.span_offsets[b]; k < e; ++k) {
      int64_t lo = s.spans[2 * k], hi = lo + s.spans[2 * k + 1];
      if (p >= lo && p < hi) {
        if (w.span_lo >= w.span_hi) {
          w.span_lo = lo;
          w.span_hi = hi;
        } else {
          w.span_lo = lo < w.span_lo ? lo : w.span_lo;
          w.span_hi = hi > w.span_hi ? hi : w.span_hi;
        }
      }
    }
  }
  return w;
}

__device__ __forceinline__ bool bad_nonpad(int64_t nonpad, int64_t max_seq) {
  return nonpad < 0 || nonpad > max_seq;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace extkv
