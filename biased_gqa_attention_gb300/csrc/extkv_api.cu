// extkv_api.cu -- the C ABI: argument validation, kernel choice, error
// reporting.  Every check here happens on the host before any launch; the
// kernels themselves only see data-dependent errors (status word).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "extkv.h"
#include "internal.h"

namespace extkv {

namespace {

thread_local char g_error[512] = "";
thread_local const char* g_last_kernel = "";
thread_local int g_launches = 0, g_last_launches = 0;
thread_local int g_algo = EXTKV_ALGO_AUTO;
thread_local uint32_t g_wait_limit_plus1 = 0;  // 0: the kernels' own limit; n + 1: n polls

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_error, sizeof g_error, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(EXTKV_ERR_CUDA, "%s: CUDA error %d (%s)", what, static_cast<int>(e),
              cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t elem_size(int dtype) { return dtype == EXTKV_F32 ? 4 : 2; }

bool valid_dtype(int dtype) { return dtype == EXTKV_F32 || dtype == EXTKV_BF16; }

int check_workspace(const AttnArgs& a, size_t need) {
  if (a.ws_bytes < need || (need && !a.workspace))
    return fail(EXTKV_ERR_INVALID_ARG,
                "attention_ext_kv: workspace of %zu bytes required (got %zu); query attention_ext_kv_workspace_size",
                need, a.ws_bytes);
  if (!aligned(a.workspace, 256))
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: workspace must be 256-byte aligned");
  return EXTKV_OK;
}

}  // namespace

void set_error(const char* msg) { snprintf(g_error, sizeof g_error, "%s", msg); }

void note_launches(int n) { g_launches = n; }

uint32_t wait_limit_setting() { return g_wait_limit_plus1; }

void note_last_call(const char* name) {
  g_last_kernel = name;
  g_last_launches = g_launches;
}

int num_sms() {
  // Cached per device; the SM count never changes for a device.
  static thread_local int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

}  // namespace extkv

using namespace extkv;

extern "C" {

int ext_kv_scatter(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                   const int64_t* write_idx, int64_t B, int64_t Hkv, int64_t S_new,
                   int64_t max_seq, int64_t D, int dtype, int32_t* status, void* stream) {
  g_error[0] = 0;
  if (!valid_dtype(dtype)) return fail(EXTKV_ERR_INVALID_ARG, "ext_kv_scatter: unknown dtype %d", dtype);
  if (B < 0 || Hkv <= 0 || S_new < 0 || max_seq <= 0 || D <= 0)
    return fail(EXTKV_ERR_INVALID_ARG,
                "ext_kv_scatter: bad sizes B=%lld Hkv=%lld S_new=%lld max_seq=%lld D=%lld",
                (long long)B, (long long)Hkv, (long long)S_new, (long long)max_seq, (long long)D);
  if (S_new > max_seq)
    return fail(EXTKV_ERR_INVALID_ARG, "ext_kv_scatter: S_new=%lld exceeds max_seq=%lld",
                (long long)S_new, (long long)max_seq);
  if (B == 0 || S_new == 0) return EXTKV_OK;  // an empty update writes nothing
  if (!k_cache || !v_cache || !k_new || !v_new || !write_idx)
    return fail(EXTKV_ERR_INVALID_ARG, "ext_kv_scatter: null pointer");
  if ((D * elem_size(dtype)) % 16)
    return fail(EXTKV_ERR_UNSUPPORTED, "ext_kv_scatter: D*sizeof(T) must be a multiple of 16 (D=%lld)",
                (long long)D);
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
      !aligned(write_idx, 8) || !aligned(status, 4))
    return fail(EXTKV_ERR_INVALID_ARG, "ext_kv_scatter: tensors must be 16-byte aligned");
  cudaError_t e = launch_scatter(k_cache, v_cache, k_new, v_new, write_idx, B, Hkv, S_new, max_seq,
                                 D, dtype, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ext_kv_scatter launch");
  return EXTKV_OK;
}

int build_static_cache_bias(void* bias, const extkv_bias_spec* spec, const int64_t* nonpad,
                            int64_t B, int64_t S_q, int64_t max_seq, int dtype, int32_t* status,
                            void* stream) {
  g_error[0] = 0;
  if (!valid_dtype(dtype)) return fail(EXTKV_ERR_INVALID_ARG, "build_static_cache_bias: unknown dtype %d", dtype);
  if (B < 0 || S_q < 0 || max_seq <= 0)
    return fail(EXTKV_ERR_INVALID_ARG, "build_static_cache_bias: bad sizes B=%lld S_q=%lld max_seq=%lld",
                (long long)B, (long long)S_q, (long long)max_seq);
  if (B == 0 || S_q == 0) return EXTKV_OK;
  if (!bias || !spec || !nonpad) return fail(EXTKV_ERR_INVALID_ARG, "build_static_cache_bias: null pointer");
  if ((spec->span_offsets == nullptr) != (spec->spans == nullptr))
    return fail(EXTKV_ERR_INVALID_ARG, "build_static_cache_bias: span_offsets and spans must be given together");
  if ((max_seq * elem_size(dtype)) % 16)
    return fail(EXTKV_ERR_UNSUPPORTED,
                "build_static_cache_bias: max_seq*sizeof(T) must be a multiple of 16 (max_seq=%lld)",
                (long long)max_seq);
  if (max_seq > 0x7fffff00)
    return fail(EXTKV_ERR_UNSUPPORTED, "build_static_cache_bias: max_seq=%lld exceeds 2^31 - 256",
                (long long)max_seq);
  if (!aligned(bias, 16) || (spec->extra && !aligned(spec->extra, 16)) || !aligned(status, 4))
    return fail(EXTKV_ERR_INVALID_ARG, "build_static_cache_bias: bias/extra must be 16-byte aligned");
  cudaError_t e = launch_bias(bias, *spec, nonpad, B, S_q, max_seq, dtype, status,
                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "build_static_cache_bias launch");
  return EXTKV_OK;
}

int build_bias_from_bool_mask(void* bias, const uint8_t* mask, int64_t B, int64_t S_q, int64_t max_seq, int dtype,
                              void* stream) {
  g_error[0] = 0;
  if (!valid_dtype(dtype)) return fail(EXTKV_ERR_INVALID_ARG, "build_bias_from_bool_mask: unknown dtype %d", dtype);
  if (B < 0 || S_q < 0 || max_seq <= 0)
    return fail(EXTKV_ERR_INVALID_ARG, "build_bias_from_bool_mask: bad sizes B=%lld S_q=%lld max_seq=%lld",
                (long long)B, (long long)S_q, (long long)max_seq);
  const int64_t n = B * S_q * max_seq;
  if (n == 0) return EXTKV_OK;
  if (!bias || !mask) return fail(EXTKV_ERR_INVALID_ARG, "build_bias_from_bool_mask: null pointer");
  if (!aligned(bias, 16) || !aligned(mask, 16))
    return fail(EXTKV_ERR_INVALID_ARG, "build_bias_from_bool_mask: bias and mask must be 16-byte aligned");
  cudaError_t e = launch_mask_bias(bias, mask, n, dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "build_bias_from_bool_mask launch");
  return EXTKV_OK;
}

size_t attention_ext_kv_workspace_size_dv(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq,
                                          int64_t Dk, int64_t Dv, int dtype) {
  // The decode kernel keeps its plan and its split-unit partials there; the
  // prefill kernel keeps the live key ranges of a materialised bias and the
  // partials of key splits.
  if (dtype != EXTKV_BF16 || B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || S_q <= 0 || max_seq <= 0) return 0;
  AttnArgs a{};
  a.dtype = dtype;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S_q = S_q;
  a.max_seq = max_seq;
  a.D = Dk;
  a.Dv = Dv;
  // enough for whichever kernel runs, automatic or chosen by extkv_set_algo
  size_t need = 0;
  if (decode_supported(a)) need = decode_workspace_bytes(B, Hq, Hkv, S_q, max_seq, Dk, Dv);
  if (prefill_supported(a)) {
    const size_t pf = prefill_workspace_bytes(B, Hq, Hkv, S_q, max_seq, Dk, Dv, true);
    need = pf > need ? pf : need;
  }
  return need;
}

size_t attention_ext_kv_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq,
                                       int64_t D, int dtype) {
  return attention_ext_kv_workspace_size_dv(B, Hq, Hkv, S_q, max_seq, D, D, dtype);
}

}  // extern "C"

namespace extkv {
namespace {

// A scatter to fuse into the attention call (ext_kv_scatter's arguments).
struct ScatterIn {
  void* k_cache;
  void* v_cache;
  const void* k_new;
  const void* v_new;
  const int64_t* write_idx;
  int64_t S_new;
};

int attention_impl(void* y, const void* q, const void* k_cache, const void* v_cache, const void* bias,
                   const extkv_bias_spec* fused, const int64_t* nonpad, float scale, int64_t B, int64_t Hq,
                   int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t D, int64_t Dv, int dtype, void* workspace,
                   size_t ws_bytes, int32_t* status, void* stream, const ScatterIn* sc, float softcap = 0.f) {
  if (!valid_dtype(dtype)) return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: unknown dtype %d", dtype);
  if (B < 0 || S_q < 0 || Hq <= 0 || Hkv <= 0 || max_seq <= 0 || D <= 0)
    return fail(EXTKV_ERR_INVALID_ARG,
                "attention_ext_kv: bad sizes B=%lld Hq=%lld Hkv=%lld S_q=%lld max_seq=%lld D=%lld",
                (long long)B, (long long)Hq, (long long)Hkv, (long long)S_q, (long long)max_seq,
                (long long)D);
  if (Hq % Hkv)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: Hq=%lld is not a multiple of Hkv=%lld",
                (long long)Hq, (long long)Hkv);
  if (D % 8 || D > 512)
    return fail(EXTKV_ERR_UNSUPPORTED, "attention_ext_kv: D=%lld unsupported (need D %% 8 == 0, D <= 512)",
                (long long)D);
  if (Dv <= 0 || Dv % 8 || Dv > 512)
    return fail(EXTKV_ERR_UNSUPPORTED, "attention_ext_kv: Dv=%lld unsupported (need Dv %% 8 == 0, 0 < Dv <= 512)",
                (long long)Dv);
  if (sc && Dv != D)
    return fail(EXTKV_ERR_UNSUPPORTED, "attention_ext_kv_scatter: one head size for keys and values");
  if (bias && fused)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: pass either a materialised bias or a fused spec, not both");
  if (B == 0 || S_q == 0) {
    if (!sc) return EXTKV_OK;
    cudaError_t e = launch_scatter(sc->k_cache, sc->v_cache, sc->k_new, sc->v_new, sc->write_idx, B, Hkv,
                                   sc->S_new, max_seq, D, dtype, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? EXTKV_OK : cuda_fail(e, "attention_ext_kv_scatter launch");
  }
  if (!y || !q || !k_cache || !v_cache || !nonpad)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: null pointer");
  if (fused && ((fused->span_offsets == nullptr) != (fused->spans == nullptr)))
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: span_offsets and spans must be given together");
  const size_t al = 16;
  if (!aligned(y, al) || !aligned(q, al) || !aligned(k_cache, al) || !aligned(v_cache, al) ||
      (bias && !aligned(bias, al)) || (fused && fused->extra && !aligned(fused->extra, al)) ||
      !aligned(nonpad, 8) || !aligned(status, 4))
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv: tensors must be 16-byte aligned");

  AttnArgs a{};
  a.y = y;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.bias = bias;
  a.fused = fused != nullptr;
  if (fused) {
    a.extra = fused->extra;
    a.span_offsets = fused->span_offsets;
    a.spans = fused->spans;
    a.q_start = fused->q_start;
    a.causal = fused->causal;
    a.window = fused->window;
  }
  a.nonpad = nonpad;
  a.scale = scale;
  a.softcap = softcap;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S_q = S_q;
  a.max_seq = max_seq;
  a.D = D;
  a.Dv = Dv;
  a.dtype = dtype;
  a.status = status;
  a.workspace = workspace;
  a.ws_bytes = ws_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_limit_plus1 = g_wait_limit_plus1;
  a.prefill_pairs = g_algo == EXTKV_ALGO_PREFILL_PAIR ? 1 : 0;
  a.decode_variant = g_algo == EXTKV_ALGO_DECODE_STREAMK   ? kDecodeStreamK
                     : g_algo == EXTKV_ALGO_DECODE_CLUSTER ? kDecodeCluster
                                                           : kDecodeAuto;

  const char* name = "";
  cudaError_t e;
  g_launches = 0;
  int extra_launches = 0;  // a scatter kernel launched ahead of an unfused path
  // the decode kernel takes the scatter; the other paths get the scatter kernel first
  auto launch_decode_with = [&](AttnArgs& aa, const ScatterIn* s, const char** nm) {
    if (s) {
      aa.kc_w = s->k_cache;
      aa.vc_w = s->v_cache;
      aa.k_new = s->k_new;
      aa.v_new = s->v_new;
      aa.write_idx = s->write_idx;
      aa.S_new = s->S_new;
    }
    return launch_attn_decode(aa, nm);
  };
  auto scatter_first = [&](const AttnArgs& aa, const ScatterIn* s) -> cudaError_t {
    if (!s) return cudaSuccess;
    ++extra_launches;
    return launch_scatter(s->k_cache, s->v_cache, s->k_new, s->v_new, s->write_idx, aa.B, aa.Hkv, s->S_new,
                          aa.max_seq, aa.D, aa.dtype, aa.status, aa.stream);
  };
  const size_t decode_ws = decode_workspace_bytes(B, Hq, Hkv, S_q, max_seq, D, Dv);
  // a materialised bias or an extra term needs the prefill kernel's column-mask table
  // the column-mask table (a materialised bias or an extra term) and the
  // partials of key splits (small grids)
  const size_t prefill_ws = prefill_workspace_bytes(B, Hq, Hkv, S_q, max_seq, D, Dv, bias || (fused && fused->extra));
  switch (g_algo) {
    case EXTKV_ALGO_GENERIC:
      if ((e = scatter_first(a, sc)) != cudaSuccess) break;
      e = launch_attn_generic(a, &name);
      break;
    case EXTKV_ALGO_DECODE:
    case EXTKV_ALGO_DECODE_STREAMK:
    case EXTKV_ALGO_DECODE_CLUSTER:
      if (!decode_supported(a))
        return fail(EXTKV_ERR_UNSUPPORTED, "attention_ext_kv: the decode kernel cannot run this shape/type");
      if (int rc = check_workspace(a, decode_ws)) return rc;
      e = launch_decode_with(a, sc, &name);
      break;
    case EXTKV_ALGO_PREFILL:
    case EXTKV_ALGO_PREFILL_PAIR:
      if (!prefill_supported(a))
        return fail(EXTKV_ERR_UNSUPPORTED, "attention_ext_kv: the prefill kernel cannot run this shape/type");
      if (int rc = check_workspace(a, prefill_ws)) return rc;
      if ((e = scatter_first(a, sc)) != cudaSuccess) break;
      e = launch_attn_prefill(a, &name);
      break;
    default:
      if (decode_supported(a)) {
        if (int rc = check_workspace(a, decode_ws)) return rc;
        e = launch_decode_with(a, sc, &name);
      } else if (prefill_supported(a)) {
        if (int rc = check_workspace(a, prefill_ws)) return rc;
        if ((e = scatter_first(a, sc)) != cudaSuccess) break;
        e = launch_attn_prefill(a, &name);
      } else {
        if ((e = scatter_first(a, sc)) != cudaSuccess) break;
        e = launch_attn_generic(a, &name);
      }
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention_ext_kv launch");
  g_last_kernel = name;
  g_last_launches = g_launches + extra_launches;
  return EXTKV_OK;
}

}  // namespace
}  // namespace extkv

extern "C" {

int attention_ext_kv(void* y, const void* q, const void* k_cache, const void* v_cache,
                     const void* bias, const extkv_bias_spec* fused, const int64_t* nonpad,
                     float scale, int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq,
                     int64_t D, int dtype, void* workspace, size_t ws_bytes, int32_t* status,
                     void* stream) {
  g_error[0] = 0;
  return attention_impl(y, q, k_cache, v_cache, bias, fused, nonpad, scale, B, Hq, Hkv, S_q, max_seq, D, D, dtype,
                        workspace, ws_bytes, status, stream, nullptr);
}

int attention_ext_kv_softcap(void* y, const void* q, const void* k_cache, const void* v_cache,
                             const void* bias, const extkv_bias_spec* fused, const int64_t* nonpad,
                             float scale, float softcap, int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q,
                             int64_t max_seq, int64_t D, int dtype, void* workspace, size_t ws_bytes,
                             int32_t* status, void* stream) {
  g_error[0] = 0;
  if (!(softcap >= 0.f) || softcap == INFINITY)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_softcap: softcap must be finite and >= 0");
  return attention_impl(y, q, k_cache, v_cache, bias, fused, nonpad, scale, B, Hq, Hkv, S_q, max_seq, D, D, dtype,
                        workspace, ws_bytes, status, stream, nullptr, softcap);
}

int attention_ext_kv_dv(void* y, const void* q, const void* k_cache, const void* v_cache, const void* bias,
                        const extkv_bias_spec* fused, const int64_t* nonpad, float scale, float softcap, int64_t B,
                        int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk, int64_t Dv, int dtype,
                        void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  g_error[0] = 0;
  if (!(softcap >= 0.f) || softcap == INFINITY)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_dv: softcap must be finite and >= 0");
  return attention_impl(y, q, k_cache, v_cache, bias, fused, nonpad, scale, B, Hq, Hkv, S_q, max_seq, Dk, Dv, dtype,
                        workspace, ws_bytes, status, stream, nullptr, softcap);
}

int attention_ext_kv_scatter(void* y, const void* q, void* k_cache, void* v_cache, const void* k_new,
                             const void* v_new, const int64_t* write_idx, int64_t S_new, const void* bias,
                             const extkv_bias_spec* fused, const int64_t* nonpad, float scale, int64_t B,
                             int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t D, int dtype,
                             void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  g_error[0] = 0;
  if (!valid_dtype(dtype))
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_scatter: unknown dtype %d", dtype);
  if (S_new < 0 || S_new > max_seq)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_scatter: S_new=%lld outside [0, max_seq=%lld]",
                (long long)S_new, (long long)max_seq);
  if (B > 0 && S_new > 0) {
    if (!k_cache || !v_cache || !k_new || !v_new || !write_idx)
      return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_scatter: null pointer");
    if (D <= 0 || (D * elem_size(dtype)) % 16)
      return fail(EXTKV_ERR_UNSUPPORTED, "attention_ext_kv_scatter: D*sizeof(T) must be a multiple of 16 (D=%lld)",
                  (long long)D);
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(write_idx, 8))
      return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_scatter: tensors must be 16-byte aligned");
  }
  const ScatterIn sc{k_cache, v_cache, k_new, v_new, write_idx, S_new};
  return attention_impl(y, q, k_cache, v_cache, bias, fused, nonpad, scale, B, Hq, Hkv, S_q, max_seq, D, D, dtype,
                        workspace, ws_bytes, status, stream, (B > 0 && S_new > 0) ? &sc : nullptr);
}

int extkv_clear_status(int32_t* status, void* stream) {
  g_error[0] = 0;
  if (!status || !aligned(status, 4)) return fail(EXTKV_ERR_INVALID_ARG, "extkv_clear_status: bad pointer");
  cudaError_t e = cudaMemsetAsync(status, 0, 16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "extkv_clear_status");
  return EXTKV_OK;
}

int extkv_read_status(const int32_t* status, void* stream) {
  g_error[0] = 0;
  if (!status || !aligned(status, 4)) return fail(EXTKV_ERR_INVALID_ARG, "extkv_read_status: bad pointer");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "extkv_read_status: stream sync");
  int32_t h[4] = {0, 0, 0, 0};
  e = cudaMemcpy(h, status, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "extkv_read_status: copy");
  if (h[0] == 0) return EXTKV_OK;
  return fail(EXTKV_ERR_DEVICE, "device status 0x%x (%d unit(s) skipped):%s%s%s%s", h[0], h[1],
              (h[0] & EXTKV_DEV_BAD_WRITE_IDX) ? " write_idx out of range;" : "",
              (h[0] & EXTKV_DEV_BAD_NONPAD) ? " nonpad out of range;" : "",
              (h[0] & EXTKV_DEV_TIMEOUT) ? " pipeline wait timed out;" : "",
              (h[0] & EXTKV_DEV_BOUNDS) ? " access outside a buffer skipped (checked build);" : "");
}

const char* extkv_last_error(void) { return g_error; }

const char* extkv_last_kernel(void) { return g_last_kernel; }

int extkv_last_launches(void) { return g_last_launches; }

int extkv_set_wait_polls(int polls) {
  const int prev = static_cast<int>(g_wait_limit_plus1) - 1;
  g_wait_limit_plus1 = polls < 0 ? 0u : static_cast<uint32_t>(polls) + 1u;
  return prev;
}

struct extkv_step {
  cudaGraphExec_t exec;
};

int extkv_step_begin(void** stream) {
  if (!stream) return fail(EXTKV_ERR_INVALID_ARG, "extkv_step_begin: null stream pointer");
  *stream = nullptr;
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "extkv_step_begin: stream");
  // thread-local mode: other threads' CUDA calls do not touch the capture
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaStreamDestroy(s);
    return cuda_fail(e, "extkv_step_begin: capture");
  }
  *stream = s;
  return EXTKV_OK;
}

int extkv_step_end(void* stream, extkv_step** step) {
  if (!stream || !step) return fail(EXTKV_ERR_INVALID_ARG, "extkv_step_end: null argument");
  *step = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(s, &g);
  cudaStreamDestroy(s);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(e, "extkv_step_end: capture");
  }
  cudaGraphExec_t x = nullptr;
  e = cudaGraphInstantiate(&x, g, 0);
  cudaGraphDestroy(g);  // the instantiated graph does not refer to it
  if (e != cudaSuccess) return cuda_fail(e, "extkv_step_end: instantiate");
  *step = new extkv_step{x};
  return EXTKV_OK;
}

int extkv_step_launch(const extkv_step* step, void* stream) {
  if (!step) return fail(EXTKV_ERR_INVALID_ARG, "extkv_step_launch: null step");
  const cudaError_t e = cudaGraphLaunch(step->exec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? EXTKV_OK : cuda_fail(e, "extkv_step_launch");
}

void extkv_step_free(extkv_step* step) {
  if (!step) return;
  cudaGraphExecDestroy(step->exec);
  delete step;
}

int extkv_set_algo(int algo) {
  if (algo < EXTKV_ALGO_AUTO || algo > EXTKV_ALGO_DECODE_CLUSTER)
    return fail(EXTKV_ERR_INVALID_ARG, "extkv_set_algo: unknown algorithm %d", algo);
  int prev = g_algo;
  g_algo = algo;
  return prev;
}

}  // extern "C"
