// attn_decode_noalloc.cu -- the decode attention with its scratch memory in a
// static device array, for callers that cannot allocate device memory.
//
// Who needs it: code that is handed only its input and output buffers --
// for example a custom operator inside an inference runtime whose operator
// interface offers no scratch allocator, or a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not acceptable.  Such a
// caller cannot provide the workspace attention_ext_kv asks for, so this
// entry point brings its own: a fixed-size array that lives in the library's
// device image.  Every GPU that loads this code holds the array until the
// process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "extkv.h"
#include "internal.h"

namespace extkv {

namespace {

// The scratch: plan tables and the fp32 partial results of units split
// across CTAs.  Shared by every call of attention_ext_kv_noalloc on a device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[EXTKV_NOALLOC_SCRATCH_BYTES];

int fail(int code, const char* msg, size_t a = 0, size_t b = 0) {
  char buf[256];
  snprintf(buf, sizeof buf, msg, a, b);
  set_error(buf);  // read back through extkv_last_error()
  return code;
}

// The calling thread's current CUDA context (the driver entry point, so the
// library needs no link-time dependency on libcuda); nullptr if unavailable.
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of g_noalloc_scratch on the current device (the symbol's
// host-side name is not a device address), looked up once per device and
// context: a device reset builds a new context and a new copy of the array,
// so an address cached for the old context is never reused.
void* scratch_address(cudaError_t* err) {
  struct Entry {
    int dev;
    CUcontext ctx;
    void* addr;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int n = 0;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  const CUcontext ctx0 = current_context();  // nullptr before the runtime made one current
  std::lock_guard<std::mutex> g(mu);
  for (int i = 0; ctx0 && i < n; ++i)
    if (cache[i].dev == dev && cache[i].ctx == ctx0) return cache[i].addr;
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // also makes the primary context current
  if (*err != cudaSuccess) return nullptr;
  const CUcontext ctx = ctx0 ? ctx0 : current_context();
  if (ctx) {
    int slot = -1;
    for (int i = 0; i < n; ++i)
      if (cache[i].dev == dev) slot = i;  // the device's earlier context is gone
    if (slot < 0) slot = n < 64 ? n++ : 63;
    cache[slot] = Entry{dev, ctx, p};
  }
  return p;
}

}  // namespace

}  // namespace extkv

using namespace extkv;

extern "C" int attention_ext_kv_noalloc(void* y, const void* q, const void* k_cache,
                                        const void* v_cache, const void* bias,
                                        const extkv_bias_spec* fused, const int64_t* nonpad,
                                        float scale, int64_t B, int64_t Hq, int64_t Hkv,
                                        int64_t S_q, int64_t max_seq, int64_t D, int dtype,
                                        int32_t* status, void* stream) {
  set_error("");
  if (dtype != EXTKV_F32 && dtype != EXTKV_BF16)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_noalloc: unknown dtype %zu", static_cast<size_t>(dtype));
  if (B < 0 || S_q < 0 || Hq <= 0 || Hkv <= 0 || max_seq <= 0 || D <= 0 || Hq % Hkv)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_noalloc: bad sizes");
  if (bias && fused)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_noalloc: pass either a bias or a fused spec, not both");
  if (B == 0 || S_q == 0) return EXTKV_OK;
  if (!y || !q || !k_cache || !v_cache || !nonpad)
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_noalloc: null pointer");
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(y) || !al16(q) || !al16(k_cache) || !al16(v_cache) || (bias && !al16(bias)) ||
      (fused && fused->extra && !al16(fused->extra)) || (reinterpret_cast<uintptr_t>(nonpad) & 7) ||
      (reinterpret_cast<uintptr_t>(status) & 3))
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_noalloc: tensors must be 16-byte aligned");
  if (fused && ((fused->span_offsets == nullptr) != (fused->spans == nullptr)))
    return fail(EXTKV_ERR_INVALID_ARG, "attention_ext_kv_noalloc: span_offsets and spans must be given together");

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
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.S_q = S_q;
  a.max_seq = max_seq;
  a.D = D;
  a.Dv = D;
  a.dtype = dtype;
  a.status = status;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_limit_plus1 = wait_limit_setting();
  if (!decode_supported(a))
    return fail(EXTKV_ERR_UNSUPPORTED,
                "attention_ext_kv_noalloc: only decode shapes run here (bf16, (Hq/Hkv)*S_q <= 8, "
                "D in {64,128,256,512})");
  const size_t need = decode_workspace_bytes(B, Hq, Hkv, S_q, max_seq, D, D);
  if (need > static_cast<size_t>(EXTKV_NOALLOC_SCRATCH_BYTES))
    return fail(EXTKV_ERR_UNSUPPORTED,
                "attention_ext_kv_noalloc: these sizes need %zu bytes of scratch, more than the "
                "library's static %zu bytes; use attention_ext_kv with a workspace",
                need, static_cast<size_t>(EXTKV_NOALLOC_SCRATCH_BYTES));
  cudaError_t e;
  void* scratch = scratch_address(&e);
  if (!scratch)
    return fail(EXTKV_ERR_CUDA, "attention_ext_kv_noalloc: cudaGetSymbolAddress failed (CUDA error %zu)",
                static_cast<size_t>(e));
  a.workspace = scratch;
  a.ws_bytes = EXTKV_NOALLOC_SCRATCH_BYTES;
  const char* name = "";
  note_launches(0);
  e = launch_attn_decode(a, &name);
  if (e != cudaSuccess)
    return fail(EXTKV_ERR_CUDA, "attention_ext_kv_noalloc: launch failed (CUDA error %zu)", static_cast<size_t>(e));
  note_last_call(name);  // extkv_last_kernel() / extkv_last_launches()
  return EXTKV_OK;
}
