"""Thin ctypes binding over libextkv (include/extkv.h).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the path runs in the library's kernels.  There is
no fallback: if libextkv.so is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libextkv.so")

EXTKV_F32, EXTKV_BF16 = 0, 1
EXTKV_OK, EXTKV_ERR_INVALID_ARG, EXTKV_ERR_UNSUPPORTED, EXTKV_ERR_CUDA, EXTKV_ERR_DEVICE = 0, -1, -2, -3, -4
EXTKV_DEV_BAD_WRITE_IDX, EXTKV_DEV_BAD_NONPAD, EXTKV_DEV_TIMEOUT, EXTKV_DEV_BOUNDS = 0x1, 0x2, 0x4, 0x8
ALGO_AUTO, ALGO_GENERIC, ALGO_DECODE, ALGO_PREFILL, ALGO_PREFILL_PAIR = 0, 1, 2, 3, 4
ALGO_DECODE_STREAMK, ALGO_DECODE_CLUSTER = 5, 6

# Every symbol include/extkv.h declares.
SYMBOLS = ("ext_kv_scatter", "build_static_cache_bias", "attention_ext_kv_workspace_size",
           "attention_ext_kv", "attention_ext_kv_scatter", "attention_ext_kv_softcap",
           "build_bias_from_bool_mask", "attention_ext_kv_dv", "attention_ext_kv_workspace_size_dv",
           "extkv_clear_status", "extkv_read_status",
           "extkv_last_error", "extkv_last_kernel", "extkv_last_launches", "extkv_set_algo",
           "extkv_set_wait_polls",
           "attention_ext_kv_noalloc",
           "extkv_step_begin", "extkv_step_end", "extkv_step_launch", "extkv_step_free")


class ExtKVError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"extkv error {code}: {message}")
        self.code = code


class _BiasSpec(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int32), ("window", ctypes.c_int32),
                ("span_offsets", ctypes.c_void_p), ("spans", ctypes.c_void_p),
                ("extra", ctypes.c_void_p), ("q_start", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libextkv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with biased_gqa_attention_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I64, I, I32P = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.ext_kv_scatter.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I, I32P, P]
    lib.build_static_cache_bias.argtypes = [P, ctypes.POINTER(_BiasSpec), P, I64, I64, I64, I, I32P, P]
    lib.build_bias_from_bool_mask.argtypes = [P, P, I64, I64, I64, I, P]
    lib.attention_ext_kv_softcap.argtypes = [P, P, P, P, P, ctypes.POINTER(_BiasSpec), P, ctypes.c_float,
                                             ctypes.c_float, I64, I64, I64, I64, I64, I64, I, P, ctypes.c_size_t,
                                             I32P, P]
    lib.attention_ext_kv_workspace_size.argtypes = [I64, I64, I64, I64, I64, I64, I]
    lib.attention_ext_kv_workspace_size.restype = ctypes.c_size_t
    lib.attention_ext_kv_workspace_size_dv.argtypes = [I64, I64, I64, I64, I64, I64, I64, I]
    lib.attention_ext_kv_workspace_size_dv.restype = ctypes.c_size_t
    lib.attention_ext_kv_dv.argtypes = [P, P, P, P, P, ctypes.POINTER(_BiasSpec), P, ctypes.c_float,
                                        ctypes.c_float, I64, I64, I64, I64, I64, I64, I64, I, P, ctypes.c_size_t,
                                        I32P, P]
    lib.attention_ext_kv.argtypes = [P, P, P, P, P, ctypes.POINTER(_BiasSpec), P, ctypes.c_float,
                                     I64, I64, I64, I64, I64, I64, I, P, ctypes.c_size_t, I32P, P]
    lib.attention_ext_kv_scatter.argtypes = [P, P, P, P, P, P, P, I64, P, ctypes.POINTER(_BiasSpec), P,
                                             ctypes.c_float, I64, I64, I64, I64, I64, I64, I, P,
                                             ctypes.c_size_t, I32P, P]
    lib.attention_ext_kv_noalloc.argtypes = [P, P, P, P, P, ctypes.POINTER(_BiasSpec), P,
                                             ctypes.c_float, I64, I64, I64, I64, I64, I64, I, I32P, P]
    lib.extkv_clear_status.argtypes = [I32P, P]
    lib.extkv_read_status.argtypes = [I32P, P]
    lib.extkv_last_error.restype = ctypes.c_char_p
    lib.extkv_last_kernel.restype = ctypes.c_char_p
    lib.extkv_last_launches.restype = ctypes.c_int
    lib.extkv_set_algo.argtypes = [I]
    lib.extkv_set_wait_polls.argtypes = [I]
    lib.extkv_set_wait_polls.restype = I
    lib.extkv_step_begin.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    lib.extkv_step_begin.restype = I
    lib.extkv_step_end.argtypes = [P, ctypes.POINTER(ctypes.c_void_p)]
    lib.extkv_step_end.restype = I
    lib.extkv_step_launch.argtypes = [P, P]
    lib.extkv_step_launch.restype = I
    lib.extkv_step_free.argtypes = [P]
    lib.extkv_step_free.restype = None
    for name in ("ext_kv_scatter", "build_static_cache_bias", "attention_ext_kv", "attention_ext_kv_noalloc",
                 "extkv_clear_status", "extkv_read_status", "extkv_set_algo"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return EXTKV_F32
    if t.dtype == torch.bfloat16:
        return EXTKV_BF16
    raise TypeError(f"unsupported element type {t.dtype}")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int):
    if code != EXTKV_OK:
        raise ExtKVError(code, load().extkv_last_error().decode())


class PreparedCall:
    """One library call with its arguments marshalled once (pointers, sizes,
    the bias specification, the stream): calling it issues the same C call
    again, without the per-call checks and conversions of the Python layer.
    For a step repeated over the same buffers; the tensors it was prepared
    with must stay alive and in place, and their contents may change between
    calls."""

    __slots__ = ("_fn", "_args", "_keep")

    def __init__(self, fn, args, keep=()):
        self._fn = fn
        # ctypes instances of the declared argument types: the call converts nothing
        self._args = tuple(a if a is None or isinstance(a, ctypes._SimpleCData) or type(a).__name__ == "CArgObject"
                           else t(a) for a, t in zip(args, fn.argtypes))
        self._keep = keep  # the objects the pointers refer to (bias specification, workspace, tensors)

    def __call__(self):
        code = self._fn(*self._args)
        if code != EXTKV_OK:
            raise ExtKVError(code, load().extkv_last_error().decode())


def _need(t, name, dims=None, dtype=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


@dataclass
class BiasSpec:
    """extkv_bias_spec: causal + sliding window + image spans + padding, with an
    optional dense extra term; tensors live on the device."""
    causal: bool = True
    window: int = 0
    span_offsets: Optional[torch.Tensor] = None  # (B+1,) int64
    spans: Optional[torch.Tensor] = None         # (n,2) int64
    extra: Optional[torch.Tensor] = None         # (B,1,S_q,max_seq)
    q_start: Optional[torch.Tensor] = None       # (B,) int64

    def _c(self) -> _BiasSpec:
        for t, n in ((self.span_offsets, "span_offsets"), (self.spans, "spans"),
                     (self.q_start, "q_start")):
            _need(t, n, dtype=torch.int64)
        _need(self.extra, "extra", dims=4)
        return _BiasSpec(int(bool(self.causal)), int(self.window), _p(self.span_offsets),
                         _p(self.spans), _p(self.extra), _p(self.q_start))


def ext_kv_scatter(k_cache, v_cache, k_new, v_new, write_idx, status=None, stream=None):
    """TensorScatter of (B,Hkv,S_new,D) rows into the (B,Hkv,max_seq,D) caches at write_idx."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, dims=4, dtype=k_cache.dtype)
    _need(write_idx, "write_idx", dims=1, dtype=torch.int64)
    B, Hkv, max_seq, D = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != v_new.shape or k_new.shape[:2] != (B, Hkv) \
            or k_new.shape[3] != D:
        raise ValueError("inconsistent cache / update shapes")
    _check(load().ext_kv_scatter(_p(k_cache), _p(v_cache), _p(k_new), _p(v_new), _p(write_idx), B,
                                 Hkv, k_new.shape[2], max_seq, D, _dt(k_cache), _p(status),
                                 _stream(stream)))


def _marshal_bias(bias, spec: BiasSpec, nonpad, status, stream):
    _need(bias, "bias", dims=4)
    _need(nonpad, "nonpad", dims=1, dtype=torch.int64)
    B, one, S_q, max_seq = bias.shape
    if one != 1:
        raise ValueError("bias must be (B,1,S_q,max_seq)")
    c = spec._c()
    lib = load()
    return lib.build_static_cache_bias, (_p(bias), ctypes.byref(c), _p(nonpad), B, S_q, max_seq, _dt(bias),
                                         _p(status), _stream(stream)), (c, bias, nonpad, status)


def build_static_cache_bias(bias, spec: BiasSpec, nonpad, status=None, stream=None):
    """Materialise the (B,1,S_q,max_seq) bias of ``spec`` into ``bias``."""
    fn, args, _ = _marshal_bias(bias, spec, nonpad, status, stream)
    _check(fn(*args))


def prepare_build_static_cache_bias(bias, spec: BiasSpec, nonpad, status=None, stream=None) -> PreparedCall:
    """build_static_cache_bias with its arguments marshalled once (PreparedCall)."""
    return PreparedCall(*_marshal_bias(bias, spec, nonpad, status, stream))


def attention_ext_kv_workspace_size(B, Hq, Hkv, S_q, max_seq, D, dtype, Dv=None) -> int:
    """Bytes of device workspace attention_ext_kv needs (queries the current device);
    ``Dv``: the value head size when it differs from D."""
    dt = EXTKV_F32 if dtype == torch.float32 else EXTKV_BF16
    if Dv is None or Dv == D:
        return int(load().attention_ext_kv_workspace_size(B, Hq, Hkv, S_q, max_seq, D, dt))
    return int(load().attention_ext_kv_workspace_size_dv(B, Hq, Hkv, S_q, max_seq, D, Dv, dt))


def new_workspace(q: torch.Tensor, k_cache: torch.Tensor, v_cache: Optional[torch.Tensor] = None
                  ) -> Optional[torch.Tensor]:
    """A workspace sized for attention over these q / cache shapes (None if none is needed)."""
    B, Hq, S_q, D = q.shape
    Dv = D if v_cache is None else v_cache.shape[3]
    n = attention_ext_kv_workspace_size(B, Hq, k_cache.shape[1], S_q, k_cache.shape[2], D, q.dtype, Dv)
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def _marshal_attention(y, q, k_cache, v_cache, nonpad, scale, bias, fused, workspace, status, stream, softcap):
    for t, n in ((y, "y"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, dims=4, dtype=q.dtype)
    _need(bias, "bias", dims=4, dtype=q.dtype)
    _need(nonpad, "nonpad", dims=1, dtype=torch.int64)
    B, Hq, S_q, D = q.shape
    Hkv, max_seq = k_cache.shape[1], k_cache.shape[2]
    Dv = v_cache.shape[3]
    if y.shape != (B, Hq, S_q, Dv) or v_cache.shape[:3] != k_cache.shape[:3] or k_cache.shape[0] != B or \
            k_cache.shape[3] != D:
        raise ValueError("inconsistent q / y / cache shapes")
    c = None if fused is None else fused._c()
    if workspace is None:
        need = attention_ext_kv_workspace_size(B, Hq, Hkv, S_q, max_seq, D, q.dtype, Dv)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load()
    keep = (c, workspace, y, q, k_cache, v_cache, bias, nonpad, status)
    args = (_p(y), _p(q), _p(k_cache), _p(v_cache), _p(bias), None if c is None else ctypes.byref(c), _p(nonpad),
            float(scale))
    if Dv != D:
        return lib.attention_ext_kv_dv, (*args, float(softcap), B, Hq, Hkv, S_q, max_seq, D, Dv, _dt(q),
                                         _p(workspace), ws, _p(status), _stream(stream)), keep
    tail = (B, Hq, Hkv, S_q, max_seq, D, _dt(q), _p(workspace), ws, _p(status), _stream(stream))
    if softcap:
        return lib.attention_ext_kv_softcap, (*args, float(softcap), *tail), keep
    return lib.attention_ext_kv, (*args, *tail), keep


def attention_ext_kv(y, q, k_cache, v_cache, nonpad, scale, bias=None, fused: Optional[BiasSpec] = None,
                     workspace=None, status=None, stream=None, softcap: float = 0.0):
    """Y = softmax(cap(scale*QK^T) + bias)V over the external cache; writes ``y`` (B,Hq,S_q,Dv).
    ``softcap`` > 0 caps the scaled scores to softcap*tanh(x/softcap) before the
    bias (attention_ext_kv_softcap); 0 is plain attention_ext_kv.  A v_cache
    whose head size Dv differs from q's and k_cache's Dk goes through
    attention_ext_kv_dv.

    ``workspace`` (uint8 device tensor of attention_ext_kv_workspace_size bytes)
    is allocated here when not given."""
    fn, args, _ = _marshal_attention(y, q, k_cache, v_cache, nonpad, scale, bias, fused, workspace, status,
                                     stream, softcap)
    _check(fn(*args))


def prepare_attention_ext_kv(y, q, k_cache, v_cache, nonpad, scale, bias=None, fused: Optional[BiasSpec] = None,
                             workspace=None, status=None, stream=None, softcap: float = 0.0) -> PreparedCall:
    """attention_ext_kv with its arguments marshalled once (PreparedCall); the
    workspace, when not given, is allocated here and kept by the call."""
    return PreparedCall(*_marshal_attention(y, q, k_cache, v_cache, nonpad, scale, bias, fused, workspace,
                                            status, stream, softcap))


def build_bias_from_bool_mask(bias, mask, stream=None):
    """Writes the additive bias of a boolean (B,1,S_q,max_seq) mask into ``bias``
    (same shape, float32 or bfloat16): 0 where the mask is true, the element
    type's lowest finite value where it is false."""
    _need(bias, "bias", dims=4)
    _need(mask, "mask", dims=4, dtype=torch.bool)
    if mask.shape != bias.shape or bias.shape[1] != 1:
        raise ValueError("mask and bias must both be (B,1,S_q,max_seq)")
    B, _, S_q, max_seq = bias.shape
    _check(load().build_bias_from_bool_mask(_p(bias), _p(mask), B, S_q, max_seq, _dt(bias), _stream(stream)))


def _marshal_attention_scatter(y, q, k_cache, v_cache, k_new, v_new, write_idx, nonpad, scale, bias, fused,
                               workspace, status, stream):
    for t, n in ((y, "y"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"),
                 (v_new, "v_new")):
        _need(t, n, dims=4, dtype=q.dtype)
    _need(bias, "bias", dims=4, dtype=q.dtype)
    _need(nonpad, "nonpad", dims=1, dtype=torch.int64)
    _need(write_idx, "write_idx", dims=1, dtype=torch.int64)
    B, Hq, S_q, D = q.shape
    Hkv, max_seq = k_cache.shape[1], k_cache.shape[2]
    S_new = k_new.shape[2]
    if y.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or \
            k_cache.shape[3] != D or k_new.shape != v_new.shape or k_new.shape[:2] != (B, Hkv) or \
            k_new.shape[3] != D or write_idx.shape[0] != B:
        raise ValueError("inconsistent q / y / cache / new-row shapes")
    c = None if fused is None else fused._c()
    if workspace is None:
        need = load().attention_ext_kv_workspace_size(B, Hq, Hkv, S_q, max_seq, D, _dt(q))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    keep = (c, workspace, y, q, k_cache, v_cache, k_new, v_new, write_idx, bias, nonpad, status)
    return load().attention_ext_kv_scatter, (_p(y), _p(q), _p(k_cache), _p(v_cache), _p(k_new), _p(v_new),
                                             _p(write_idx), S_new, _p(bias),
                                             None if c is None else ctypes.byref(c), _p(nonpad), float(scale),
                                             B, Hq, Hkv, S_q, max_seq, D, _dt(q), _p(workspace), ws,
                                             _p(status), _stream(stream)), keep


def attention_ext_kv_scatter(y, q, k_cache, v_cache, k_new, v_new, write_idx, nonpad, scale, bias=None,
                             fused: Optional[BiasSpec] = None, workspace=None, status=None, stream=None):
    """ext_kv_scatter of (k_new, v_new) at write_idx, then attention_ext_kv over
    the updated caches, in one call (fused into the decode kernel where it runs)."""
    fn, args, _ = _marshal_attention_scatter(y, q, k_cache, v_cache, k_new, v_new, write_idx, nonpad, scale,
                                             bias, fused, workspace, status, stream)
    _check(fn(*args))


def prepare_attention_ext_kv_scatter(y, q, k_cache, v_cache, k_new, v_new, write_idx, nonpad, scale, bias=None,
                                     fused: Optional[BiasSpec] = None, workspace=None, status=None,
                                     stream=None) -> PreparedCall:
    """attention_ext_kv_scatter with its arguments marshalled once (PreparedCall)."""
    return PreparedCall(*_marshal_attention_scatter(y, q, k_cache, v_cache, k_new, v_new, write_idx, nonpad,
                                                    scale, bias, fused, workspace, status, stream))


def attention_ext_kv_noalloc(y, q, k_cache, v_cache, nonpad, scale, bias=None,
                             fused: Optional[BiasSpec] = None, status=None, stream=None):
    """attention_ext_kv without a workspace, for callers that cannot allocate
    device memory (for instance an operator that is handed only its input and
    output buffers).  Decode shapes only; the scratch is a static 8 MiB array
    inside the library, shared by every call on the device, so calls that may
    overlap on the GPU must not use it concurrently."""
    for t, n in ((y, "y"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, dims=4, dtype=q.dtype)
    _need(bias, "bias", dims=4, dtype=q.dtype)
    _need(nonpad, "nonpad", dims=1, dtype=torch.int64)
    B, Hq, S_q, D = q.shape
    Hkv, max_seq = k_cache.shape[1], k_cache.shape[2]
    if y.shape != q.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or \
            k_cache.shape[3] != D:
        raise ValueError("inconsistent q / y / cache shapes")
    c = None if fused is None else fused._c()
    _check(load().attention_ext_kv_noalloc(_p(y), _p(q), _p(k_cache), _p(v_cache), _p(bias),
                                           None if c is None else ctypes.byref(c), _p(nonpad),
                                           float(scale), B, Hq, Hkv, S_q, max_seq, D, _dt(q),
                                           _p(status), _stream(stream)))


def new_status(device="cuda") -> torch.Tensor:
    """A zeroed 16-byte device status word."""
    return torch.zeros(4, dtype=torch.int32, device=device)


def extkv_clear_status(status, stream=None):
    _check(load().extkv_clear_status(_p(status), _stream(stream)))


def extkv_read_status(status, stream=None) -> int:
    """Synchronises; returns EXTKV_OK or EXTKV_ERR_DEVICE (message in extkv_last_error)."""
    code = load().extkv_read_status(_p(status), _stream(stream))
    if code not in (EXTKV_OK, EXTKV_ERR_DEVICE):
        _check(code)
    return code


def extkv_last_error() -> str:
    return load().extkv_last_error().decode()


def extkv_last_kernel() -> str:
    return load().extkv_last_kernel().decode()


def extkv_last_launches() -> int:
    """Kernels the calling thread's last attention_ext_kv launched."""
    return int(load().extkv_last_launches())


def extkv_set_algo(algo: int) -> int:
    prev = load().extkv_set_algo(int(algo))
    if prev < 0:
        _check(prev)
    return prev


def extkv_set_wait_polls(polls: int) -> int:
    """Poll limit of the kernels' pipeline waits for this thread (0: give up
    at once; negative: the kernels' own limit); returns the previous setting.
    For failure-detection tests."""
    return int(load().extkv_set_wait_polls(int(polls)))


class wait_polls:
    """Context manager setting the pipeline-wait poll limit for the calling thread."""

    def __init__(self, polls: int):
        self.polls = polls

    def __enter__(self):
        self.prev = extkv_set_wait_polls(self.polls)
        return self

    def __exit__(self, *exc):
        extkv_set_wait_polls(self.prev)


class use_algo:
    """Context manager forcing one attention kernel for the calling thread."""

    def __init__(self, algo: int):
        self.algo = algo

    def __enter__(self):
        self.prev = extkv_set_algo(self.algo)
        return self

    def __exit__(self, *exc):
        extkv_set_algo(self.prev)


class RecordedStep:
    """A step recorded with StepRecorder: calling it starts every recorded
    library call again with one launch, on ``stream`` (a torch stream or a raw
    handle; default the current stream)."""

    __slots__ = ("_h",)

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)

    def __call__(self, stream=None):
        code = load().extkv_step_launch(self._h, _stream(stream))
        if code != EXTKV_OK:
            raise ExtKVError(code, load().extkv_last_error().decode())

    def __del__(self):
        if _lib is not None and self._h:
            _lib.extkv_step_free(self._h)
            self._h = ctypes.c_void_p()


class StepRecorder:
    """Records the library calls issued with ``stream=rec.stream`` inside the
    block into ``rec.step`` (extkv_step_begin / extkv_step_end).  Issue each
    call once before recording it, and call nothing that synchronises inside."""

    def __enter__(self):
        h = ctypes.c_void_p()
        _check(load().extkv_step_begin(ctypes.byref(h)))
        self.stream = h.value
        self.step = None
        return self

    def __exit__(self, exc_type, exc, tb):
        out = ctypes.c_void_p()
        code = load().extkv_step_end(ctypes.c_void_p(self.stream), ctypes.byref(out))
        if exc_type is not None:
            if out.value:
                load().extkv_step_free(out)
            return False
        _check(code)
        self.step = RecordedStep(out.value)
        return False
