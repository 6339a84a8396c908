"""fp64 CPU oracle for biased grouped-query attention over an external static KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  It shares no code
with the CUDA path (``biased_gqa_attention_gb300``) and never imports it.

The arithmetic lives in ``extkv_oracle.c`` (plain C, fp64, one loop per
definition step); this module only compiles it with gcc, loads it with ctypes
and marshals numpy arrays.  Element types are named ``"f32"`` and ``"bf16"``;
bf16 arrays travel as their raw ``uint16`` bit patterns.

Pages followed (see the C file for the step-by-step citations):
  * "Emit bias-aware external-KV (TensorScatter + nonpad_kv_seqlen) attention
    for float-bias decoders" (mobius issue #366) -- bias builder contract.
  * "ONNX Domain Attention (Opset 23/24) CUDA Patterns" -- op order (section 4),
    fully-masked rows (section 6), CPU sentinel (section 8), causal alignment
    with an external cache (section 11).
  * "Skill: Attention Optimization" -- TensorScatter static cache, sliding window.
  * "[GQA] Support KV-shared layers with empty K/V inputs" -- KV-shared layers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "extkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_extkv.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "bf16": 1}
_RAW = {"f32": np.float32, "bf16": np.uint16}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, IEEE semantics: no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB lets the mutation test load a deliberately broken copy
            override = os.environ.get("ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_scatter.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I]
            lib.oracle_scatter.restype = I64
            lib.oracle_bias.argtypes = [P, I, I64, P, P, P, P, P, I64, I64, I64, I]
            lib.oracle_bias.restype = I64
            lib.oracle_bias_from_mask.argtypes = [P, P, I64, I]
            lib.oracle_bias_from_mask.restype = None
            lib.oracle_attention.argtypes = [P, P, P, P, P, P, ctypes.c_float, I64, I64, I64,
                                             I64, I64, I64, I, P, I64]
            lib.oracle_attention.restype = I64
            lib.oracle_attention_softcap.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, I64,
                                                     I64, I64, I64, I64, I64, I, P, I64]
            lib.oracle_attention_softcap.restype = I64
            lib.oracle_attention_dv.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, I64,
                                                I64, I64, I64, I64, I64, I64, I, P, I64]
            lib.oracle_attention_dv.restype = I64
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = I
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's attention uses (rows are split across them)."""
    return int(_load().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _raw(a, dt):
    a = np.asarray(a)
    want = _RAW[dt]
    if a.dtype != want:
        raise TypeError(f"oracle expects {dt} data as {np.dtype(want).name}, got {a.dtype}")
    return np.ascontiguousarray(a)


def dtype_of(a) -> str:
    a = np.asarray(a)
    if a.dtype == np.float32:
        return "f32"
    if a.dtype == np.uint16:
        return "bf16"
    raise TypeError(f"unsupported oracle element type {a.dtype}")


def scatter(k_cache, v_cache, k_new, v_new, write_idx) -> int:
    """TensorScatter along the sequence axis, in place on ``k_cache``/``v_cache``.

    cache (B,Hkv,max_seq,D), new (B,Hkv,S_new,D), write_idx (B,).  Returns the
    number of batches skipped because their rows would leave the cache.
    """
    dt = dtype_of(k_cache)
    for a in (k_cache, v_cache):
        if not (isinstance(a, np.ndarray) and a.flags.c_contiguous):
            raise TypeError("caches must be C-contiguous numpy arrays (updated in place)")
    k_new, v_new = _raw(k_new, dt), _raw(v_new, dt)
    B, Hkv, max_seq, D = k_cache.shape
    S_new = k_new.shape[2]
    w = _c(write_idx, np.int64)
    return int(_load().oracle_scatter(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                      _ptr(w), B, Hkv, S_new, max_seq, D, DTYPES[dt]))


def spans_csr(spans_per_batch):
    """[[(start,len),...] per batch] -> (span_offsets (B+1,), spans (n,2)) int64."""
    offs = [0]
    flat = []
    for lst in spans_per_batch:
        flat.extend(lst)
        offs.append(len(flat))
    return np.asarray(offs, np.int64), np.asarray(flat, np.int64).reshape(-1, 2)


def bias(nonpad, S_q, max_seq, dt, causal=True, window=0, spans=None, extra=None, q_start=None):
    """The (B,1,S_q,max_seq) static-cache bias in type ``dt`` (raw bits).

    ``spans`` is a list (one entry per batch) of (start, len) image spans.
    Batches with an out-of-range nonpad are left filled with zero bits and
    counted in the second return value.
    """
    np_ = _c(nonpad, np.int64)
    B = np_.shape[0]
    out = np.zeros((B, 1, S_q, max_seq), _RAW[dt])
    so, sp = (None, None) if spans is None else spans_csr(spans)
    ex = None if extra is None else _raw(extra, dt)
    qs = _c(q_start, np.int64)
    bad = _load().oracle_bias(_ptr(out), int(bool(causal)), int(window), _ptr(so), _ptr(sp),
                              _ptr(ex), _ptr(qs), _ptr(np_), B, S_q, max_seq, DTYPES[dt])
    return out, int(bad)


def bias_from_mask(mask, dt):
    """The additive bias of a boolean (B,1,S_q,max_seq) mask in type ``dt``
    (raw bits): 0 where the mask is true, lowest(dt) where it is false."""
    m = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
    out = np.zeros(m.shape, _RAW[dt])
    _load().oracle_bias_from_mask(_ptr(out), _ptr(m), int(m.size), DTYPES[dt])
    return out


def attention(q, k_cache, v_cache, bias_, nonpad, scale, rows=None, softcap=0.0):
    """fp64 attention output.  q (B,Hq,S_q,Dk), k_cache (B,Hkv,max_seq,Dk),
    v_cache (B,Hkv,max_seq,Dv) (Dv may differ from Dk), ``bias_`` None or
    (B,1,S_q,max_seq), all in one element type.  ``softcap`` > 0 caps the
    scaled scores, cap * tanh(x / cap), before the bias.

    With ``rows`` (flat indices (b*Hq+h)*S_q+i) only those rows are computed
    and the result is (len(rows), Dv); otherwise it is (B,Hq,S_q,Dv).
    """
    dt = dtype_of(q)
    q, k_cache, v_cache = _raw(q, dt), _raw(k_cache, dt), _raw(v_cache, dt)
    b_ = None if bias_ is None else _raw(bias_, dt)
    B, Hq, S_q, Dk = q.shape
    Hkv, max_seq = k_cache.shape[1], k_cache.shape[2]
    Dv = v_cache.shape[3]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if k_cache.shape[3] != Dk or v_cache.shape[:3] != k_cache.shape[:3]:
        raise ValueError("cache shapes do not match q")
    np_ = _c(nonpad, np.int64)
    r = _c(rows, np.int64)
    n = B * Hq * S_q if r is None else r.shape[0]
    y = np.zeros((n, Dv), np.float64)
    _load().oracle_attention_dv(_ptr(y), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(b_), _ptr(np_),
                                float(scale), float(softcap), B, Hq, Hkv, S_q, max_seq, Dk, Dv, DTYPES[dt],
                                _ptr(r), n)
    return y.reshape(B, Hq, S_q, Dv) if r is None else y


# --- exact conversions between torch-free numpy arrays and element types ------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen raw bf16 bits exactly to float64."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_f64(a) -> np.ndarray:
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


LOWEST_BITS = {"f32": 0xFF7FFFFF, "bf16": 0xFF7F}
