"""The C ABI library loads and exports every symbol include/extkv.h declares,
and rejects bad arguments on the host (CPU only: no call here reaches a
kernel launch)."""
import ctypes
import os
import re

import pytest

from biased_gqa_attention_gb300 import build as B
from biased_gqa_attention_gb300 import extkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "extkv.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return extkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(extkv.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_validation_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: validation fails first
    # Hq not a multiple of Hkv
    rc = lib.attention_ext_kv(fake, fake, fake, fake, None, None, fake, 1.0, 1, 6, 4, 1, 64, 64,
                              extkv.EXTKV_BF16, None, 0, None, None)
    assert rc == extkv.EXTKV_ERR_INVALID_ARG
    assert "multiple of Hkv" in extkv.extkv_last_error()
    # D not supported
    rc = lib.attention_ext_kv(fake, fake, fake, fake, None, None, fake, 1.0, 1, 4, 2, 1, 64, 12,
                              extkv.EXTKV_BF16, None, 0, None, None)
    assert rc == extkv.EXTKV_ERR_UNSUPPORTED
    # both a materialised bias and a fused spec
    spec = extkv._BiasSpec(1, 0, None, None, None, None)
    rc = lib.attention_ext_kv(fake, fake, fake, fake, fake, ctypes.byref(spec), fake, 1.0, 1, 4, 2,
                              1, 64, 64, extkv.EXTKV_BF16, None, 0, None, None)
    assert rc == extkv.EXTKV_ERR_INVALID_ARG
    # misaligned tensors
    odd = P(0x10002)
    rc = lib.attention_ext_kv(odd, fake, fake, fake, None, None, fake, 1.0, 1, 4, 2, 1, 64, 64,
                              extkv.EXTKV_BF16, None, 0, None, None)
    assert rc == extkv.EXTKV_ERR_INVALID_ARG
    # unknown dtype
    rc = lib.ext_kv_scatter(fake, fake, fake, fake, fake, 1, 1, 1, 8, 64, 7, None, None)
    assert rc == extkv.EXTKV_ERR_INVALID_ARG
    # S_new larger than the cache
    rc = lib.ext_kv_scatter(fake, fake, fake, fake, fake, 1, 1, 9, 8, 64, extkv.EXTKV_BF16, None, None)
    assert rc == extkv.EXTKV_ERR_INVALID_ARG
    # bias row stride not a multiple of 16 bytes
    rc = lib.build_static_cache_bias(fake, ctypes.byref(spec), fake, 1, 1, 12, extkv.EXTKV_BF16,
                                     None, None)
    assert rc == extkv.EXTKV_ERR_UNSUPPORTED
    # empty problems are valid no-ops (nothing is launched)
    assert lib.attention_ext_kv(None, None, None, None, None, None, None, 1.0, 0, 4, 2, 1, 64, 64,
                                extkv.EXTKV_BF16, None, 0, None, None) == extkv.EXTKV_OK
    assert lib.ext_kv_scatter(None, None, None, None, None, 2, 2, 0, 64, 64, extkv.EXTKV_BF16, None,
                              None) == extkv.EXTKV_OK
    # algorithm selection: every value the header defines, nothing past the last
    assert lib.extkv_set_algo(99) == extkv.EXTKV_ERR_INVALID_ARG
    assert lib.extkv_set_algo(extkv.ALGO_DECODE_CLUSTER + 1) == extkv.EXTKV_ERR_INVALID_ARG
    assert lib.extkv_set_algo(-1) == extkv.EXTKV_ERR_INVALID_ARG
    prev = lib.extkv_set_algo(extkv.ALGO_GENERIC)
    for algo in (extkv.ALGO_DECODE, extkv.ALGO_PREFILL, extkv.ALGO_PREFILL_PAIR, extkv.ALGO_DECODE_STREAMK,
                 extkv.ALGO_DECODE_CLUSTER, extkv.ALGO_AUTO):
        lib.extkv_set_algo(algo)
    assert lib.extkv_set_algo(prev) == extkv.ALGO_AUTO


def test_workspace_size_is_queryable(lib):
    assert extkv.attention_ext_kv_workspace_size(8, 16, 8, 1, 4096, 256, None) >= 0


def test_host_validation_of_two_head_sizes(lib):
    """attention_ext_kv_dv's own checks, all on the host before any launch."""
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: validation fails first

    def dv_call(dk, dv, softcap=0.0, B=1):
        return lib.attention_ext_kv_dv(fake, fake, fake, fake, None, None, fake, 1.0, softcap, B, 4, 2, 1, 64,
                                       dk, dv, extkv.EXTKV_BF16, None, 0, None, None)

    assert dv_call(128, 12) == extkv.EXTKV_ERR_UNSUPPORTED       # Dv not a multiple of 8
    assert dv_call(128, 520) == extkv.EXTKV_ERR_UNSUPPORTED      # Dv above 512
    assert dv_call(128, 0) == extkv.EXTKV_ERR_UNSUPPORTED
    assert "Dv=" in extkv.extkv_last_error()
    assert dv_call(12, 128) == extkv.EXTKV_ERR_UNSUPPORTED       # Dk not a multiple of 8
    assert dv_call(128, 256, softcap=-1.0) == extkv.EXTKV_ERR_INVALID_ARG
    assert dv_call(128, 256, softcap=float("nan")) == extkv.EXTKV_ERR_INVALID_ARG
    assert dv_call(128, 256, B=0) == extkv.EXTKV_OK               # an empty problem launches nothing


def test_workspace_size_with_two_head_sizes(lib):
    # one head size: the same as the plain query; an empty batch needs nothing
    same = extkv.attention_ext_kv_workspace_size(1, 16, 8, 2048, 8192, 256, None)
    assert extkv.attention_ext_kv_workspace_size(1, 16, 8, 2048, 8192, 256, None, Dv=256) == same
    assert int(lib.attention_ext_kv_workspace_size_dv(0, 16, 8, 2048, 8192, 256, 256, extkv.EXTKV_BF16)) == 0


def test_prepared_calls_marshal_once_and_reissue_the_call(lib):
    """extkv.prepare_*: the arguments are converted once to the declared ctypes
    types, and every call re-issues the C function (its host checks included).
    CPU only: an empty batch launches nothing, an odd head size fails its
    host check before any pointer is used."""
    import torch

    q = torch.zeros((0, 4, 1, 64), dtype=torch.bfloat16)
    kc = torch.zeros((0, 2, 64, 64), dtype=torch.bfloat16)
    nonpad = torch.zeros(0, dtype=torch.int64)
    call = extkv.prepare_attention_ext_kv(torch.empty_like(q), q, kc, kc, nonpad, 0.125, stream=0)
    assert all(a is None or isinstance(a, ctypes._SimpleCData) or type(a).__name__ == "CArgObject"
               for a in call._args)
    call()
    call()
    spec = extkv.BiasSpec(causal=True, window=16)
    bias = torch.zeros((0, 1, 1, 64), dtype=torch.bfloat16)
    extkv.prepare_build_static_cache_bias(bias, spec, nonpad, stream=0)()
    scat = extkv.prepare_attention_ext_kv_scatter(torch.empty_like(q), q, kc, kc, kc[:, :, :1], kc[:, :, :1],
                                                  nonpad, nonpad, 0.125, fused=spec, stream=0)
    scat()
    # a head size that is not a multiple of 8: refused on every call
    q12 = torch.zeros((1, 4, 1, 12), dtype=torch.bfloat16)
    k12 = torch.zeros((1, 2, 64, 12), dtype=torch.bfloat16)
    bad = extkv.prepare_attention_ext_kv(torch.empty_like(q12), q12, k12, k12, torch.ones(1, dtype=torch.int64),
                                         0.125, stream=0)
    for _ in range(2):
        with pytest.raises(extkv.ExtKVError) as e:
            bad()
        assert e.value.code == extkv.EXTKV_ERR_UNSUPPORTED


def test_recorded_step_entry_points_check_their_arguments(lib):
    """extkv_step_*: null arguments are refused on the host (no CUDA call)."""
    P = ctypes.c_void_p
    assert lib.extkv_step_begin(None) == extkv.EXTKV_ERR_INVALID_ARG
    out = ctypes.c_void_p(0x1234)
    assert lib.extkv_step_end(None, ctypes.byref(out)) == extkv.EXTKV_ERR_INVALID_ARG
    assert lib.extkv_step_end(P(0x10000), None) == extkv.EXTKV_ERR_INVALID_ARG
    assert lib.extkv_step_launch(None, None) == extkv.EXTKV_ERR_INVALID_ARG
    assert "null" in extkv.extkv_last_error()
    lib.extkv_step_free(None)  # releasing nothing is a no-op
