"""Biased grouped-query attention over an external static KV cache, native to
GB300 (sm_103a).

The compute path lives in ``libextkv.so`` (hand-written CUDA behind the C ABI
of ``include/extkv.h``); :mod:`.extkv` is its thin ctypes binding, and
:mod:`.workloads` draws the seeded synthetic inputs.  Importing the package
does not load the library; the first call does, and fails loudly if it was not
built (``biased_gqa_attention_gb300.build.build()``).
"""
from .extkv import (ALGO_AUTO, ALGO_DECODE, ALGO_GENERIC, ALGO_PREFILL, BiasSpec, ExtKVError,
                    attention_ext_kv, attention_ext_kv_workspace_size, build_static_cache_bias,
                    ext_kv_scatter, extkv_clear_status, extkv_last_error, extkv_last_kernel,
                    extkv_read_status, extkv_set_algo, new_status, new_workspace, use_algo)

__all__ = ["ALGO_AUTO", "ALGO_DECODE", "ALGO_GENERIC", "ALGO_PREFILL", "BiasSpec", "ExtKVError",
           "attention_ext_kv", "attention_ext_kv_workspace_size", "build_static_cache_bias",
           "ext_kv_scatter", "extkv_clear_status", "extkv_last_error", "extkv_last_kernel",
           "extkv_read_status", "extkv_set_algo", "new_status", "new_workspace", "use_algo"]
