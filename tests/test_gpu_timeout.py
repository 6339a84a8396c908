"""Failure detection on the GPU without a fault: pipeline waits that run out.

Every barrier wait in the attention kernels is bounded; when one runs out
the kernel flags EXTKV_DEV_TIMEOUT in the status word, waits at the full
limit for its own copies still in flight, frees its tensor memory and
returns, so the context stays usable ("ONNX Domain Attention (Opset 23/24)
CUDA Patterns", section 5: a failure never passes silently).  These tests
make the waits run out by setting the poll limit of the pipeline waits to
zero for one call (extkv_set_wait_polls), check that the call is reported
through the status word, and that the next normal call on the same stream
matches the oracle.  Nothing here faults, traps or hangs the GPU.
"""
import numpy as np
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu, spec_of

# two decode shapes on each decode kernel, two single-SM prefill shapes (with key splits) and the
# prefill on CTA pairs, on a shape large enough for the prefill on CTA pairs (head size 256, group of 2)
PAIR_SHAPE = wl.Workload("timeout_pair", 322, B=2, Hq=8, Hkv=4, D=256, S_q=700, max_seq=2048,
                         dtype=torch.bfloat16, causal=True, window=500, nonpad_fixed=1900)
CASES = [
    (ek.ALGO_DECODE_STREAMK, wl.small(wl.C2), "bias"),
    (ek.ALGO_DECODE_STREAMK, wl.small(wl.C4), "fused"),
    (ek.ALGO_DECODE_CLUSTER, wl.small(wl.C2), "bias"),
    (ek.ALGO_DECODE_CLUSTER, wl.small(wl.C4), "fused"),
    (ek.ALGO_PREFILL, wl.small(wl.C5), "bias"),
    (ek.ALGO_PREFILL, wl.small(wl.C3), "fused"),
    (ek.ALGO_PREFILL_PAIR, PAIR_SHAPE, "bias"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("algo,w,mode", CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_waits_that_run_out_are_reported_and_the_next_call_is_exact(algo, w, mode):
    inp = wl.make_inputs(w, "cuda")
    # the caches and the bias the normal call uses, prepared on the device
    ref = run_gpu(inp, mode=mode, algo=algo)
    bias = ref["bias"] if mode == "bias" else None
    fused = spec_of(inp) if mode == "fused" else None
    y_bad = torch.empty_like(ref["y"])
    st = ek.new_status()
    with ek.use_algo(algo), ek.wait_polls(0):
        ek.attention_ext_kv(y_bad, inp.q, ref["k"], ref["v"], inp.nonpad, w.scale, bias=bias, fused=fused,
                            status=st)
        assert ek.extkv_last_kernel().startswith("attn_decode" if algo in (ek.ALGO_DECODE_STREAMK, ek.ALGO_DECODE_CLUSTER) else "attn_prefill")
    assert ek.extkv_read_status(st) == ek.EXTKV_ERR_DEVICE
    assert "timed out" in ek.extkv_last_error()
    flags = int(st[0].item())
    assert flags & ek.EXTKV_DEV_TIMEOUT

    # the same stream, a normal limit again: exact against the oracle
    y = torch.empty_like(ref["y"])
    st2 = ek.new_status()
    with ek.use_algo(algo):
        ek.attention_ext_kv(y, inp.q, ref["k"], ref["v"], inp.nonpad, w.scale, bias=bias, fused=fused, status=st2)
    assert ek.extkv_read_status(st2) == ek.EXTKV_OK, ek.extkv_last_error()
    o = oracle_path(inp, mode=mode)
    assert max_err(y, o["y"]) <= TOL[w.dtype]
    assert torch.equal(y, ref["y"])  # the same kernel on the same inputs: the same bits


def test_wait_limit_setting_is_per_thread_and_restores():
    """Host logic of the setter: negative restores the default; the previous
    value comes back; another thread keeps its own setting."""
    import threading
    prev = ek.extkv_set_wait_polls(5)
    try:
        assert ek.extkv_set_wait_polls(0) == 5
        seen = []
        t = threading.Thread(target=lambda: seen.append(ek.extkv_set_wait_polls(-1)))
        t.start()
        t.join()
        assert seen == [-1]  # a fresh thread starts at the default
        assert ek.extkv_set_wait_polls(-7) == 0
        assert ek.extkv_set_wait_polls(-1) == -1
    finally:
        ek.extkv_set_wait_polls(prev)
    with ek.wait_polls(3):
        assert ek.extkv_set_wait_polls(3) == 3
    assert ek.extkv_set_wait_polls(-1) == -1
