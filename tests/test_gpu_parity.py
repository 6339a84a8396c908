"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bars: the scatter and the bias are bit-exact; attention outputs are within
max-abs 1e-5 (fp32) or 1.5e-2 (bf16, fp32 accumulation) of the oracle.
Small workloads (same structure, sizes the oracle finishes in seconds, several
tiles plus ragged tails) are compared element by element; the full-size
workloads on sampled rows, in the launch configuration the bench times.
"""
import numpy as np
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu, sample_rows
from helpers import raw

pytestmark = pytest.mark.gpu

SMALL = [wl.small(w) for w in (wl.C2, wl.C3, wl.C4, wl.C5)] + [wl.C1_PREFILL]
FULL = [wl.C2, wl.C3, wl.C4, wl.C5]
ALGOS = {"auto": ek.ALGO_AUTO, "generic": ek.ALGO_GENERIC}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()
    torch.cuda.init()


def _bits_equal(t: torch.Tensor, a: np.ndarray) -> bool:
    return raw(t).tobytes() == a.tobytes()


@pytest.mark.parametrize("w", SMALL + FULL, ids=lambda w: w.name)
def test_scatter_and_bias_bit_exact(w):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias", algo=ek.ALGO_GENERIC)
    o = oracle_path(inp, rows=np.zeros(0, np.int64))
    assert _bits_equal(g["k"], o["k"]) and _bits_equal(g["v"], o["v"])
    assert _bits_equal(g["bias"], o["bias"])


@pytest.mark.parametrize("algo", list(ALGOS), ids=str)
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_attention_small_elementwise(w, mode, algo):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ALGOS[algo])
    o = oracle_path(inp, mode=mode)
    err = max_err(g["y"], o["y"])
    assert err <= TOL[w.dtype], (err, g["kernel"])


@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_attention_full_size_sampled_rows(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode)
    rows = sample_rows(w, 256 if w.S_q > 1 else 512)
    o = oracle_path(inp, rows=rows, mode=mode)
    err = max_err(g["y"], o["y"], rows)
    assert err <= TOL[w.dtype], (err, g["kernel"])


def test_c1_prefill_then_decode_fp32():
    """The tiny fp32 case: prefill 16 tokens at slots 0-15, then decode one
    token at slot 16 on the cache the prefill left behind."""
    pre, dec = wl.c1_chain("cuda")
    g1 = run_gpu(pre, mode="bias")
    o1 = oracle_path(pre, mode="bias")
    assert _bits_equal(g1["k"], o1["k"]) and _bits_equal(g1["bias"], o1["bias"])
    assert max_err(g1["y"], o1["y"]) <= 1e-5
    g2 = run_gpu(dec, mode="bias", k_cache=g1["k"], v_cache=g1["v"])
    o2 = oracle_path(dec, mode="bias", k_cache=o1["k"], v_cache=o1["v"])
    assert _bits_equal(g2["k"], o2["k"]) and _bits_equal(g2["bias"], o2["bias"])
    assert max_err(g2["y"], o2["y"]) <= 1e-5
