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


@pytest.mark.parametrize("S_q", [1, 2])
def test_decode_bias_mask_only_and_valued_batches(S_q):
    """Decode with a materialised bias whose batches differ: mask-only rows
    (0 and the sentinel) and rows carrying other values (finite, a very
    negative finite value that stays unmasked, a NaN that masks, a -0.0 that
    adds nothing).  The bias is built by the oracle and edited on the host."""
    from helpers import from_raw
    import oracle
    w = wl.Workload("dec_mixed_bias", 209, B=5, Hq=8, Hkv=4, D=128, S_q=S_q, max_seq=1024,
                    dtype=torch.bfloat16, causal=True, window=300, nonpad_range=(200, 1024))
    inp = wl.make_inputs(w, "cuda")
    nonpad = raw(inp.nonpad)
    bias, bad = oracle.bias(nonpad, w.S_q, w.max_seq, "bf16", causal=True, window=w.window)
    assert bad == 0
    b16 = bias.copy()
    lowest = 0xFF7F
    rng = np.random.default_rng(9)
    live1 = np.nonzero(b16[1, 0, 0] != lowest)[0]
    vals = (rng.standard_normal(live1.size) * 2).astype(np.float32).view(np.uint32)
    b16[1, 0, 0, live1] = ((vals + 0x7FFF + ((vals >> 16) & 1)) >> 16).astype(np.uint16)  # valued row
    live2 = np.nonzero(b16[2, 0, -1] != lowest)[0]
    b16[2, 0, -1, live2[len(live2) // 2]] = 0x7FC1      # NaN: masked
    live3 = np.nonzero(b16[3, 0, -1] != lowest)[0]
    b16[3, 0, -1, live3[0]] = 0x8000                    # -0.0
    b16[4, 0, 0, live1[-1] if live1[-1] < nonpad[4] else 0] = 0xFF70  # about -3.2e38, not masked
    bias_t = from_raw(b16, torch.bfloat16).cuda()
    y = torch.empty_like(inp.q)
    ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, bias=bias_t)
    assert ek.extkv_last_kernel().startswith("attn_decode")
    ref = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache), b16, nonpad, np.float32(w.scale))
    assert max_err(y, ref) <= TOL[w.dtype]
