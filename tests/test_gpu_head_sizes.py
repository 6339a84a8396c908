"""GPU parity of the head-size variants against the fp64 oracle.

* Query-key head size 512 on the tensor-core prefill kernel: the value
  columns are split over two CTAs (256 each), with and without key splits
  (small grids), in every bias mode, with a softcap, with an extra term.
* A value head size that differs from the query-key head size (head_size !=
  v_head_size, "Skill: Attention Optimization", "ORT CUDA Attention Kernel
  Dispatch"): every pair of 128, 256 and 512 on the prefill kernel and, for
  decode steps, on the decode kernel (with a softcap: the prefill kernel), and
  the exact SIMT kernel for other head sizes.
Each case checks the kernel that ran by name.
"""
import numpy as np
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu

pytestmark = pytest.mark.gpu

PRE = "attn_prefill_tcgen05"
GEN = "attn_generic_bf16"
DEC = "attn_decode_streamk_mma"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


def _w(name, seed, D, Dv=None, **kw):
    base = dict(B=2, Hq=4, Hkv=2, S_q=200, max_seq=640, dtype=torch.bfloat16, causal=True, window=150,
                nonpad_range=(200, 640))
    base.update(kw)
    return wl.Workload(name, seed, D=D, Dv=Dv, **base)


# (2 batches x 4 heads x 2 column chunks x 2 query tiles = 32 CTAs: key splits)
D512_SPLIT = _w("pf_d512_split", 301, 512)
# 2 x 8 heads x 2 chunks x 3 tiles = 96 CTAs: no key split; ragged query tail
D512_GRID = _w("pf_d512_grid", 302, 512, Hq=8, Hkv=2, S_q=300, max_seq=768, nonpad_range=(300, 768))
D512_SPANS_EXTRA = _w("pf_d512_spans_extra", 303, 512, B=1, Hq=8, Hkv=1, S_q=160, max_seq=1024, window=64,
                      nonpad_fixed=900, n_spans=2, span_len=40, span_start_range=(740, 860), extra=True,
                      nonpad_range=None)


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", [D512_SPLIT, D512_GRID, D512_SPANS_EXTRA], ids=lambda w: w.name)
def test_prefill_head_size_512(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL)
    assert g["kernel"].startswith(PRE)
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


def test_prefill_head_size_512_is_the_automatic_choice():
    inp = wl.make_inputs(D512_GRID, "cuda")
    assert run_gpu(inp, mode="bias")["kernel"].startswith(PRE)


@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_prefill_head_size_512_softcap(mode):
    inp = wl.make_inputs(D512_SPLIT, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL, softcap=2.0)
    assert g["kernel"].startswith(PRE)
    o = oracle_path(inp, mode=mode, softcap=2.0)
    assert max_err(g["y"], o["y"]) <= TOL[torch.bfloat16]


def test_prefill_head_size_512_poison_never_reaches_the_output():
    """NaN in every cache slot at or beyond nonpad (both 256-column chunks
    zero the V rows of dead keys before P V)."""
    inp = wl.make_inputs(D512_SPLIT, "cuda", poison=True)
    for mode in ("bias", "fused"):
        g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL, scatter=False)
        o = oracle_path(inp, mode=mode, scatter=False)
        assert max_err(g["y"], o["y"]) <= TOL[torch.bfloat16]


PAIRS = [(128, 256), (256, 128), (512, 128), (512, 256), (128, 512), (256, 512)]


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("dk,dv", PAIRS, ids=lambda x: str(x))
def test_prefill_value_head_size_differs(dk, dv, mode):
    w = _w(f"pf_dk{dk}_dv{dv}", 310 + dk // 64 + dv // 32, dk, dv, Hq=8, Hkv=2, S_q=150,
           nonpad_range=(150, 640))
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL, scatter=False)
    assert g["kernel"].startswith(PRE)
    assert g["y"].shape[-1] == dv
    o = oracle_path(inp, mode=mode, scatter=False)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("dk,dv", [(128, 256), (512, 128)], ids=lambda x: str(x))
def test_prefill_value_head_size_differs_key_splits_and_extra(dk, dv):
    # 1 batch x 4 heads x 1 tile: a small grid, so the key ranges are split
    w = _w(f"pf_dk{dk}_dv{dv}_split", 330 + dk // 64 + dv // 32, dk, dv, B=1, Hq=4, Hkv=1, S_q=100,
           max_seq=1024, window=600, nonpad_range=(700, 1024), extra=True)
    inp = wl.make_inputs(w, "cuda")
    for mode in ("bias", "fused"):
        g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL, scatter=False)
        assert g["kernel"].startswith(PRE)
        o = oracle_path(inp, mode=mode, scatter=False)
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("dk,dv,S_q,kernel", [(64, 128, 40, GEN), (96, 200, 7, GEN), (64, 128, 1, GEN)],
                         ids=lambda x: str(x))
def test_value_head_size_differs_other_shapes(dk, dv, S_q, kernel):
    """Head sizes outside the kernels' pairs run on the exact SIMT kernel."""
    w = _w(f"gen_dk{dk}_dv{dv}", 340 + dk // 32 + dv // 8, dk, dv, S_q=S_q, max_seq=520,
           nonpad_range=(max(S_q, 50), 520))
    inp = wl.make_inputs(w, "cuda")
    for mode in ("bias", "fused"):
        g = run_gpu(inp, mode=mode, scatter=False)
        assert g["kernel"] == kernel
        o = oracle_path(inp, mode=mode, scatter=False)
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


def test_value_head_size_binding_checks_shapes():
    w = _w("dv_shapes", 350, 128, 256, S_q=16, max_seq=128, nonpad_range=(16, 128))
    inp = wl.make_inputs(w, "cuda")
    y_bad = torch.empty_like(inp.q)  # Dk columns instead of Dv
    with pytest.raises(ValueError):
        ek.attention_ext_kv(y_bad, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale)


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("dk,dv", PAIRS, ids=lambda x: str(x))
def test_decode_value_head_size_differs(dk, dv, mode):
    """A decode step (one query row per head, group of 4) on the decode kernel,
    K of Dk and V of Dv columns, ragged nonpad."""
    w = _w(f"dec_dk{dk}_dv{dv}", 360 + dk // 64 + dv // 32, dk, dv, B=5, Hq=8, Hkv=2, S_q=1, max_seq=1024,
           window=300, nonpad_range=(1, 1024))
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, scatter=False)
    assert g["kernel"] == DEC
    assert g["y"].shape[-1] == dv
    o = oracle_path(inp, mode=mode, scatter=False)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("dk,dv", [(256, 512), (512, 128)], ids=lambda x: str(x))
def test_decode_value_head_size_differs_two_rows_spans_extra_and_poison(dk, dv):
    """Two query rows per head (S_q = 2), image spans and an extra term in the
    fused spec, and NaN in every slot at or beyond nonpad."""
    w = _w(f"dec2_dk{dk}_dv{dv}", 370 + dk // 64 + dv // 32, dk, dv, B=3, Hq=8, Hkv=2, S_q=2, max_seq=768,
           window=200, nonpad_fixed=600, nonpad_range=None, n_spans=1, span_len=40,
           span_start_range=(500, 540), extra=True)
    inp = wl.make_inputs(w, "cuda", poison=True)
    for mode in ("bias", "fused"):
        g = run_gpu(inp, mode=mode, scatter=False)
        assert g["kernel"] == DEC
        o = oracle_path(inp, mode=mode, scatter=False)
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


def test_decode_value_head_size_differs_with_softcap_runs_on_the_prefill_kernel():
    w = _w("dec_cap_dk256_dv128", 380, 256, 128, B=3, Hq=8, Hkv=2, S_q=1, max_seq=512, nonpad_range=(50, 512))
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias", scatter=False, softcap=3.0)
    assert g["kernel"].startswith(PRE)
    o = oracle_path(inp, mode="bias", scatter=False, softcap=3.0)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]
