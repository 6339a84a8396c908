"""Decode steps outside the decode kernel's shapes: more than 256 batches (its
batch tables) and more than 8 query rows per KV head (its rows per unit, the
N of its mma).  The decode kernel refuses them on the host; the automatic
choice runs them on the tcgen05 prefill kernel, checked here against the
oracle ("ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 1: the
GQA map of query heads onto KV heads; section 6: masking), small in both bias
modes and at full size on sampled rows.  bench.py reports their speed beside
the decode workloads.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu, sample_rows


@pytest.mark.gpu
@pytest.mark.parametrize("w", wl.CLIFFS, ids=lambda w: w.name)
def test_the_decode_kernel_refuses_the_shape(w):
    inp = wl.make_inputs(wl.small(w), "cuda")
    y = torch.empty_like(inp.q)
    with ek.use_algo(ek.ALGO_DECODE), pytest.raises(ek.ExtKVError) as e:
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale,
                            fused=ek.BiasSpec(causal=True, window=w.window))
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", wl.CLIFFS, ids=lambda w: w.name)
def test_small_cliff_shapes_match_the_oracle(w, mode):
    inp = wl.make_inputs(wl.small(w), "cuda")
    g = run_gpu(inp, mode=mode)
    assert g["kernel"].startswith("attn_prefill")
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("w", wl.CLIFFS, ids=lambda w: w.name)
def test_full_size_cliff_shapes_on_sampled_rows(w):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias")
    rows = sample_rows(w, 512)
    o = oracle_path(inp, rows=rows, mode="bias")
    assert max_err(g["y"], o["y"], rows=rows) <= TOL[w.dtype]
