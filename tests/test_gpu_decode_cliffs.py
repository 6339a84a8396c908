"""Decode steps at the edges of the decode kernel's shapes.  Its per-batch
tables and its slice's work list live in shared memory, sized per call: 512
batches (more than the default 256) run on the decode kernel with larger
tables, and 16 query heads per KV head as two row groups of 8; more than 1024
batches, or more than 64 query rows per KV head, are refused on the host, and
the automatic choice runs them on the tcgen05 prefill kernel with packed
query rows.  Checked against the
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

DEC = "attn_decode_streamk_mma"
PACKED = "attn_prefill_tcgen05_packed"
# more batches than the decode kernel's largest tables
B1100 = wl.Workload("decode_b1100_hq4_hkv2_d128", 340, B=1100, Hq=4, Hkv=2, D=128, S_q=1, max_seq=256,
                    dtype=torch.bfloat16, causal=True, window=100, nonpad_range=(1, 256))
# more query rows per KV head than its row groups hold (32 heads x 4 positions)
G32S4 = wl.Workload("decode_g32_s4_d64", 341, B=2, Hq=32, Hkv=1, D=64, S_q=4, max_seq=256,
                    dtype=torch.bfloat16, causal=True, window=0, nonpad_range=(10, 256))
# 512 batches: stream-K (more units than clusters fit); 16 heads per KV head: one of
# the decode kernels (two row groups of 8 per KV head), chosen by the call's bounds
KERNEL = {wl.DECODE_B512.name: DEC, wl.DECODE_G16.name: "attn_decode", B1100.name: PACKED, G32S4.name: PACKED}


@pytest.mark.gpu
@pytest.mark.parametrize("w", [B1100, G32S4], ids=lambda w: w.name)
def test_the_decode_kernel_refuses_the_shape(w):
    inp = wl.make_inputs(w, "cuda")
    y = torch.empty_like(inp.q)
    with ek.use_algo(ek.ALGO_DECODE), pytest.raises(ek.ExtKVError) as e:
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale,
                            fused=ek.BiasSpec(causal=True, window=w.window))
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [wl.small(wl.DECODE_B512), wl.small(wl.DECODE_G16), B1100, G32S4],
                         ids=lambda w: w.name)
def test_small_edge_shapes_match_the_oracle(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode)
    assert g["kernel"].startswith(KERNEL[w.name.replace("_small", "")]), g["kernel"]
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("w", wl.CLIFFS, ids=lambda w: w.name)
def test_full_size_edge_shapes_on_sampled_rows(w):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias")
    assert g["kernel"].startswith(KERNEL[w.name]), g["kernel"]
    rows = sample_rows(w, 512)
    o = oracle_path(inp, rows=rows, mode="bias")
    assert max_err(g["y"], o["y"], rows=rows) <= TOL[w.dtype]
