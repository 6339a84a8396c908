"""The prefill kernel on CTA pairs (head size 256, an even number of query
heads per KV head): the two query heads of a pair run as one M = 256
tcgen05 MMA over two SMs ("ONNX Domain Attention (Opset 23/24) CUDA
Patterns", section 1: query heads share their KV head).  Checked element by
element against the oracle in every bias mode and with a softcap, against the
single-SM kernel on the same inputs, and for the guard cases: poisoned cache
slots beyond nonpad never reach the output, an empty batch gives exact zero
rows.  The shapes are large enough that the grid is not split over keys (the
pair kernel's condition), with a ragged last query tile.  The kernel runs only
when asked for (EXTKV_ALGO_PREFILL_PAIR); the default prefill is one CTA per
query tile.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu

PAIR = "attn_prefill_tcgen05_pair"
ONE = "attn_prefill_tcgen05"

# group of 2, causal + window + two image spans, 700 rows (5 full query tiles and 60)
P1 = wl.Workload("pair_g2_spans", 320, B=2, Hq=8, Hkv=4, D=256, S_q=700, max_seq=2048, dtype=torch.bfloat16,
                 causal=True, window=500, nonpad_fixed=1900, n_spans=2, span_len=100,
                 span_start_range=(1250, 1750))
# group of 4, causal only, a dense extra term, 640 rows
P2 = wl.Workload("pair_g4_extra", 321, B=1, Hq=16, Hkv=4, D=256, S_q=640, max_seq=1536, dtype=torch.bfloat16,
                 causal=True, window=0, nonpad_fixed=1400, extra=True)


@pytest.mark.gpu
@pytest.mark.parametrize("cap", [0.0, 20.0])
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", [P1, P2], ids=lambda w: w.name)
def test_pair_kernel_matches_the_oracle(w, mode, cap):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL_PAIR, softcap=cap)
    assert g["kernel"] == PAIR
    o = oracle_path(inp, mode=mode, softcap=cap)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [P1, P2], ids=lambda w: w.name)
def test_pair_and_single_sm_kernels_agree(w, mode):
    inp = wl.make_inputs(w, "cuda")
    a = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL_PAIR)
    b = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL)
    assert a["kernel"] == PAIR and b["kernel"] == ONE
    d = (a["y"].double() - b["y"].double()).abs().max().item()
    assert d <= TOL[w.dtype], d


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_pair_poison_beyond_nonpad_never_reaches_the_output(mode):
    clean = run_gpu(wl.make_inputs(P1, "cuda"), mode=mode, algo=ek.ALGO_PREFILL_PAIR)
    poisoned = run_gpu(wl.make_inputs(P1, "cuda", poison=True), mode=mode, algo=ek.ALGO_PREFILL_PAIR)
    assert clean["kernel"] == PAIR and poisoned["kernel"] == PAIR
    assert torch.equal(clean["y"], poisoned["y"])


@pytest.mark.gpu
def test_pair_empty_batch_gives_exact_zero_rows():
    inp = wl.make_inputs(P1, "cuda")
    inp.nonpad[1] = 0  # batch 1 has no valid slot
    g = run_gpu(inp, mode="fused", algo=ek.ALGO_PREFILL_PAIR, scatter=False)
    assert g["kernel"] == PAIR
    assert (g["y"][1] == 0).all()
    o = oracle_path(inp, mode="fused", scatter=False)
    assert max_err(g["y"], o["y"]) <= TOL[P1.dtype]
