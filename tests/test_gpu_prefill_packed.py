"""The prefill kernel with packed query rows: when all positions of a query
fit one tile (S_q <= 128) and a KV head serves several query heads, a tile
holds the rows (head, position) of the group's heads one after the other, so
each KV tile is read once for the group ("ONNX Domain Attention (Opset 23/24)
CUDA Patterns", section 1: query heads share their KV head).  Rows of one tile
then belong to several heads and a head's rows may straddle two tiles; the
bias and the fused specification are looked up by position.  Checked against
the oracle element by element, in every bias mode, with a softcap, with key
splits (small grids) and without, at head sizes 64, 128 and 256.  Rows are
packed only where that takes fewer tiles than one per query head.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu

W = [
    # group 8, 3 positions: 24 rows, one tile; few CTAs, so keys are split
    wl.Workload("packed_g8_s3", 330, B=2, Hq=16, Hkv=2, D=128, S_q=3, max_seq=1536, dtype=torch.bfloat16,
                causal=True, window=700, nonpad_range=(300, 1536)),
    # group 32, 5 positions: 160 rows, the second tile partial; head size 64
    wl.Workload("packed_g32_s5", 331, B=3, Hq=32, Hkv=1, D=64, S_q=5, max_seq=1024, dtype=torch.bfloat16,
                causal=True, window=0, nonpad_range=(10, 1024)),
    # group 4, 50 positions: 200 rows in 2 tiles (4 unpacked), the third head straddling them;
    # spans and an extra term
    wl.Workload("packed_g4_s50", 332, B=2, Hq=8, Hkv=2, D=256, S_q=50, max_seq=1200, dtype=torch.bfloat16,
                causal=True, window=300, nonpad_fixed=1100, n_spans=2, span_len=20, span_start_range=(1040, 1080),
                extra=True),
    # group 16 decode step on many batches (no key splits)
    wl.Workload("packed_g16_s1", 333, B=80, Hq=32, Hkv=2, D=128, S_q=1, max_seq=768, dtype=torch.bfloat16,
                causal=True, window=256, nonpad_range=(1, 768)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", W, ids=lambda w: w.name)
def test_packed_rows_match_the_oracle(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL)
    assert g["kernel"] == "attn_prefill_tcgen05_packed"
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("w", W[:2], ids=lambda w: w.name)
def test_packed_rows_with_a_softcap(w):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias", algo=ek.ALGO_PREFILL, softcap=15.0)
    o = oracle_path(inp, mode="bias", softcap=15.0)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
def test_packed_rows_poison_beyond_nonpad_never_reaches_the_output():
    w = W[0]
    clean = run_gpu(wl.make_inputs(w, "cuda"), mode="bias", algo=ek.ALGO_PREFILL)
    dirty = run_gpu(wl.make_inputs(w, "cuda", poison=True), mode="bias", algo=ek.ALGO_PREFILL)
    assert torch.equal(clean["y"], dirty["y"])


@pytest.mark.gpu
def test_rows_are_not_packed_where_it_saves_no_tile():
    """128 positions of a group of 2 (one tile per head either way) keep the
    unpacked tiles."""
    w = wl.small(wl.C5).replace(S_q=128, max_seq=1400)
    g = run_gpu(wl.make_inputs(w, "cuda"), mode="bias", algo=ek.ALGO_PREFILL)
    assert g["kernel"] == "attn_prefill_tcgen05"
