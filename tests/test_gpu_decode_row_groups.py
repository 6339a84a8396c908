"""The decode kernel with more than 8 query rows per KV head: the (Hq/Hkv) *
S_q rows of a KV head form units of up to 8 rows (row groups) that stream the
same K/V tiles ("ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 1:
query heads share their KV head).  A row r of group rg is query row 8 rg + r of
the KV head: head (8 rg + r) / S_q of the group, position (8 rg + r) % S_q, so
the bias and the fused specification's windows are looked up per position.
Checked against the oracle element by element with each decode kernel forced
(stream-K, and the cluster kernel, which gives each row group a cluster):
two groups, a partial second group, eight groups, image spans (the plan with
the fused specification), a softcap, two head sizes; and the scatter fused
into the call bit for bit against the two separate calls.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu, spec_of

DEC = "attn_decode_streamk_mma"
CL = "attn_decode_cluster"
VARIANTS = [(ek.ALGO_DECODE_STREAMK, DEC), (ek.ALGO_DECODE_CLUSTER, CL)]
VIDS = ["streamk", "cluster"]


def cluster_takes(w, mode):
    """The cluster kernel's shapes: one head size; with the fused specification
    no spans at several positions (their live tiles are not in closed form)."""
    return w.dv == w.D and not (mode == "fused" and w.S_q > 1 and w.n_spans > 0)
W = [
    # 16 heads per KV head, one position: two full groups
    wl.Workload("rg_g16_s1", 350, B=5, Hq=32, Hkv=2, D=128, S_q=1, max_seq=1200, dtype=torch.bfloat16,
                causal=True, window=400, nonpad_range=(1, 1200)),
    # 4 heads x 3 positions: 12 rows, the second group partial (rows of one head straddle groups)
    wl.Workload("rg_g4_s3", 351, B=3, Hq=16, Hkv=4, D=256, S_q=3, max_seq=1024, dtype=torch.bfloat16,
                causal=True, window=300, nonpad_range=(3, 1024)),
    # 8 heads x 8 positions: eight groups, the most a KV head takes
    wl.Workload("rg_g8_s8", 352, B=2, Hq=8, Hkv=1, D=64, S_q=8, max_seq=640, dtype=torch.bfloat16,
                causal=True, window=0, nonpad_range=(8, 640)),
    # 2 heads x 5 positions with image spans (the fused specification needs the plan)
    wl.Workload("rg_g2_s5_spans", 353, B=2, Hq=8, Hkv=4, D=128, S_q=5, max_seq=896, dtype=torch.bfloat16,
                causal=True, window=100, nonpad_fixed=800, n_spans=1, span_len=60, span_start_range=(740, 740)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("algo,name", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", W, ids=lambda w: w.name)
def test_row_groups_match_the_oracle(w, mode, algo, name):
    inp = wl.make_inputs(w, "cuda")
    if name == CL and not cluster_takes(w, mode):
        with pytest.raises(ek.ExtKVError) as e:
            run_gpu(inp, mode=mode, algo=algo)
        assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED
        return
    g = run_gpu(inp, mode=mode, algo=algo)
    assert g["kernel"] == name
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("algo,name", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("w", W[:2], ids=lambda w: w.name)
def test_row_groups_with_a_softcap(w, algo, name):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias", algo=algo, softcap=12.0)
    assert g["kernel"] == name
    o = oracle_path(inp, mode="bias", softcap=12.0)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
def test_row_groups_with_two_head_sizes():
    w = wl.Workload("rg_dk128_dv256", 354, B=3, Hq=32, Hkv=2, D=128, Dv=256, S_q=1, max_seq=704,
                    dtype=torch.bfloat16, causal=True, window=250, nonpad_range=(1, 700))
    inp = wl.make_inputs(w, "cuda")
    for mode in ("bias", "fused"):
        g = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE, scatter=False)
        assert g["kernel"] == DEC  # two head sizes: the stream-K kernel
        o = oracle_path(inp, mode=mode, scatter=False)
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("algo,name", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", W[:2], ids=lambda w: w.name)
def test_row_groups_with_the_fused_scatter(w, mode, algo, name):
    inp = wl.make_inputs(w, "cuda")
    ref = run_gpu(inp, mode=mode, algo=algo)  # separate scatter, then attention
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    y = torch.empty_like(inp.q)
    st = ek.new_status()
    with ek.use_algo(algo):
        ek.attention_ext_kv_scatter(y, inp.q, k, v, inp.k_new, inp.v_new, inp.write_idx, inp.nonpad, w.scale,
                                    bias=ref["bias"] if mode == "bias" else None,
                                    fused=spec_of(inp) if mode == "fused" else None, status=st)
        assert ek.extkv_last_kernel() == name + "_scatter"
    assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
    assert torch.equal(y, ref["y"]) and torch.equal(k, ref["k"]) and torch.equal(v, ref["v"])
