"""The cluster decode kernel: one thread-block cluster per (batch, KV head),
each CTA streaming an equal share of the unit's live tiles and the shares
combined through distributed shared memory ("Skill: Attention Optimization":
decode is memory-bandwidth bound; "ONNX Domain Attention (Opset 23/24) CUDA
Patterns", section 1: the query heads of a KV group share its K/V rows).

Checked against the oracle element by element with the kernel forced: every
bias mode, head sizes 64-512, two and three query positions, row groups (more
than 8 query rows per KV head), units with fewer live tiles than CTAs, empty
batches, poisoned slots; the decode
workloads at full size on sampled rows; the automatic choice for the decode
workload; bit-for-bit repeatability (the shares are combined in a fixed
order); and the shapes the kernel refuses.
"""
import numpy as np
import pytest
import torch

import oracle
from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu, sample_rows, spec_of
from helpers import from_raw, raw
from test_gpu_invariants import EXTRA_DECODE

pytestmark = pytest.mark.gpu

CL = "attn_decode_cluster"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


SHAPES = [
    # C2's structure, small: group of 2, window, ragged nonpad
    wl.small(wl.C2),
    # units whose live tiles are fewer than the cluster's CTAs (nonpad 1-40:
    # at most 3 tiles for 8 CTAs, so some CTAs have no tile at all)
    wl.Workload("cl_short", 401, B=6, Hq=8, Hkv=4, D=256, S_q=1, max_seq=256, dtype=torch.bfloat16,
                causal=True, window=0, nonpad_range=(1, 40)),
    # head size 128, group of 8 (8 rows per unit), a long window
    wl.Workload("cl_d128_g8", 402, B=3, Hq=16, Hkv=2, D=128, S_q=1, max_seq=2048, dtype=torch.bfloat16,
                causal=True, window=1500, nonpad_range=(600, 2048)),
    # head size 512 with key spans at one position
    wl.Workload("cl_d512_spans", 403, B=2, Hq=8, Hkv=2, D=512, S_q=1, max_seq=1536, dtype=torch.bfloat16,
                causal=True, window=64, nonpad_fixed=1400, n_spans=2, span_len=48,
                span_start_range=(900, 1300)),
    # two query positions per head (4 heads x 2 positions = 8 rows), head size 64
    wl.Workload("cl_d64_sq2", 404, B=4, Hq=8, Hkv=2, D=64, S_q=2, max_seq=4096, dtype=torch.bfloat16,
                causal=True, window=700, nonpad_range=(2, 4096)),
    # 16 heads per KV head: two row groups, each a cluster of its own
    wl.Workload("cl_g16", 409, B=3, Hq=32, Hkv=2, D=128, S_q=1, max_seq=1024, dtype=torch.bfloat16,
                causal=True, window=300, nonpad_range=(1, 1024)),
    # 6 heads x 3 positions = 18 rows: three groups, the last of 2 rows
    wl.Workload("cl_g6_s3", 410, B=2, Hq=12, Hkv=2, D=256, S_q=3, max_seq=512, dtype=torch.bfloat16,
                causal=True, window=100, nonpad_range=(3, 512)),
] + EXTRA_DECODE


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_cluster_decode_matches_the_oracle(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    assert g["kernel"] == CL
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [wl.C2, wl.C4], ids=lambda w: w.name)
def test_cluster_decode_full_size_sampled_rows(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    assert g["kernel"] == CL
    rows = sample_rows(w, 48)
    o = oracle_path(inp, rows=rows, mode=mode)
    assert max_err(g["y"], o["y"], rows=rows) <= TOL[w.dtype]


def test_the_decode_workload_runs_on_the_cluster_kernel():
    inp = wl.make_inputs(wl.C2, "cuda")
    for mode in ("bias", "fused"):
        assert run_gpu(inp, mode=mode)["kernel"] == CL


@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_cluster_decode_is_repeatable_bit_for_bit(mode):
    inp = wl.make_inputs(wl.small(wl.C2), "cuda")
    a = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    b = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    assert torch.equal(a["y"].view(torch.int16), b["y"].view(torch.int16))


@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_cluster_decode_agrees_with_stream_k(mode):
    inp = wl.make_inputs(wl.small(wl.C4), "cuda")
    a = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    b = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_STREAMK)
    assert a["kernel"] == CL and b["kernel"] == "attn_decode_streamk_mma"
    assert (a["y"].float() - b["y"].float()).abs().max().item() <= TOL[torch.bfloat16]


def test_cluster_decode_poison_beyond_nonpad_is_invisible():
    w = wl.small(wl.C2).replace(name="cl_poison")
    clean = wl.make_inputs(w, "cuda")
    poisoned = wl.make_inputs(w, "cuda", poison=True)
    for mode in ("bias", "fused", "none"):
        a = run_gpu(clean, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
        b = run_gpu(poisoned, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
        assert torch.equal(a["y"].view(torch.int16), b["y"].view(torch.int16))


def test_cluster_decode_empty_batches_are_zero_rows():
    w = wl.small(wl.C2).replace(name="cl_empty")
    inp = wl.make_inputs(w, "cuda")
    inp.nonpad[1] = 0
    inp.write_idx[1] = 0
    for mode in ("bias", "fused", "none"):
        g = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER, scatter=False)
        o = oracle_path(inp, mode=mode, scatter=False)
        assert (g["y"][1] == 0).all()
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("w,mode", [
    (wl.Workload("cl_g32_s4", 408, B=2, Hq=32, Hkv=1, D=64, S_q=4, max_seq=256, dtype=torch.bfloat16,
                 causal=True, window=0, nonpad_range=(10, 256)), "bias"),  # 128 rows per KV head
    (wl.small(wl.C2).replace(name="cl_long", max_seq=8200, nonpad_range=(1, 8200)), "bias"),  # scan > 16 KB
    (wl.Workload("cl_sq2_spans", 405, B=2, Hq=4, Hkv=2, D=128, S_q=2, max_seq=512, dtype=torch.bfloat16,
                 causal=True, window=50, nonpad_fixed=500, n_spans=1, span_len=40,
                 span_start_range=(300, 300)), "fused"),              # spans at two positions
], ids=["g32_s4", "long_bias", "sq2_spans"])
def test_the_cluster_kernel_refuses_the_shape(w, mode):
    inp = wl.make_inputs(w, "cuda")
    with pytest.raises(ek.ExtKVError) as e:
        run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED
    # the automatic choice still runs the shape, on another kernel
    g = run_gpu(inp, mode=mode)
    assert g["kernel"] != CL


def test_cluster_decode_two_head_sizes_are_refused():
    w = wl.Workload("cl_dk128_dv256", 406, B=2, Hq=8, Hkv=4, D=128, Dv=256, S_q=1, max_seq=512,
                    dtype=torch.bfloat16, causal=True, window=100, nonpad_range=(1, 512))
    inp = wl.make_inputs(w, "cuda")
    with pytest.raises(ek.ExtKVError) as e:
        run_gpu(inp, mode="bias", algo=ek.ALGO_DECODE_CLUSTER, scatter=False)
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED


def test_cluster_scan_reads_special_bias_values():
    """The live-tile scan against section 6's rule (a key is unmasked iff it is
    below nonpad and its bias is above lowest(T); NaN is not above it): a value
    just above lowest, NaN, -inf and lowest side by side, the only unmasked
    key in a partial last tile, a zero bias beyond nonpad, an empty batch."""
    w = wl.Workload("cl_scan", 407, B=4, Hq=8, Hkv=4, D=128, S_q=1, max_seq=512, dtype=torch.bfloat16,
                    causal=False, window=0, nonpad_fixed=512)
    inp = wl.make_inputs(w, "cuda")
    nonpad = np.array([100, 37, 512, 0], np.int64)
    inp.nonpad = torch.tensor(nonpad, device="cuda")
    low, neg_inf, nan, one, minus_one = 0xFF7F, 0xFF80, 0x7FC0, 0x3F80, 0xBF80
    bias = np.full((4, 1, 1, 512), low, np.uint16)
    bias[0, 0, 0, 5] = 0xFF7E          # the value next above lowest: unmasked
    bias[0, 0, 0, 50] = nan            # masked
    bias[0, 0, 0, 99] = 0              # unmasked, the last key below nonpad
    bias[1, 0, 0, 36] = one            # the only unmasked key, in the partial last tile
    bias[1, 0, 0, 40] = 0              # beyond nonpad: masked whatever its bias
    bias[2, 0, 0, ::2] = neg_inf
    bias[2, 0, 0, 400:416] = nan       # a whole tile of NaN
    bias[2, 0, 0, 300] = minus_one     # the only unmasked key of the batch
    y = torch.full_like(inp.q, float("nan"))
    st = ek.new_status()
    with ek.use_algo(ek.ALGO_DECODE_CLUSTER):
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale,
                            bias=from_raw(bias, w.dtype).cuda(), status=st)
        assert ek.extkv_last_kernel() == CL
    assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
    ref = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache), bias, nonpad, np.float32(w.scale))
    assert (y[3] == 0).all()
    assert max_err(y, ref) <= TOL[w.dtype]


# few units: several clusters per unit, each leaving a partial for the merge kernel
FEW = [
    # one sequence: 8 units
    wl.Workload("cl_b1", 411, B=1, Hq=16, Hkv=8, D=256, S_q=1, max_seq=4096, dtype=torch.bfloat16,
                causal=True, window=0, nonpad_fixed=4000),
    # one sequence, two KV heads with two row groups each (8 heads x 2 positions)
    wl.Workload("cl_b1_rg", 412, B=1, Hq=16, Hkv=2, D=128, S_q=2, max_seq=2048, dtype=torch.bfloat16,
                causal=True, window=600, nonpad_fixed=1900),
    # two sequences at head size 64 with a short one (empty shares)
    wl.Workload("cl_b2_d64", 413, B=2, Hq=8, Hkv=2, D=64, S_q=1, max_seq=1024, dtype=torch.bfloat16,
                causal=True, window=0, nonpad_range=(5, 1024)),
]


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", FEW, ids=lambda w: w.name)
def test_cluster_decode_split_units_match_the_oracle(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)
    assert g["kernel"] == CL
    assert ek.extkv_last_launches() == 2  # the clusters, then the merge of their partials
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_cluster_decode_split_units_with_the_fused_scatter(mode):
    w = FEW[0]
    inp = wl.make_inputs(w, "cuda")
    ref = run_gpu(inp, mode=mode, algo=ek.ALGO_DECODE_CLUSTER)  # separate scatter, then attention
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    y = torch.empty_like(inp.q)
    st = ek.new_status()
    with ek.use_algo(ek.ALGO_DECODE_CLUSTER):
        ek.attention_ext_kv_scatter(y, inp.q, k, v, inp.k_new, inp.v_new, inp.write_idx, inp.nonpad, w.scale,
                                    bias=ref["bias"] if mode == "bias" else None,
                                    fused=spec_of(inp) if mode == "fused" else None, status=st)
        assert ek.extkv_last_kernel() == CL + "_scatter"
    assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
    assert torch.equal(y.view(torch.int16), ref["y"].view(torch.int16))
    assert torch.equal(k.view(torch.int16), ref["k"].view(torch.int16))
    assert torch.equal(v.view(torch.int16), ref["v"].view(torch.int16))


def test_cluster_decode_split_units_timeout_is_reported():
    w = FEW[0]
    inp = wl.make_inputs(w, "cuda")
    ref = run_gpu(inp, mode="bias", algo=ek.ALGO_DECODE_CLUSTER)
    y = torch.empty_like(ref["y"])
    st = ek.new_status()
    with ek.use_algo(ek.ALGO_DECODE_CLUSTER), ek.wait_polls(0):
        ek.attention_ext_kv(y, inp.q, ref["k"], ref["v"], inp.nonpad, w.scale, bias=ref["bias"], status=st)
    assert int(st[0].item()) & ek.EXTKV_DEV_TIMEOUT
    y2 = torch.empty_like(ref["y"])
    st2 = ek.new_status()
    with ek.use_algo(ek.ALGO_DECODE_CLUSTER):
        ek.attention_ext_kv(y2, inp.q, ref["k"], ref["v"], inp.nonpad, w.scale, bias=ref["bias"], status=st2)
    assert ek.extkv_read_status(st2) == ek.EXTKV_OK
    assert torch.equal(y2.view(torch.int16), ref["y"].view(torch.int16))


def test_one_long_sequence_picks_the_split_cluster_kernel():
    w = wl.Workload("cl_b1_long", 414, B=1, Hq=16, Hkv=8, D=256, S_q=1, max_seq=8192, dtype=torch.bfloat16,
                    causal=True, window=0, nonpad_fixed=8000)
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode="bias")
    assert g["kernel"] == CL and ek.extkv_last_launches() == 2
    rows = sample_rows(w, 64)
    o = oracle_path(inp, rows=rows, mode="bias")
    assert max_err(g["y"], o["y"], rows=rows) <= TOL[w.dtype]
