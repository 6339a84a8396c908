"""The scatter fused into the attention call (attention_ext_kv_scatter).

Where the decode kernel runs, it writes the new rows and takes the tiles that
hold them from k_new / v_new; the result must be the one of the two calls it
replaces ("Skill: Attention Optimization", "In-place KV for ONNX Attention via
TensorScatter (static cache)": the scatter, then the attention over the
updated cache): caches bit for bit equal to ext_kv_scatter's, y bit for bit
equal to attention_ext_kv's over those caches (same kernel, same tile data),
and within the tolerance of the oracle.  Shapes the decode kernel does not take
run the scatter kernel first and must give the same results too.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, spec_of
from test_gpu_invariants import EXTRA_DECODE

pytestmark = pytest.mark.gpu

FUSED = "attn_decode_streamk_mma_scatter"
# the two decode kernels, forced one at a time, with the name each reports
# for the call with the scatter fused
VARIANTS = [(ek.ALGO_DECODE_STREAMK, FUSED), (ek.ALGO_DECODE_CLUSTER, "attn_decode_cluster_scatter")]
VIDS = ["streamk", "cluster"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


def _bias_for(inp, mode):
    w = inp.w
    if mode != "bias":
        return None
    bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda")
    ek.build_static_cache_bias(bias, spec_of(inp), inp.nonpad)
    return bias


def _two_calls(inp, mode, write_idx=None, algo=ek.ALGO_AUTO):
    w = inp.w
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    st = ek.new_status()
    ek.ext_kv_scatter(k, v, inp.k_new, inp.v_new, inp.write_idx if write_idx is None else write_idx, status=st)
    y = torch.empty_like(inp.q)
    bias = _bias_for(inp, mode)
    with ek.use_algo(algo):
        ek.attention_ext_kv(y, inp.q, k, v, inp.nonpad, w.scale, bias=bias,
                            fused=spec_of(inp) if mode == "fused" else None, status=st)
    return k, v, y, st


def _one_call(inp, mode, write_idx=None, algo=ek.ALGO_AUTO):
    w = inp.w
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    st = ek.new_status()
    y = torch.empty_like(inp.q)
    bias = _bias_for(inp, mode)
    with ek.use_algo(algo):
        ek.attention_ext_kv_scatter(y, inp.q, k, v, inp.k_new, inp.v_new,
                                    inp.write_idx if write_idx is None else write_idx, inp.nonpad, w.scale,
                                    bias=bias, fused=spec_of(inp) if mode == "fused" else None, status=st)
        kernel = ek.extkv_last_kernel()
    return k, v, y, st, kernel


DECODE = EXTRA_DECODE + [wl.small(wl.C2), wl.small(wl.C4), wl.C2]


@pytest.mark.parametrize("algo,fused_name", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", DECODE, ids=lambda w: w.name)
def test_fused_scatter_decode_equals_the_two_calls(w, mode, algo, fused_name):
    inp = wl.make_inputs(w, "cuda")
    k1, v1, y1, st1, kernel = _one_call(inp, mode, algo=algo)
    k2, v2, y2, st2 = _two_calls(inp, mode, algo=algo)
    assert kernel == fused_name
    assert ek.extkv_read_status(st1) == ek.EXTKV_OK and ek.extkv_read_status(st2) == ek.EXTKV_OK
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("algo,fused_name", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [EXTRA_DECODE[0], EXTRA_DECODE[3], wl.small(wl.C2)], ids=lambda w: w.name)
def test_fused_scatter_decode_matches_the_oracle(w, mode, algo, fused_name):
    inp = wl.make_inputs(w, "cuda")
    k, v, y, st, kernel = _one_call(inp, mode, algo=algo)
    assert kernel == fused_name and ek.extkv_read_status(st) == ek.EXTKV_OK
    o = oracle_path(inp, mode=mode)
    assert max_err(y, o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [wl.C1_DECODE, wl.small(wl.C5), wl.small(wl.C3)], ids=lambda w: w.name)
def test_fused_scatter_other_paths_run_the_scatter_first(w):
    inp = wl.make_inputs(w, "cuda")
    k1, v1, y1, st1, kernel = _one_call(inp, "bias")
    k2, v2, y2, st2 = _two_calls(inp, "bias")
    assert kernel != FUSED
    assert ek.extkv_read_status(st1) == ek.EXTKV_OK
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(y1, y2)
    o = oracle_path(inp, mode="bias")
    assert max_err(y1, o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("algo,fused_name", VARIANTS, ids=VIDS)
def test_fused_scatter_bad_write_index_is_skipped_and_flagged(algo, fused_name):
    w = wl.small(wl.C2)
    inp = wl.make_inputs(w, "cuda")
    wi = inp.write_idx.clone()
    wi[1] = w.max_seq  # one row past the end
    k1, v1, y1, st1, kernel = _one_call(inp, "bias", write_idx=wi, algo=algo)
    k2, v2, y2, st2 = _two_calls(inp, "bias", write_idx=wi, algo=algo)
    assert kernel == fused_name
    assert ek.extkv_read_status(st1) == ek.EXTKV_ERR_DEVICE and "WRITE_IDX" in ek.extkv_last_error().upper()
    assert torch.equal(k1[1].view(torch.int16), inp.k_cache[1].view(torch.int16))  # batch 1 not written
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("algo,fused_name", VARIANTS, ids=VIDS)
def test_fused_scatter_with_no_new_rows_is_plain_attention(algo, fused_name):
    w = wl.small(wl.C2)
    inp = wl.make_inputs(w, "cuda")
    empty = inp.k_new[:, :, :0].contiguous()
    y1 = torch.empty_like(inp.q)
    k = inp.k_cache.clone()
    with ek.use_algo(algo):
        ek.attention_ext_kv_scatter(y1, inp.q, k, inp.v_cache.clone(), empty, empty, inp.write_idx, inp.nonpad,
                                    w.scale)
        assert ek.extkv_last_kernel() == fused_name[:-len("_scatter")]
        y2 = torch.empty_like(inp.q)
        ek.attention_ext_kv(y2, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(k.view(torch.int16), inp.k_cache.view(torch.int16))


@pytest.mark.parametrize("algo,fused_name", VARIANTS, ids=VIDS)
def test_fused_scatter_writes_the_rows_when_no_tile_is_live(algo, fused_name):
    """nonpad = 0 everywhere: no CTA has a tile, every CTA still writes its
    share of the new rows, and every row of y is zero."""
    w = EXTRA_DECODE[0]
    inp = wl.make_inputs(w, "cuda")
    inp.nonpad = torch.zeros_like(inp.nonpad)
    k1, v1, y1, st1, kernel = _one_call(inp, "none", algo=algo)
    k2, v2, y2, st2 = _two_calls(inp, "none", algo=algo)
    assert kernel == fused_name and ek.extkv_read_status(st1) == ek.EXTKV_OK
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    assert (y1 == 0).all()
