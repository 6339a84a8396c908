"""Softcap on every attention path (attention_ext_kv_softcap).

"ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 4: scale*QK^T,
then softcap*tanh(x/softcap), then + bias / mask (a masked slot stays masked),
then softmax.  Each kernel (decode, tcgen05 prefill, generic) against the fp64
oracle in every bias mode, the pages' guard case (a small cap with poison V
under masked slots), and softcap 0 being plain attention_ext_kv.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu, spec_of
from test_gpu_invariants import EXTRA_DECODE
from test_gpu_prefill import EXTRA_PREFILL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


def _run(inp, mode, cap, algo=ek.ALGO_AUTO, k=None, v=None):
    w = inp.w
    k = inp.k_cache if k is None else k
    v = inp.v_cache if v is None else v
    bias = None
    st = ek.new_status()
    if mode == "bias":
        bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda")
        ek.build_static_cache_bias(bias, spec_of(inp), inp.nonpad, status=st)
    y = torch.empty_like(inp.q)
    with ek.use_algo(algo):
        ek.attention_ext_kv(y, inp.q, k, v, inp.nonpad, w.scale, bias=bias,
                            fused=spec_of(inp) if mode == "fused" else None, status=st, softcap=cap)
        kernel = ek.extkv_last_kernel()
    assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
    return y, kernel


CASES = [
    (EXTRA_DECODE[0], "attn_decode"), (EXTRA_DECODE[3], "attn_decode"),
    (wl.small(wl.C2), "attn_decode"), (wl.small(wl.C4), "attn_decode"),
    (wl.small(wl.C3), "attn_prefill_tcgen05"), (wl.small(wl.C5), "attn_prefill_tcgen05"),
    (EXTRA_PREFILL[0], "attn_prefill_tcgen05"), (EXTRA_PREFILL[2], "attn_prefill_tcgen05"),
    (wl.C1_PREFILL, "attn_generic_f32"), (wl.C1_DECODE, "attn_generic_f32"),
]


@pytest.mark.parametrize("cap", [2.0, 30.0])
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w,kernel", CASES, ids=lambda x: x.name if hasattr(x, "name") else "")
def test_softcap_matches_the_oracle(w, kernel, mode, cap):
    inp = wl.make_inputs(w, "cuda")
    y, ran = _run(inp, mode, cap)
    assert ran.startswith(kernel), ran
    o = oracle_path(inp, mode=mode, scatter=False, softcap=cap)
    assert max_err(y, o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [EXTRA_DECODE[0], wl.small(wl.C3), wl.C1_PREFILL], ids=lambda w: w.name)
def test_tiny_cap_keeps_poison_under_masked_slots_invisible(w):
    """The pages' guard case: with the cap applied before the mask, a masked
    slot's score stays -inf however small the cap; NaN K/V rows at and beyond
    nonpad must not change one bit of the output."""
    clean, _ = _run(wl.make_inputs(w, "cuda"), "bias", 0.05)
    dirty, _ = _run(wl.make_inputs(w, "cuda", poison=True), "bias", 0.05)
    assert torch.equal(clean.view(torch.int16) if clean.dtype == torch.bfloat16 else clean,
                       dirty.view(torch.int16) if dirty.dtype == torch.bfloat16 else dirty)
    assert torch.isfinite(clean.float()).all()


@pytest.mark.parametrize("w", [wl.small(wl.C2), wl.small(wl.C3), wl.C1_DECODE], ids=lambda w: w.name)
def test_softcap_zero_is_plain_attention(w):
    inp = wl.make_inputs(w, "cuda")
    y0, _ = _run(inp, "bias", 0.0)
    g = run_gpu(inp, mode="bias", scatter=False)
    assert torch.equal(y0, g["y"])


def test_invalid_softcap_is_rejected():
    w = wl.small(wl.C2)
    inp = wl.make_inputs(w, "cuda")
    y = torch.empty_like(inp.q)
    for bad in (-1.0, float("inf"), float("nan")):
        with pytest.raises(ek.ExtKVError) as e:
            ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, softcap=bad)
        assert e.value.code == ek.EXTKV_ERR_INVALID_ARG


@pytest.mark.parametrize("algo,kernel", [(ek.ALGO_DECODE_STREAMK, "attn_decode_streamk_mma"),
                                         (ek.ALGO_DECODE_CLUSTER, "attn_decode_cluster")],
                         ids=["streamk", "cluster"])
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [EXTRA_DECODE[0], EXTRA_DECODE[3], wl.small(wl.C2)], ids=lambda w: w.name)
def test_softcap_on_each_decode_kernel(w, mode, algo, kernel):
    inp = wl.make_inputs(w, "cuda")
    y, ran = _run(inp, mode, 5.0, algo=algo)
    assert ran == kernel
    o = oracle_path(inp, mode=mode, scatter=False, softcap=5.0)
    assert max_err(y, o["y"]) <= TOL[w.dtype]
