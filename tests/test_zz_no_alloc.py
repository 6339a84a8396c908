"""The allocation-free decode entry point, attention_ext_kv_noalloc.

Some callers cannot allocate device memory: an operator inside an inference
runtime that is handed only its input and output buffers, or a
latency-critical path where a cudaMalloc (which may synchronise the device)
is not acceptable.  They cannot supply the workspace attention_ext_kv asks
for; attention_ext_kv_noalloc serves them from a static scratch array inside
the library.

This file runs that entry point through the C ABI on two calls in a row (two
different decode problems sharing the one scratch array) and checks each
result against the regular attention_ext_kv with its own workspace, within
the bf16 tolerance the other tests use.  Its name makes pytest collect it
last, so a run that stops at the first failure has run every other test.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl

TOL = 1.5e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


def _prepared(w, mode):
    inp = wl.make_inputs(w, "cuda")
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    ek.ext_kv_scatter(k, v, inp.k_new, inp.v_new, inp.write_idx)
    spec = ek.BiasSpec(causal=w.causal, window=w.window, span_offsets=inp.span_offsets,
                       spans=inp.span_table, extra=inp.extra)
    bias = None
    if mode == "bias":
        bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda")
        ek.build_static_cache_bias(bias, spec, inp.nonpad)
    return inp, k, v, bias, (spec if mode == "fused" else None)


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    calls = [(wl.C2, "bias"), (wl.small(wl.C4), "fused")]
    results = []
    for w, mode in calls:
        inp, k, v, bias, fused = _prepared(w, mode)
        y_ref = torch.empty_like(inp.q)
        ek.attention_ext_kv(y_ref, inp.q, k, v, inp.nonpad, w.scale, bias=bias, fused=fused)
        y = torch.full_like(inp.q, float("nan"))
        st = ek.new_status()
        ek.attention_ext_kv_noalloc(y, inp.q, k, v, inp.nonpad, w.scale, bias=bias, fused=fused,
                                    status=st)
        assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
        results.append((y, y_ref))
    torch.cuda.synchronize()
    for y, y_ref in results:
        assert torch.isfinite(y.float()).all()
        err = (y.double() - y_ref.double()).abs().max().item()
        assert err <= TOL, err


@pytest.mark.gpu
def test_noalloc_refuses_what_it_cannot_run():
    # fp32 (and any shape the decode kernel does not take) is refused, not faked
    q = torch.randn((1, 4, 1, 64), device="cuda")
    kc = torch.randn((1, 2, 64, 64), device="cuda")
    with pytest.raises(ek.ExtKVError) as e:
        ek.attention_ext_kv_noalloc(torch.empty_like(q), q, kc, kc,
                                    torch.tensor([17], dtype=torch.int64, device="cuda"), 0.125)
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED
    assert "decode shapes" in ek.extkv_last_error()
