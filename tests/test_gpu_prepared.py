"""Prepared calls (extkv.prepare_*) issue the same library call as the eager
functions: bit for bit the same outputs, also after the inputs change in
place between calls (the call keeps pointers, not values)."""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import spec_of


@pytest.mark.gpu
@pytest.mark.parametrize("w,mode", [(wl.small(wl.C2), "bias"), (wl.small(wl.C3), "fused"),
                                    (wl.small(wl.C5), "bias")], ids=["decode_bias", "prefill_fused", "splits_bias"])
def test_prepared_calls_match_the_eager_calls(w, mode):
    inp = wl.make_inputs(w, "cuda")
    spec = spec_of(inp)
    st = ek.new_status()

    def buffers():
        return dict(k=inp.k_cache.clone(), v=inp.v_cache.clone(), y=torch.empty_like(inp.q),
                    bias=torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda"))

    eager, prep = buffers(), buffers()
    q = inp.q.clone()
    ws = ek.new_workspace(q, inp.k_cache)
    ws2 = ek.new_workspace(q, inp.k_cache)
    calls = []
    if mode == "bias":
        calls.append(ek.prepare_build_static_cache_bias(prep["bias"], spec, inp.nonpad, status=st))
    calls.append(ek.prepare_attention_ext_kv_scatter(
        prep["y"], q, prep["k"], prep["v"], inp.k_new, inp.v_new, inp.write_idx, inp.nonpad, w.scale,
        bias=prep["bias"] if mode == "bias" else None, fused=spec if mode == "fused" else None,
        workspace=ws2, status=st))
    for step in range(2):
        if step == 1:
            q.mul_(0.5)  # new query values in place: the prepared call sees them
            eager["k"].copy_(inp.k_cache)
            eager["v"].copy_(inp.v_cache)
            prep["k"].copy_(inp.k_cache)
            prep["v"].copy_(inp.v_cache)
        if mode == "bias":
            ek.build_static_cache_bias(eager["bias"], spec, inp.nonpad, status=st)
        ek.attention_ext_kv_scatter(eager["y"], q, eager["k"], eager["v"], inp.k_new, inp.v_new, inp.write_idx,
                                    inp.nonpad, w.scale, bias=eager["bias"] if mode == "bias" else None,
                                    fused=spec if mode == "fused" else None, workspace=ws, status=st)
        for c in calls:
            c()
        torch.cuda.synchronize()
        assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
        assert torch.equal(prep["y"], eager["y"]), step
        assert torch.equal(prep["k"], eager["k"]) and torch.equal(prep["v"], eager["v"])
