"""Recorded steps (extkv_step_begin / _end / _launch): the library calls of a
step recorded once and started again with one launch give bit for bit the
outputs of the same calls issued eagerly, also after the inputs change in
place between launches (the recording keeps addresses, not values)."""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import spec_of


@pytest.mark.gpu
@pytest.mark.parametrize("w,mode", [(wl.small(wl.C2), "bias"), (wl.small(wl.C3), "fused"),
                                    (wl.small(wl.C5), "bias")], ids=["decode_bias", "prefill_fused", "splits_bias"])
def test_recorded_step_matches_the_eager_calls(w, mode):
    inp = wl.make_inputs(w, "cuda")
    spec = spec_of(inp)
    st = ek.new_status()
    q = inp.q.clone()

    def buffers():
        return dict(k=inp.k_cache.clone(), v=inp.v_cache.clone(), y=torch.empty_like(inp.q),
                    bias=torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda"),
                    ws=ek.new_workspace(q, inp.k_cache))

    eager, rec_b = buffers(), buffers()

    def calls(b, stream=None):
        if mode == "bias":
            ek.build_static_cache_bias(b["bias"], spec, inp.nonpad, status=st, stream=stream)
        ek.attention_ext_kv_scatter(b["y"], q, b["k"], b["v"], inp.k_new, inp.v_new, inp.write_idx, inp.nonpad,
                                    w.scale, bias=b["bias"] if mode == "bias" else None,
                                    fused=spec if mode == "fused" else None, workspace=b["ws"], status=st,
                                    stream=stream)

    calls(rec_b)  # first-use setup outside the recording
    torch.cuda.synchronize()
    with ek.StepRecorder() as rec:
        calls(rec_b, stream=rec.stream)
    step = rec.step
    for n in range(2):
        if n == 1:
            q.mul_(0.5)
        for b in (eager, rec_b):
            b["k"].copy_(inp.k_cache)
            b["v"].copy_(inp.v_cache)
        calls(eager)
        step()
        torch.cuda.synchronize()
        assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
        assert torch.equal(rec_b["y"], eager["y"]), n
        assert torch.equal(rec_b["k"], eager["k"]) and torch.equal(rec_b["v"], eager["v"])
