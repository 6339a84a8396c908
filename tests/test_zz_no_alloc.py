"""The allocation-free decode entry point, attention_ext_kv_noalloc.

Some callers cannot allocate device memory: an operator inside an inference
runtime that is handed only its input and output buffers, or a
latency-critical path where a cudaMalloc (which may synchronise the device)
is not acceptable.  They cannot supply the workspace attention_ext_kv asks
for; attention_ext_kv_noalloc serves them from a static scratch array inside
the library.

This file runs that entry point through the C ABI on two calls in a row (two
different decode problems sharing the one scratch array) and checks each
result bit for bit against the regular attention_ext_kv with its own
workspace (the same kernels on the same inputs) and against the oracle within
the bf16 tolerance the other tests use.  It also checks what it refuses: an
unknown element type, fp32, and sizes whose scratch would not fit the array
(refused before any launch).  Its name makes pytest collect it last, so a run
that stops at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import max_err, oracle_path

TOL = 1.5e-2
SCRATCH_BYTES = 8 << 20  # EXTKV_NOALLOC_SCRATCH_BYTES in include/extkv.h
# a second decode problem of another head size and group, sharing the scratch
D128 = wl.Workload("noalloc_decode_d128", 310, B=6, Hq=8, Hkv=2, D=128, S_q=1, max_seq=1536,
                   dtype=torch.bfloat16, causal=True, window=500, nonpad_range=(1, 1536))


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
    calls = [(wl.C2, "bias"), (D128, "fused")]
    results = []
    for w, mode in calls:
        inp, k, v, bias, fused = _prepared(w, mode)
        y_ref = torch.empty_like(inp.q)
        ek.attention_ext_kv(y_ref, inp.q, k, v, inp.nonpad, w.scale, bias=bias, fused=fused)
        ref_kernel, ref_launches = ek.extkv_last_kernel(), ek.extkv_last_launches()
        y = torch.full_like(inp.q, float("nan"))
        st = ek.new_status()
        ek.attention_ext_kv_noalloc(y, inp.q, k, v, inp.nonpad, w.scale, bias=bias, fused=fused,
                                    status=st)
        # the same decode kernels ran, and the call says so
        assert ek.extkv_last_kernel() == ref_kernel and ref_kernel.startswith("attn_decode")
        assert ek.extkv_last_launches() == ref_launches >= 1
        assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
        results.append((w, mode, inp, y, y_ref))
    torch.cuda.synchronize()
    for w, mode, inp, y, y_ref in results:
        assert torch.equal(y, y_ref)  # bit for bit: the same kernels on the same inputs
        o = oracle_path(inp, mode=mode)
        assert max_err(y, o["y"]) <= TOL


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
    # an element type the library does not know is an invalid argument
    lib = ek.load()
    qb = q.to(torch.bfloat16)
    kb = kc.to(torch.bfloat16)
    nonpad = torch.tensor([17], dtype=torch.int64, device="cuda")
    code = lib.attention_ext_kv_noalloc(qb.data_ptr(), qb.data_ptr(), kb.data_ptr(), kb.data_ptr(), None, None,
                                        nonpad.data_ptr(), ctypes.c_float(0.125), 1, 4, 2, 1, 64, 64, 7, None,
                                        torch.cuda.current_stream().cuda_stream)
    assert code == ek.EXTKV_ERR_INVALID_ARG
    assert "dtype" in ek.extkv_last_error()


@pytest.mark.gpu
def test_noalloc_refuses_sizes_beyond_its_scratch_before_any_launch():
    """The global-layer decode shape (B=32, Hq=16, Hkv=2, D=512: 8 query rows
    per unit) is one the decode kernel takes, but its scratch (two fp32
    partials of 8 rows x 512 columns per CTA of the full grid, about 10 MB)
    is larger than the static array: refused with EXTKV_ERR_UNSUPPORTED, and
    nothing is launched (the output keeps its contents and the last-kernel
    record still names the previous call)."""
    B, Hq, Hkv, S_q, max_seq, D = 32, 16, 2, 1, 8192, 512
    need = ek.attention_ext_kv_workspace_size(B, Hq, Hkv, S_q, max_seq, D, torch.bfloat16)
    assert need > SCRATCH_BYTES, need
    # a successful small call first, so the last-kernel record has a known value
    w = wl.small(wl.C2)
    inp, k, v, bias, _ = _prepared(w, "bias")
    ek.attention_ext_kv_noalloc(torch.empty_like(inp.q), inp.q, k, v, inp.nonpad, w.scale, bias=bias)
    before = (ek.extkv_last_kernel(), ek.extkv_last_launches())
    # real tensors of the claimed sizes (nothing may be read, but nothing could be out of bounds)
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn((B, Hq, S_q, D), device="cuda", generator=g).to(torch.bfloat16)
    kc = torch.zeros((B, Hkv, max_seq, D), dtype=torch.bfloat16, device="cuda")
    y = torch.full_like(q, float("nan"))
    nonpad = torch.full((B,), max_seq, dtype=torch.int64, device="cuda")
    with pytest.raises(ek.ExtKVError) as e:
        ek.attention_ext_kv_noalloc(y, q, kc, kc, nonpad, D ** -0.5)
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED
    assert "bytes of scratch" in ek.extkv_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(y.float()).all()
    assert (ek.extkv_last_kernel(), ek.extkv_last_launches()) == before
