"""GPU invariants and edge cases, each kernel checked against the oracle.

Invariants the pages state, on the GPU path:
  * poison (NaN) beyond nonpad and huge finite values under bias-masked slots
    leave the output bit-for-bit unchanged ("ONNX Domain Attention (Opset
    23/24) CUDA Patterns", section 6: masked slots never reach the output);
  * a decode step equals the last row of the matching prefill, and a chunked
    prefill equals the one-shot prefill (section 11), within the tolerance;
  * a KV-shared layer ("[GQA] Support KV-shared layers with empty K/V
    inputs", Design) is attention over the borrowed cache with no scatter; an
    empty scatter leaves the cache unchanged.
Edge cases: an empty batch (nonpad = 0), nonpad < S_q (negative offset
clamped), rows with no allowed key, out-of-range nonpad and write indices
(status flags), empty calls, and kernel selection.
"""
import numpy as np
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu
from helpers import raw

pytestmark = pytest.mark.gpu

DEC = "attn_decode_streamk_mma"
# the two decode kernels, forced one at a time, with the name each reports
VARIANTS = [(ek.ALGO_DECODE_STREAMK, DEC), (ek.ALGO_DECODE_CLUSTER, "attn_decode_cluster")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


# decode-kernel shapes beyond the five workloads: other head dims, a query
# group of 4 with two query rows per unit, ragged max_seq, spans
EXTRA_DECODE = [
    wl.Workload("dec_d64_g4_sq2", 101, B=3, Hq=8, Hkv=2, D=64, S_q=2, max_seq=776,
                dtype=torch.bfloat16, causal=True, window=100, nonpad_range=(2, 776)),
    wl.Workload("dec_d128_g8_spans", 102, B=2, Hq=16, Hkv=2, D=128, S_q=1, max_seq=1024,
                dtype=torch.bfloat16, causal=True, window=64, nonpad_fixed=900, n_spans=2,
                span_len=40, span_start_range=(700, 860)),
    wl.Workload("dec_d256_g1_noncausal", 103, B=5, Hq=4, Hkv=4, D=256, S_q=1, max_seq=520,
                dtype=torch.bfloat16, causal=False, window=0, nonpad_range=(1, 520), extra=True),
    wl.Workload("dec_d512_g8_sq1_short", 104, B=6, Hq=8, Hkv=1, D=512, S_q=1, max_seq=64,
                dtype=torch.bfloat16, causal=True, nonpad_range=(1, 64), garbage_sigma=10.0),
]


@pytest.mark.parametrize("algo,kernel", VARIANTS, ids=["streamk", "cluster"])
@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", EXTRA_DECODE + [wl.small(wl.C2), wl.small(wl.C4)], ids=lambda w: w.name)
def test_decode_kernel_forced(w, mode, algo, kernel):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=algo)
    assert g["kernel"] == kernel
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [wl.C2, wl.C4, wl.small(wl.C2), wl.small(wl.C4)], ids=lambda w: w.name)
def test_decode_workloads_pick_the_decode_kernel(w):
    inp = wl.make_inputs(w, "cuda")
    assert run_gpu(inp, mode="bias")["kernel"].startswith("attn_decode")
    assert run_gpu(inp, mode="fused")["kernel"].startswith("attn_decode")


@pytest.mark.parametrize("algo", [ek.ALGO_AUTO, ek.ALGO_GENERIC])
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [wl.C4, wl.small(wl.C2), wl.small(wl.C3), wl.small(wl.C5)],
                         ids=lambda w: w.name)
def test_poison_beyond_nonpad_is_bitwise_invisible(w, mode, algo):
    clean = run_gpu(wl.make_inputs(w, "cuda"), mode=mode, algo=algo)
    dirty = run_gpu(wl.make_inputs(w, "cuda", poison=True), mode=mode, algo=algo)
    assert torch.equal(clean["y"].view(torch.int16), dirty["y"].view(torch.int16))


@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_huge_values_under_masked_bias_are_invisible(mode):
    w = wl.C2
    inp = wl.make_inputs(w, "cuda")
    clean = run_gpu(inp, mode=mode)
    # slots below nonpad - window are masked by the sliding window
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    for b in range(w.B):
        lo = max(int(inp.nonpad[b]) - w.window, 0)
        k[b, :, :lo] = 3.0e38
        v[b, :, :lo] = -3.0e38
    dirty = run_gpu(inp, mode=mode, k_cache=k, v_cache=v)
    assert torch.equal(clean["y"].view(torch.int16), dirty["y"].view(torch.int16))


def _prefill_then(w, n_last):
    """A prefill workload and the inputs of its last n_last rows as a later call."""
    inp = wl.make_inputs(w, "cuda")
    cut = w.replace(S_q=n_last)
    tail = wl.Inputs(cut, inp.q[:, :, -n_last:].contiguous(), inp.k_new[:, :, -n_last:].contiguous(),
                     inp.v_new[:, :, -n_last:].contiguous(), None, None, inp.nonpad - n_last,
                     inp.nonpad, inp.spans, inp.span_offsets, inp.span_table,
                     None if inp.extra is None else inp.extra[:, :, -n_last:].contiguous())
    return inp, tail


@pytest.mark.parametrize("w", [wl.small(wl.C3), wl.small(wl.C5)], ids=lambda w: w.name)
def test_decode_equals_last_prefill_row(w):
    inp, last = _prefill_then(w, 1)
    full = run_gpu(inp, mode="fused")
    # the prefill already wrote every row; decode only attends
    dec = run_gpu(last, mode="fused", scatter=False, k_cache=full["k"], v_cache=full["v"])
    d = (dec["y"].double() - full["y"][:, :, -1:].double()).abs().max().item()
    assert d <= TOL[w.dtype]


@pytest.mark.parametrize("w", [wl.small(wl.C3).replace(name="prefill_small_nospans", n_spans=0),
                               wl.small(wl.C5)], ids=lambda w: w.name)
def test_chunked_prefill_equals_one_shot(w):
    # (image spans are left out: a span crossing the chunk boundary lets the
    # first chunk's rows see tokens the first chunk has not written yet)
    inp = wl.make_inputs(w, "cuda")
    one = run_gpu(inp, mode="bias")
    h = w.S_q // 2
    first = w.replace(S_q=h)
    second = w.replace(S_q=w.S_q - h)
    sl = lambda t, a, b: None if t is None else t[:, :, a:b].contiguous()
    a = wl.Inputs(first, sl(inp.q, 0, h), sl(inp.k_new, 0, h), sl(inp.v_new, 0, h), inp.k_cache,
                  inp.v_cache, inp.write_idx, inp.nonpad - (w.S_q - h), inp.spans,
                  inp.span_offsets, inp.span_table, sl(inp.extra, 0, h))
    ga = run_gpu(a, mode="bias")
    b = wl.Inputs(second, sl(inp.q, h, w.S_q), sl(inp.k_new, h, w.S_q), sl(inp.v_new, h, w.S_q),
                  None, None, inp.write_idx + h, inp.nonpad, inp.spans, inp.span_offsets,
                  inp.span_table, sl(inp.extra, h, w.S_q))
    gb = run_gpu(b, mode="bias", k_cache=ga["k"], v_cache=ga["v"])
    y = torch.cat([ga["y"], gb["y"]], dim=2)
    assert torch.equal(gb["k"].view(torch.int16), one["k"].view(torch.int16))
    assert (y.double() - one["y"].double()).abs().max().item() <= TOL[w.dtype]


def test_kv_shared_layer_reuses_the_borrowed_cache():
    w = wl.C5
    inp = wl.make_inputs(w, "cuda")
    src = run_gpu(inp, mode="bias")
    k0, v0 = src["k"].clone(), src["v"].clone()
    # the KV-shared layer writes no K/V: an empty scatter is a no-op
    empty = torch.empty((w.B, w.Hkv, 0, w.D), dtype=w.dtype, device="cuda")
    ek.ext_kv_scatter(src["k"], src["v"], empty, empty, inp.write_idx)
    assert torch.equal(src["k"].view(torch.int16), k0.view(torch.int16))
    shared = run_gpu(inp, mode="bias", scatter=False, k_cache=src["k"], v_cache=src["v"])
    assert torch.equal(shared["y"].view(torch.int16), src["y"].view(torch.int16))
    rows = np.arange(0, w.B * w.Hq * w.S_q, 37, dtype=np.int64)
    o = oracle_path(inp, rows=rows)
    assert max_err(shared["y"], o["y"], rows) <= TOL[w.dtype]


@pytest.mark.parametrize("algo", [ek.ALGO_AUTO, ek.ALGO_GENERIC])
def test_empty_batch_and_negative_offset(algo):
    w = wl.Workload("edge_sq4", 120, B=3, Hq=4, Hkv=2, D=64, S_q=4, max_seq=64,
                    dtype=torch.bfloat16, causal=True, window=0, nonpad_fixed=8)
    inp = wl.make_inputs(w, "cuda")
    inp.nonpad = torch.tensor([0, 2, 8], dtype=torch.int64, device="cuda")  # empty, 2 < S_q, full
    inp.write_idx = torch.tensor([0, 0, 4], dtype=torch.int64, device="cuda")
    for mode in ("bias", "fused", "none"):
        g = run_gpu(inp, mode=mode, algo=algo)
        o = oracle_path(inp, mode=mode)
        assert (g["y"][0] == 0).all()
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("algo", [ek.ALGO_AUTO, ek.ALGO_GENERIC, ek.ALGO_DECODE_STREAMK, ek.ALGO_DECODE_CLUSTER])
def test_rows_with_no_allowed_key_are_exact_zeros(algo):
    """q_start pushes some rows before slot 0, so causal masking leaves them
    nothing to attend."""
    w = wl.Workload("edge_qstart", 121, B=2, Hq=4, Hkv=2, D=128, S_q=4, max_seq=32,
                    dtype=torch.bfloat16, causal=True, nonpad_fixed=20)
    inp = wl.make_inputs(w, "cuda")
    qs = torch.tensor([-2, 5], dtype=torch.int64, device="cuda")
    spec = ek.BiasSpec(causal=True, window=0, q_start=qs)
    y = torch.empty_like(inp.q)
    with ek.use_algo(algo):
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, fused=spec)
    assert (y[0, :, :2] == 0).all()          # positions -2, -1
    assert (y[0, :, 2:].abs().sum() > 0)
    bias = torch.empty((2, 1, 4, 32), dtype=w.dtype, device="cuda")
    ek.build_static_cache_bias(bias, spec, inp.nonpad)
    y2 = torch.empty_like(inp.q)
    with ek.use_algo(algo):
        ek.attention_ext_kv(y2, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, bias=bias)
    assert torch.equal(y.view(torch.int16)[0, :, :2], y2.view(torch.int16)[0, :, :2])
    assert (y - y2).abs().max().item() <= TOL[w.dtype]


@pytest.mark.parametrize("algo", [ek.ALGO_AUTO, ek.ALGO_GENERIC])
def test_out_of_range_indices_set_status_flags(algo):
    w = wl.small(wl.C2)
    inp = wl.make_inputs(w, "cuda")
    st = ek.new_status()
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    bad_w = inp.write_idx.clone()
    bad_w[1] = w.max_seq  # one past the end
    ek.ext_kv_scatter(k, v, inp.k_new, inp.v_new, bad_w, status=st)
    assert ek.extkv_read_status(st) == ek.EXTKV_ERR_DEVICE
    assert "write_idx" in ek.extkv_last_error()
    assert torch.equal(k[1].view(torch.int16), inp.k_cache[1].view(torch.int16))  # skipped
    ek.extkv_clear_status(st)
    assert ek.extkv_read_status(st) == ek.EXTKV_OK
    bad_np = inp.nonpad.clone()
    bad_np[0] = w.max_seq + 1
    y = torch.full_like(inp.q, 7.0)
    with ek.use_algo(algo):
        ek.attention_ext_kv(y, inp.q, k, v, bad_np, w.scale, status=st)
    assert ek.extkv_read_status(st) == ek.EXTKV_ERR_DEVICE
    assert "nonpad" in ek.extkv_last_error()
    assert (y[0] == 0).all()
    bias = torch.empty((w.B, 1, 1, w.max_seq), dtype=w.dtype, device="cuda")
    ek.extkv_clear_status(st)
    ek.build_static_cache_bias(bias, ek.BiasSpec(), bad_np, status=st)
    assert ek.extkv_read_status(st) == ek.EXTKV_ERR_DEVICE


def test_empty_calls_and_forced_kernel_refusal():
    q = torch.empty((0, 4, 1, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((0, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    ek.attention_ext_kv(torch.empty_like(q), q, kc, kc, torch.zeros(0, dtype=torch.int64, device="cuda"), 1.0)
    # the decode kernel cannot run fp32; forcing it is refused, not faked
    w = wl.C1_DECODE
    qf = torch.randn((1, 4, 1, 64), device="cuda")
    kf = torch.randn((1, 2, 64, 64), device="cuda")
    with ek.use_algo(ek.ALGO_DECODE):
        with pytest.raises(ek.ExtKVError) as e:
            ek.attention_ext_kv(torch.empty_like(qf), qf, kf, kf,
                                torch.tensor([17], dtype=torch.int64, device="cuda"), w.scale)
    assert e.value.code == ek.EXTKV_ERR_UNSUPPORTED


def test_decode_workspace_is_checked():
    w = wl.small(wl.C2)
    inp = wl.make_inputs(w, "cuda")
    need = ek.attention_ext_kv_workspace_size(w.B, w.Hq, w.Hkv, w.S_q, w.max_seq, w.D, w.dtype)
    assert need > 0
    y = torch.empty_like(inp.q)
    small_ws = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(ek.ExtKVError) as e:
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, workspace=small_ws)
    assert e.value.code == ek.EXTKV_ERR_INVALID_ARG and "workspace" in str(e.value)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # one workspace serves consecutive calls on the stream
    for _ in range(2):
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, workspace=ws)
    o = oracle_path(inp, mode="none", scatter=False)
    assert max_err(y, o["y"]) <= TOL[w.dtype]
