"""Extreme finite biases on every attention path, against the oracle.

"ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 6: a bias
equal to lowest(T) (or -inf) masks its key, a finite bias above lowest(T)
does not, however negative it is; section 2 warns that scaling such a bias
by log2(e) before the row maximum is subtracted overflows fp32 (|b| above
about 2.36e38) and turns it into a mask.  These tests give whole rows only
huge finite biases in (lowest, -2.4e38), and single keys +3e38, through a
materialised bias and through the fused specification's extra term, on the
decode kernels (stream-K and cluster), the tcgen05 prefill kernel (with and
without key splits) and the generic kernel, and compare each element with the
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, spec_of
from helpers import dt_name, from_raw, raw

LOWEST = {torch.bfloat16: 0xFF7F, torch.float32: 0xFF7FFFFF}
# finite values beyond the fp32 range of b*log2(e), none of them a mask
HUGE_NEG = (-3.0e38, -2.9e38, -2.5e38, -3.19e38)


def _bits(x: np.ndarray, dtype) -> np.ndarray:
    """float32 values -> the element type's bit pattern (round to nearest even)."""
    b = np.asarray(x, np.float32).view(np.uint32)
    if dtype == torch.float32:
        return b
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _edit_rows(bias: np.ndarray, dtype, nonpad, rng) -> np.ndarray:
    """Per batch b (row i = last query row for b odd, first for b even):
    b % 4 == 1: every live key of the row gets a huge negative bias, varying;
    b % 4 == 2: one live key gets +3e38, the others keep their values;
    b % 4 == 3: every live key gets the same huge negative bias;
    b % 4 == 0: the row is left as the spec built it."""
    out = bias.copy()
    u = out.view(np.uint32) if dtype == torch.float32 else out  # edited through the bit pattern
    low = LOWEST[dtype]
    B, _, S_q, _ = out.shape
    for b in range(B):
        i = S_q - 1 if b % 2 else 0
        live = np.nonzero(u[b, 0, i, :int(nonpad[b])] != low)[0]
        if live.size == 0 or b % 4 == 0:
            continue
        if b % 4 == 1:
            vals = np.array([HUGE_NEG[k % len(HUGE_NEG)] for k in range(live.size)], np.float32)
            rng.shuffle(vals)
            u[b, 0, i, live] = _bits(vals, dtype)
        elif b % 4 == 2:
            u[b, 0, i, live[rng.integers(live.size)]] = _bits(np.float32(3.0e38), dtype)
        else:
            u[b, 0, i, live] = _bits(np.full(live.size, -3.0e38, np.float32), dtype)
    return out


def _run(w: wl.Workload, algo: int, mode: str, seed: int):
    inp = wl.make_inputs(w, "cuda")
    nonpad = raw(inp.nonpad)
    rng = np.random.default_rng(seed)
    dt = dt_name(w.dtype)
    base, bad = oracle.bias(nonpad, w.S_q, w.max_seq, dt, causal=w.causal, window=w.window)
    assert bad == 0
    edited = _edit_rows(base, w.dtype, nonpad, rng)
    y = torch.full((w.B, w.Hq, w.S_q, w.D), float("nan"), dtype=w.dtype, device="cuda")
    st = ek.new_status()
    if mode == "bias":
        bias_t = from_raw(edited, w.dtype).cuda()
        ref_bias = edited
        with ek.use_algo(algo):
            ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, bias=bias_t, status=st)
            kernel = ek.extkv_last_kernel()
    else:
        # the extra term carries the values; the spec's mask stays the same
        low = LOWEST[w.dtype]
        ebits = edited.view(np.uint32) if w.dtype == torch.float32 else edited
        extra = np.where(ebits == low, _bits(np.float32(0.0), w.dtype), ebits).astype(ebits.dtype)
        if w.dtype == torch.float32:
            extra = extra.view(np.float32)
        extra_t = from_raw(extra, w.dtype).cuda()
        spec = spec_of(inp)
        spec.extra = extra_t
        ref_bias, bad = oracle.bias(nonpad, w.S_q, w.max_seq, dt, causal=w.causal, window=w.window, extra=extra)
        assert bad == 0
        with ek.use_algo(algo):
            ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, fused=spec, status=st)
            kernel = ek.extkv_last_kernel()
    assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
    ref = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache), ref_bias, nonpad, np.float32(w.scale))
    return y, ref, kernel


DECODE = wl.Workload("extreme_decode", 301, B=8, Hq=8, Hkv=4, D=128, S_q=1, max_seq=2048,
                     dtype=torch.bfloat16, causal=True, window=700, nonpad_range=(40, 2048))
DECODE_G = DECODE.replace(name="extreme_decode_g4", config_id=302, Hq=16, D=256, window=0)
PREFILL_SPLIT = wl.Workload("extreme_prefill_split", 303, B=4, Hq=4, Hkv=2, D=128, S_q=160, max_seq=1024,
                            dtype=torch.bfloat16, causal=True, window=300, nonpad_range=(160, 1024))
PREFILL_WIDE = wl.Workload("extreme_prefill_wide", 304, B=4, Hq=16, Hkv=8, D=256, S_q=200, max_seq=1024,
                           dtype=torch.bfloat16, causal=True, window=0, nonpad_range=(200, 1024))


@pytest.mark.gpu
@pytest.mark.parametrize("algo,name", [(ek.ALGO_DECODE_STREAMK, "attn_decode_streamk_mma"),
                                       (ek.ALGO_DECODE_CLUSTER, "attn_decode_cluster")], ids=["streamk", "cluster"])
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [DECODE, DECODE_G], ids=lambda w: w.name)
def test_decode_kernel_extreme_biases(w, mode, algo, name):
    y, ref, kernel = _run(w, algo, mode, seed=11)
    assert kernel == name, kernel
    assert max_err(y, ref) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [PREFILL_SPLIT, PREFILL_WIDE, DECODE], ids=lambda w: w.name)
def test_prefill_kernel_extreme_biases(w, mode):
    y, ref, kernel = _run(w, ek.ALGO_PREFILL, mode, seed=12)
    assert kernel.startswith("attn_prefill_tcgen05"), kernel
    assert max_err(y, ref) <= TOL[w.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("mode", ["bias", "fused"])
def test_generic_kernel_extreme_biases(dtype, mode):
    w = PREFILL_SPLIT.replace(name=f"extreme_generic_{dtype}", dtype=dtype, S_q=40, max_seq=512,
                              nonpad_range=(40, 512))
    y, ref, kernel = _run(w, ek.ALGO_GENERIC, mode, seed=13)
    assert kernel.startswith("attn_generic"), kernel
    assert max_err(y, ref) <= TOL[w.dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_edited_rows_keep_the_cases_they_claim(dtype):
    """Host check of the fixture: the edited rows hold what the docstring
    says (huge finite values only, never the sentinel), so the GPU tests test
    what they claim."""
    w = DECODE.replace(dtype=dtype)
    nonpad = raw(wl.make_inputs(w, "cpu").nonpad)
    base, _ = oracle.bias(nonpad, w.S_q, w.max_seq, dt_name(dtype), causal=True, window=w.window)
    ed = _edit_rows(base, dtype, nonpad, np.random.default_rng(11))
    as_f = ed if dtype == torch.float32 else (ed.astype(np.uint32) << 16).view(np.float32)
    low = np.array([LOWEST[dtype]], np.uint32 if dtype == torch.float32 else np.uint16)
    low_f = low.view(np.float32)[0] if dtype == torch.float32 else (low.astype(np.uint32) << 16).view(np.float32)[0]
    n_checked = 0
    for b in range(w.B):
        row = as_f[b, 0, 0, :int(nonpad[b])]
        live = row > low_f
        n_checked += int(live.any())
        if b % 4 in (1, 3) and live.any():
            assert (row[live] < -2.4e38).all()
        if b % 4 == 2 and live.any():
            assert (row[live] > 2.9e38).sum() == 1
    assert n_checked >= 4
