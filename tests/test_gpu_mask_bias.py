"""A boolean attention mask turned into the additive bias (build_bias_from_bool_mask),
and the maskless causal layer.

"ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 6: a bool mask is
converted to an additive bias; the attention-mask skill, "Bool mask vs float
additive bias": both represent any pattern, and is_causal=1 with nonpad and no
mask is the plain static-cache case.  The conversion is bit-exact against the
oracle; attention over a converted mask matches the oracle, and a causal +
window mask gives what the same pattern as a fused spec gives.
"""
import numpy as np
import pytest
import torch

import oracle
from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err
from helpers import dt_name, raw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 1, 1, 16), (3, 1, 5, 777), (2, 1, 130, 1024), (1, 1, 3, 9)])
def test_mask_bias_is_bit_exact(shape, dtype):
    g = torch.Generator().manual_seed(7)
    mask = (torch.rand(shape, generator=g) < 0.6).cuda()
    bias = torch.empty(shape, dtype=dtype, device="cuda")
    ek.build_bias_from_bool_mask(bias, mask)
    want = oracle.bias_from_mask(mask.cpu().numpy(), dt_name(dtype))
    assert np.array_equal(raw(bias), want)


def _causal_window_mask(nonpad, S_q, max_seq, window):
    B = len(nonpad)
    m = torch.zeros((B, 1, S_q, max_seq), dtype=torch.bool)
    j = torch.arange(max_seq)
    for b, n in enumerate(nonpad):
        qs = max(n - S_q, 0)
        for i in range(S_q):
            p = qs + i
            m[b, 0, i] = (j <= p) & (j < n) & ((p - j < window) if window > 0 else True)
    return m


@pytest.mark.parametrize("w", [wl.small(wl.C2), wl.small(wl.C3), wl.C1_PREFILL], ids=lambda w: w.name)
def test_causal_window_mask_equals_the_fused_spec(w):
    inp = wl.make_inputs(w, "cuda")
    mask = _causal_window_mask(inp.nonpad.tolist(), w.S_q, w.max_seq, w.window).cuda()
    bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda")
    ek.build_bias_from_bool_mask(bias, mask)
    y_mask = torch.empty_like(inp.q)
    ek.attention_ext_kv(y_mask, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, bias=bias)
    y_spec = torch.empty_like(inp.q)
    ek.attention_ext_kv(y_spec, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale,
                        fused=ek.BiasSpec(causal=True, window=w.window))
    assert max_err(y_mask, y_spec.float().cpu().numpy().astype(np.float64)) <= TOL[w.dtype]
    o = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache),
                         oracle.bias_from_mask(mask.cpu().numpy(), dt_name(w.dtype)), raw(inp.nonpad), w.scale)
    assert max_err(y_mask, o) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [wl.small(wl.C2), wl.small(wl.C5)], ids=lambda w: w.name)
def test_random_mask_with_a_fully_masked_row(w):
    inp = wl.make_inputs(w, "cuda")
    g = torch.Generator().manual_seed(11)
    mask = torch.rand((w.B, 1, w.S_q, w.max_seq), generator=g) < 0.5
    mask[0, 0, 0, :] = False  # row 0 of batch 0 attends nothing: an exact zero row
    mask = mask.cuda()
    bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda")
    ek.build_bias_from_bool_mask(bias, mask)
    y = torch.empty_like(inp.q)
    ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, bias=bias)
    o = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache),
                         oracle.bias_from_mask(mask.cpu().numpy(), dt_name(w.dtype)), raw(inp.nonpad), w.scale)
    assert (y[0, :, 0] == 0).all()
    assert max_err(y, o) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [wl.C1_PREFILL, wl.C1_DECODE, wl.small(wl.C3).replace(window=0, n_spans=0)],
                         ids=lambda w: w.name)
def test_maskless_causal_layer_is_the_causal_spec(w):
    """is_causal = 1 with nonpad and no mask (section 11 bottom-right alignment):
    the fused spec {causal = 1} and no bias tensor, against the oracle's causal bias."""
    inp = wl.make_inputs(w, "cuda")
    y = torch.empty_like(inp.q)
    ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, fused=ek.BiasSpec(causal=True))
    b, bad = oracle.bias(raw(inp.nonpad), w.S_q, w.max_seq, dt_name(w.dtype), causal=True, window=0)
    assert bad == 0
    o = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache), b, raw(inp.nonpad), w.scale)
    assert max_err(y, o) <= TOL[w.dtype]
