"""Pins for the oracle's static-cache bias builder (CPU only).

Each check is a closed form stated by the pages or by the workload definition,
not a retyped copy of the oracle's predicate:
  * "Skill: Attention Optimization", "GQA sliding window via local_window_size":
    the query at position i sees exactly keys [i-W+1, i].
  * "ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 11: with an
    external cache, query i sits at nonpad - S_q + i (clamped offset >= 0), so
    a decode row sees every valid key and nonpad < S_q gives offset 0.
  * mobius issue #366, deliverable: (B,1,S_q,max_seq), valid only where
    slot < nonpad; the block overlay makes a span's tokens see each other.
  * section 8 of the ORT page: masked entries hold lowest(T), finite.
"""
import numpy as np
import pytest

import oracle
from biased_gqa_attention_gb300 import workloads as wl

LOW = {"f32": np.uint32(0xFF7FFFFF), "bf16": np.uint16(0xFF7F)}


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def allowed_mask(bias, dt):
    """True where the entry is not the sentinel."""
    return _bits(bias) != LOW[dt]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_entries_are_zero_or_lowest(dt):
    b, bad = oracle.bias([37, 5], S_q=6, max_seq=48, dt=dt, causal=True, window=9)
    assert bad == 0
    bits = _bits(b)
    assert set(np.unique(bits).tolist()) <= {0, int(LOW[dt])}
    # lowest(T) is finite: about -3.40e38 for fp32 (ORT page, section 2), and
    # the largest-magnitude finite bf16, -(2 - 2^-7) * 2^127, for bf16
    f = oracle.to_f64(b)
    assert np.isfinite(f).all()
    if dt == "f32":
        assert f.min() == pytest.approx(-3.40e38, rel=2e-3)
    else:
        assert f.min() == -(2 - 2.0 ** -7) * 2.0 ** 127


def test_c1_prefill_lower_triangle_and_decode_row():
    pre, _ = oracle.bias([16], S_q=16, max_seq=64, dt="f32", causal=True)
    m = allowed_mask(pre[0, 0], "f32")
    expect = np.zeros((16, 64), bool)
    for i in range(16):
        expect[i, : i + 1] = True
    assert (m == expect).all()
    dec, _ = oracle.bias([17], S_q=1, max_seq=64, dt="f32", causal=True)
    md = allowed_mask(dec[0, 0], "f32")
    assert md[0, :17].all() and not md[0, 17:].any()
    assert (dec[0, 0, 0, :17] == 0).all()


def test_window_sees_exactly_last_w_keys():
    # decode at position p = nonpad-1 with W=3 sees {p-2, p-1, p}
    b, _ = oracle.bias([6], S_q=1, max_seq=16, dt="bf16", causal=True, window=3)
    assert np.flatnonzero(allowed_mask(b[0, 0, 0], "bf16")).tolist() == [3, 4, 5]
    # prefill rows: row i at position p = 10 - 4 + i sees [max(p-2,0), p]
    b, _ = oracle.bias([10], S_q=4, max_seq=16, dt="bf16", causal=True, window=3)
    for i in range(4):
        p = 6 + i
        assert np.flatnonzero(allowed_mask(b[0, 0, i], "bf16")).tolist() == [p - 2, p - 1, p]


def test_c2_rows_count_min_nonpad_window():
    w = wl.C2
    nonpad, _, _ = wl.structure(w)
    b, bad = oracle.bias(nonpad.numpy(), S_q=1, max_seq=w.max_seq, dt="bf16", causal=True,
                         window=w.window)
    assert bad == 0
    for bi, npv in enumerate(nonpad.tolist()):
        idx = np.flatnonzero(allowed_mask(b[bi, 0, 0], "bf16"))
        assert len(idx) == min(npv, 1024)
        assert idx[0] == max(npv - 1024, 0) and idx[-1] == npv - 1
        assert (np.diff(idx) == 1).all()


def test_c3_span_rows_closed_form():
    w = wl.C3
    nonpad, _, spans = wl.structure(w)
    so, sp = oracle.spans_csr(spans)
    b, bad = oracle.bias(nonpad.numpy(), S_q=w.S_q, max_seq=w.max_seq, dt="bf16", causal=True,
                         window=w.window, spans=spans)
    assert bad == 0
    m = allowed_mask(b[0, 0], "bf16")
    counts = m.sum(axis=1)
    q0 = 4096 - 2048
    in_span = {}
    for s, L in spans[0]:
        assert 2048 <= s <= 4096 - 256 and L == 256
        for k in range(L):
            in_span[s + k - q0] = (s, k)
    for i in range(w.S_q):
        p = q0 + i
        if i in in_span:
            s, k = in_span[i]
            assert counts[i] == 1024 + (255 - k)
            expect = set(range(p - 1023, p + 1)) | set(range(s, s + 256))
        else:
            assert counts[i] == 1024
            expect = set(range(p - 1023, p + 1))
        if i % 97 == 0 or i in (0, w.S_q - 1) or i in in_span and in_span[i][1] in (0, 255):
            assert set(np.flatnonzero(m[i]).tolist()) == expect
    assert not m[:, 4096:].any()


def test_negative_offset_clamps_to_zero():
    # nonpad=3 < S_q=5: offset nonpad-S_q = -2 clamps to 0, so row i sits at i
    b, _ = oracle.bias([3], S_q=5, max_seq=8, dt="f32", causal=True)
    for i in range(5):
        assert np.flatnonzero(allowed_mask(b[0, 0, i], "f32")).tolist() == list(range(min(i, 2) + 1))


def test_block_overlay_or_composition_and_padding_wins():
    # non-causal off, window 2, one span [4,8) with nonpad 6: padding cuts the span
    b, _ = oracle.bias([6], S_q=6, max_seq=10, dt="bf16", causal=True, window=2,
                       spans=[[(4, 4)]])
    m = allowed_mask(b[0, 0], "bf16")
    # row 4 (p=4) is in the span: window {3,4} plus span {4,5} (6,7 are padding)
    assert np.flatnonzero(m[4]).tolist() == [3, 4, 5]
    # row 3 (p=3) is outside the span: only {2,3}
    assert np.flatnonzero(m[3]).tolist() == [2, 3]
    # row 5 sees {4,5} by window, and span gives nothing new
    assert np.flatnonzero(m[5]).tolist() == [4, 5]


def test_extra_only_on_allowed_slots():
    rng = np.random.default_rng(0)
    extra = rng.standard_normal((2, 1, 3, 16)).astype(np.float32)
    b, _ = oracle.bias([9, 16], S_q=3, max_seq=16, dt="f32", causal=True, window=4, extra=extra)
    m = allowed_mask(b, "f32")
    assert (b[m] == extra[m]).all()
    assert (b.view(np.uint32)[~m] == 0xFF7FFFFF).all()


def test_explicit_q_start_overrides_offset():
    b, _ = oracle.bias([12], S_q=2, max_seq=16, dt="f32", causal=True, q_start=[3])
    assert np.flatnonzero(allowed_mask(b[0, 0, 0], "f32")).tolist() == [0, 1, 2, 3]
    assert np.flatnonzero(allowed_mask(b[0, 0, 1], "f32")).tolist() == [0, 1, 2, 3, 4]


def test_out_of_range_nonpad_is_reported():
    b, bad = oracle.bias([5, 17, -1], S_q=1, max_seq=16, dt="f32")
    assert bad == 2
    assert allowed_mask(b[0, 0], "f32")[0, :5].all()


# ---- a boolean attention mask turned into the additive bias ------------------
# "ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 6 ("Additive-bias
# path", bool mask converted to bias) and the attention-mask skill ("Bool mask
# vs float additive bias": both represent any pattern; the bool mask becomes a
# float bias internally).  Pinned against independent paths: the spec builder
# above, and the attention with and without a bias.

def _causal_window_mask(nonpad, S_q, max_seq, window):
    """Boolean mask from the closed form of the section-11 positions: query i of
    batch b sits at max(nonpad - S_q, 0) + i and sees j in (p - window, p], j < nonpad."""
    B = len(nonpad)
    m = np.zeros((B, 1, S_q, max_seq), bool)
    j = np.arange(max_seq)
    for b, n in enumerate(nonpad):
        qs = max(n - S_q, 0)
        for i in range(S_q):
            p = qs + i
            m[b, 0, i] = (j <= p) & (j < n) & ((p - j < window) if window > 0 else True)
    return m


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_bool_mask_bias_equals_the_spec_builder(dt):
    nonpad, S_q, max_seq, W = [37, 5, 48], 6, 48, 9
    mask = _causal_window_mask(nonpad, S_q, max_seq, W)
    from_mask = oracle.bias_from_mask(mask, dt)
    from_spec, bad = oracle.bias(nonpad, S_q=S_q, max_seq=max_seq, dt=dt, causal=True, window=W)
    assert bad == 0
    assert np.array_equal(from_mask, from_spec)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_bool_mask_all_true_is_no_bias_and_a_false_row_is_a_zero_row(dt):
    rng = np.random.default_rng(5)
    B, Hq, Hkv, S_q, max_seq, D = 2, 4, 2, 3, 24, 8

    def rand(shape):  # fp32 values, or their bf16 bits (round to nearest even)
        x = rng.standard_normal(shape).astype(np.float32)
        if dt == "f32":
            return x
        u = x.view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    q, k, v = rand((B, Hq, S_q, D)), rand((B, Hkv, max_seq, D)), rand((B, Hkv, max_seq, D))
    nonpad = np.array([24, 17], np.int64)
    mask = np.ones((B, 1, S_q, max_seq), bool)
    y_all = oracle.attention(q, k, v, oracle.bias_from_mask(mask, dt), nonpad, 0.35)
    y_none = oracle.attention(q, k, v, None, nonpad, 0.35)
    assert np.array_equal(y_all, y_none)
    mask[1, 0, 2, :] = False  # query row 2 of batch 1 attends nothing
    y = oracle.attention(q, k, v, oracle.bias_from_mask(mask, dt), nonpad, 0.35)
    assert np.all(y[1, :, 2] == 0.0)
    assert np.array_equal(y[0], y_none[0])
