"""Pins for the oracle's attention (CPU only).

What fixes the result, independently of the oracle's own code:
  * a library routine on the special case it covers: torch CPU fp64
    scaled_dot_product_attention (math path) with K/V heads repeated by the
    group size and the bias (with -inf at masked keys) as its float mask;
  * closed forms: Q = 0 or identical keys give the mean of V over the unmasked
    set, a single unmasked key gives that key's V row exactly, a hand-worked
    row (tests/golden/hand_worked_softmax.txt), an empty unmasked set or an
    empty batch gives an exact zero row ("ONNX Domain Attention (Opset 23/24)
    CUDA Patterns", section 6);
  * invariants the pages state, exact in fp64 because the summation order does
    not change: poison values beyond nonpad or under masked bias never reach
    the output; GQA equals MHA with repeated KV heads (section 1, reshape-Q);
    a decode step equals the last row of the matching prefill and a chunked
    prefill equals the one-shot prefill (section 11, bottom-right alignment);
    a KV-shared layer ("[GQA] Support KV-shared layers with empty K/V inputs",
    Design) equals attention over the borrowed cache;
  * value rows of another head size (head_size != v_head_size, "Skill:
    Attention Optimization", "ORT CUDA Attention Kernel Dispatch"): torch SDPA
    on the same asymmetric shapes, and the output columns of a V split by
    columns are the columns of the whole (each output column is the same
    weighted sum over its own V column).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, dt, rng, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    if dt == "f32":
        return x
    # round to nearest even into bf16 bits
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _sdpa(q, k, v, bias, nonpad, scale, dt):
    """torch fp64 SDPA with repeated KV heads; masked keys get -inf."""
    qf, kf, vf = (torch.from_numpy(oracle.to_f64(a)) for a in (q, k, v))
    B, Hq, S_q, D = qf.shape
    Hkv, L = kf.shape[1], kf.shape[2]
    g = Hq // Hkv
    kf = kf.repeat_interleave(g, dim=1)
    vf = vf.repeat_interleave(g, dim=1)
    if dt == "f32":
        lowest = float(np.array([0xFF7FFFFF], np.uint32).view(np.float32)[0])
    else:
        lowest = float(oracle.to_f64(np.array([0xFF7F], np.uint16))[0])
    if bias is None:
        mask = torch.zeros((B, 1, S_q, L), dtype=torch.float64)
    else:
        mask = torch.from_numpy(oracle.to_f64(bias)).clone()
        mask[mask <= lowest] = -math.inf
    j = torch.arange(L)
    mask[(j[None, :] >= torch.as_tensor(nonpad)[:, None])[:, None, None, :].expand_as(mask)] = -math.inf
    with torch.no_grad():
        y = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=mask, scale=scale)
    live = torch.isfinite(mask).any(dim=-1)  # (B,1,S_q)
    return y.numpy(), live.expand(B, Hq, S_q).numpy()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["causal_window_spans", "extra_noncausal", "nobias"])
def test_matches_torch_sdpa_fp64(dt, kind):
    rng = np.random.default_rng(11)
    B, Hq, Hkv, S_q, L, D = 3, 6, 2, 5, 29, 16
    nonpad = np.array([29, 17, 9], np.int64)
    q = _rand((B, Hq, S_q, D), dt, rng)
    k = _rand((B, Hkv, L, D), dt, rng)
    v = _rand((B, Hkv, L, D), dt, rng)
    if kind == "causal_window_spans":
        bias, _ = oracle.bias(nonpad, S_q, L, dt, causal=True, window=6,
                              spans=[[(20, 6)], [(10, 4), (14, 2)], []])
    elif kind == "extra_noncausal":
        extra = _rand((B, 1, S_q, L), dt, rng, scale=2.0)
        bias, _ = oracle.bias(nonpad, S_q, L, dt, causal=False, window=7, extra=extra)
    else:
        bias = None
    scale = 1.0 / math.sqrt(D)
    y = oracle.attention(q, k, v, bias, nonpad, np.float32(scale))
    ref, live = _sdpa(q, k, v, bias, nonpad, float(np.float32(scale)), dt)
    assert live.any()
    np.testing.assert_allclose(y[live], ref[live], rtol=0, atol=1e-12)
    assert (y[~live] == 0).all()


def test_q_zero_and_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(3)
    B, H, S_q, L, D = 1, 2, 3, 12, 8
    nonpad = [10]
    v = _rand((B, H, L, D), "f32", rng)
    bias, _ = oracle.bias(nonpad, S_q, L, "f32", causal=True, window=4)
    vf = v.astype(np.float64)
    # Q = 0
    y = oracle.attention(np.zeros((B, H, S_q, D), np.float32), _rand((B, H, L, D), "f32", rng), v,
                         bias, nonpad, 0.3)
    for i in range(S_q):
        p = 7 + i
        np.testing.assert_allclose(y[0, :, i], vf[0, :, p - 3 : p + 1].mean(axis=1), atol=1e-14)
    # identical keys, nonzero Q
    k = np.repeat(_rand((B, H, 1, D), "f32", rng), L, axis=2)
    y = oracle.attention(_rand((B, H, S_q, D), "f32", rng), k, v, bias, nonpad, 0.3)
    for i in range(S_q):
        p = 7 + i
        np.testing.assert_allclose(y[0, :, i], vf[0, :, p - 3 : p + 1].mean(axis=1), atol=1e-14)


def test_single_unmasked_key_returns_its_value_row_exactly():
    rng = np.random.default_rng(4)
    for dt in ("f32", "bf16"):
        B, Hq, Hkv, L, D = 2, 4, 2, 16, 8
        nonpad = np.array([9, 16], np.int64)
        q, k, v = (_rand((B, Hq, 1, D), dt, rng), _rand((B, Hkv, L, D), dt, rng),
                   _rand((B, Hkv, L, D), dt, rng))
        bias, _ = oracle.bias(nonpad, 1, L, dt, causal=True, window=1)
        y = oracle.attention(q, k, v, bias, nonpad, 0.25)
        vf = oracle.to_f64(v)
        for b in range(B):
            for h in range(Hq):
                assert (y[b, h, 0] == vf[b, h // 2, nonpad[b] - 1]).all()


def _golden():
    rows = {}
    with open(os.path.join(GOLDEN, "hand_worked_softmax.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append([float(x) for x in vals])
    return rows


def test_hand_worked_row():
    g = _golden()
    q = np.array(g["q"], np.float32).reshape(1, 1, 1, 4)
    k = np.array(g["k"], np.float32).reshape(1, 1, 4, 4)
    v = np.array(g["v"], np.float32).reshape(1, 1, 4, 4)
    bias = np.array(g["bias"], np.float32).reshape(1, 1, 1, 4)
    y = oracle.attention(q, k, v, bias, [4], g["scale"][0][0])
    np.testing.assert_allclose(y[0, 0, 0], np.array(g["y"][0]), rtol=0, atol=1e-15)


def test_sentinel_and_minus_inf_mask_but_finite_negative_does_not():
    v = np.array([[1, 2], [3, 4], [5, 6]], np.float32).reshape(1, 1, 3, 2)
    k = np.zeros((1, 1, 3, 2), np.float32)
    q = np.zeros((1, 1, 1, 2), np.float32)
    low = np.array([0xFF7FFFFF], np.uint32).view(np.float32)[0]
    # -inf and lowest are masked; the remaining key gets all the weight
    b = np.array([-np.inf, low, 0.0], np.float32).reshape(1, 1, 1, 3)
    assert (oracle.attention(q, k, v, b, [3], 1.0)[0, 0, 0] == [5, 6]).all()
    # a finite -1e30 key alone is not masked: the row is not zeroed
    b = np.array([low, -1e30, low], np.float32).reshape(1, 1, 1, 3)
    assert (oracle.attention(q, k, v, b, [3], 1.0)[0, 0, 0] == [3, 4]).all()
    # every key at the sentinel: exact zero row
    b = np.full((1, 1, 1, 3), low, np.float32)
    assert (oracle.attention(q, k, v, b, [3], 1.0)[0, 0, 0] == 0).all()
    # nonpad = 0: the batch is empty, exact zero even with poisoned values
    vn = np.full_like(v, np.nan)
    assert (oracle.attention(q, k, vn, None, [0], 1.0) == 0).all()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_huge_finite_biases_stay_unmasked_and_compete_among_themselves(dt):
    """Biases in (lowest, -2.4e38) are finite, so they do not mask (section 6
    of the ORT page); only their differences count (softmax is invariant to a
    shared shift).  Two live keys at -3.0e38 and -2.9e38: the gap of about
    1e37 gives the first a weight exp(-1e37) = 0, so the row is the second
    key's value row exactly.  Equal huge values on three keys: the scores'
    own differences vanish next to them in fp64, so the row is the mean of
    the three value rows.  +3e38 on one key among ordinary biases: that key's
    row exactly."""
    rng = np.random.default_rng(5)
    v = np.array([[1, 2], [3, 4], [5, 6], [7, 8]], np.float32).reshape(1, 1, 4, 2)
    k = rng.standard_normal((1, 1, 4, 2)).astype(np.float32)
    q = rng.standard_normal((1, 1, 1, 2)).astype(np.float32)
    if dt == "bf16":
        to = lambda a: _rand_bits(np.asarray(a, np.float32))  # noqa: E731
        v, k, q = to(v), to(k), to(q)
        low = np.uint16(0xFF7F)
    else:
        to = lambda a: np.asarray(a, np.float32)  # noqa: E731
        low = np.array([0xFF7FFFFF], np.uint32).view(np.float32)[0]
    vf = oracle.to_f64(v)[0, 0]

    def row(vals):
        b = to(np.array(vals, np.float32)).reshape(1, 1, 1, 4)
        b[0, 0, 0, [i for i, x in enumerate(vals) if x is None]] = low
        return oracle.attention(q, k, v, b, [4], 1.0)[0, 0, 0]

    assert (row([None, -3.0e38, -2.9e38, None]) == vf[2]).all()
    y = row([-3.0e38, -3.0e38, None, -3.0e38])
    np.testing.assert_allclose(y, (vf[0] + vf[1] + vf[3]) / 3, rtol=0, atol=1e-15)
    assert (row([0.0, 3.0e38, 0.0, 0.0]) == vf[1]).all()


def _rand_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (None entries are filled after)."""
    x = np.nan_to_num(x.astype(np.float32), nan=0.0)
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _setup(dt, rng, B=2, Hq=4, Hkv=2, S_q=6, L=40, D=8):
    nonpad = np.array([33, 21], np.int64)[:B]
    q = _rand((B, Hq, S_q, D), dt, rng)
    k = _rand((B, Hkv, L, D), dt, rng)
    v = _rand((B, Hkv, L, D), dt, rng)
    return nonpad, q, k, v


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_poison_beyond_nonpad_and_under_masked_bias_never_reaches_output(dt):
    rng = np.random.default_rng(5)
    nonpad, q, k, v = _setup(dt, rng)
    L = k.shape[2]
    bias, _ = oracle.bias(nonpad, 6, L, dt, causal=True, window=5, spans=[[(25, 5)], []])
    y0 = oracle.attention(q, k, v, bias, nonpad, 0.35)
    kp, vp = k.copy(), v.copy()
    nan = np.float32(np.nan) if dt == "f32" else np.uint16(0x7FC0)
    big = np.float32(1e30) if dt == "f32" else np.uint16(0x7149)  # ~1e30 in bf16
    for b in range(2):
        kp[b, :, nonpad[b]:] = nan
        vp[b, :, nonpad[b]:] = nan
        # slots below nonpad that no query row of batch b can see
        m = (bias[b, 0].view(np.uint32) if dt == "f32" else bias[b, 0]) != oracle.LOWEST_BITS[dt]
        dead = ~m.any(axis=0)
        dead[nonpad[b]:] = False
        kp[b, :, dead] = big
        vp[b, :, dead] = big
    y1 = oracle.attention(q, kp, vp, bias, nonpad, 0.35)
    assert y0.tobytes() == y1.tobytes()


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(6)
    nonpad, q, k, v = _setup("bf16", rng, Hq=6, Hkv=2)
    bias, _ = oracle.bias(nonpad, 6, 40, "bf16", causal=True, window=9)
    y_gqa = oracle.attention(q, k, v, bias, nonpad, 0.4)
    y_mha = oracle.attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), bias, nonpad, 0.4)
    assert y_gqa.tobytes() == y_mha.tobytes()


def test_decode_equals_last_prefill_row_and_chunked_equals_one_shot():
    rng = np.random.default_rng(7)
    nonpad, q, k, v = _setup("bf16", rng, S_q=8)
    L = 40
    full_bias, _ = oracle.bias(nonpad, 8, L, "bf16", causal=True, window=7)
    y_full = oracle.attention(q, k, v, full_bias, nonpad, 0.3)
    # decode: the last query alone, nonpad unchanged
    dec_bias, _ = oracle.bias(nonpad, 1, L, "bf16", causal=True, window=7)
    y_dec = oracle.attention(q[:, :, 7:8].copy(), k, v, dec_bias, nonpad, 0.3)
    assert y_dec.tobytes() == y_full[:, :, 7:8].tobytes()
    # two chunks of 4: the first sees nonpad-4 valid slots, the second all of them
    np1 = nonpad - 4
    b1, _ = oracle.bias(np1, 4, L, "bf16", causal=True, window=7)
    b2, _ = oracle.bias(nonpad, 4, L, "bf16", causal=True, window=7)
    y1 = oracle.attention(q[:, :, :4].copy(), k, v, b1, np1, 0.3)
    y2 = oracle.attention(q[:, :, 4:].copy(), k, v, b2, nonpad, 0.3)
    assert np.concatenate([y1, y2], axis=2).tobytes() == y_full.tobytes()


def test_kv_shared_layer_attends_the_borrowed_cache():
    """A KV-shared layer writes no K/V (an empty scatter) and attends the
    source layer's cache; the result equals attention over that cache alone,
    which here is checked against fp64 SDPA over the first nonpad slots."""
    rng = np.random.default_rng(8)
    B, Hq, Hkv, S_q, L, D = 2, 4, 2, 4, 32, 8
    kc, vc = _rand((B, Hkv, L, D), "bf16", rng), _rand((B, Hkv, L, D), "bf16", rng)
    kn, vn = _rand((B, Hkv, S_q, D), "bf16", rng), _rand((B, Hkv, S_q, D), "bf16", rng)
    w = np.array([10, 20], np.int64)
    nonpad = w + S_q
    oracle.scatter(kc, vc, kn, vn, w)
    q_src, q_shared = _rand((B, Hq, S_q, D), "bf16", rng), _rand((B, Hq, S_q, D), "bf16", rng)
    bias, _ = oracle.bias(nonpad, S_q, L, "bf16", causal=True, window=9)
    before = (kc.copy(), vc.copy())
    empty = np.zeros((B, Hkv, 0, D), np.uint16)
    assert oracle.scatter(kc, vc, empty, empty, nonpad) == 0
    assert kc.tobytes() == before[0].tobytes() and vc.tobytes() == before[1].tobytes()
    y_shared = oracle.attention(q_shared, kc, vc, bias, nonpad, 0.5)
    ref, live = _sdpa(q_shared, kc, vc, bias, nonpad, 0.5, "bf16")
    assert live.all()
    np.testing.assert_allclose(y_shared, ref, rtol=0, atol=1e-12)


def test_row_subset_matches_full_and_threads_do_not_change_bits():
    rng = np.random.default_rng(9)
    nonpad, q, k, v = _setup("bf16", rng)
    bias, _ = oracle.bias(nonpad, 6, 40, "bf16", causal=True, window=11)
    y = oracle.attention(q, k, v, bias, nonpad, 0.3)
    rows = np.array([0, 5, 17, 47, 23], np.int64)
    ys = oracle.attention(q, k, v, bias, nonpad, 0.3, rows=rows)
    assert ys.tobytes() == y.reshape(-1, 8)[rows].tobytes()


# ---- softcap: cap * tanh(x / cap) on the scaled scores, before the bias -------
# "ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 4 (op order:
# scale, softcap, + bias / mask, softmax).

def _softcap_case(dt, seed=3):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, S_q, max_seq, D = 2, 4, 2, 3, 40, 16
    q = _rand((B, Hq, S_q, D), dt, rng)
    k = _rand((B, Hkv, max_seq, D), dt, rng)
    v = _rand((B, Hkv, max_seq, D), dt, rng)
    nonpad = np.array([40, 23], np.int64)
    return q, k, v, nonpad, 1.0 / np.sqrt(D)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_softcap_large_cap_converges_to_no_cap_within_the_taylor_bound(dt):
    """cap * tanh(x / cap) = x - x^3 / (3 cap^2) + ..., so with |x| <= X the
    scores move by at most X^3 / (3 cap^2) and the output by less than
    2 * max|v| * (exp(2 delta) - 1)."""
    q, k, v, nonpad, scale = _softcap_case(dt)
    b, _ = oracle.bias(nonpad, 3, 40, dt, causal=True, window=0)
    cap = 200.0
    qf, kf = oracle.to_f64(q), oracle.to_f64(k)
    X = scale * np.abs(np.einsum("bhsd,bkjd->bhskj", qf, kf)).max()
    delta = X ** 3 / (3 * cap ** 2)
    y0 = oracle.attention(q, k, v, b, nonpad, scale)
    y1 = oracle.attention(q, k, v, b, nonpad, scale, softcap=cap)
    bound = 2 * np.abs(oracle.to_f64(v)).max() * (np.exp(2 * delta) - 1)
    assert 0 < np.abs(y1 - y0).max() <= bound


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_softcap_before_the_bias_keeps_softmax_shift_invariance(dt):
    """Adding one constant to every allowed bias entry of a row leaves the
    output unchanged only if the cap acts before the bias (with the cap after
    it, tanh would see the shifted scores)."""
    q, k, v, nonpad, scale = _softcap_case(dt)
    rng = np.random.default_rng(9)
    ex = (np.round(np.clip(rng.standard_normal((2, 1, 3, 40)), -3, 3) * 4) / 4).astype(np.float32)  # exact in bf16, +1.5 too
    extra = ex if dt == "f32" else (ex.view(np.uint32) >> 16).astype(np.uint16)
    b, _ = oracle.bias(nonpad, 3, 40, dt, causal=True, window=0, extra=extra)
    b2, _ = oracle.bias(nonpad, 3, 40, dt, causal=True, window=0,
                        extra=(ex + 1.5) if dt == "f32" else ((ex + 1.5).view(np.uint32) >> 16).astype(np.uint16))
    for cap in (1.0, 3.0):
        y1 = oracle.attention(q, k, v, b, nonpad, scale, softcap=cap)
        y2 = oracle.attention(q, k, v, b2, nonpad, scale, softcap=cap)
        assert np.abs(y1 - y2).max() <= 1e-12
    assert np.abs(oracle.attention(q, k, v, b, nonpad, scale, softcap=1.0) -
                  oracle.attention(q, k, v, b, nonpad, scale)).max() > 1e-3  # the cap does act


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_softcap_single_key_and_poison_under_the_mask(dt):
    """One unmasked key: y is its value row, whatever the cap.  A tiny cap with
    NaN V rows under masked slots (the pages' guard case): the masked slots
    stay out of the softmax, the output is finite and equals the output
    without the poison."""
    q, k, v, nonpad, scale = _softcap_case(dt)
    b, _ = oracle.bias(nonpad, 3, 40, dt, causal=True, window=1)  # each row: its own key only
    y = oracle.attention(q, k, v, b, nonpad, scale, softcap=0.5)
    vf = oracle.to_f64(v)
    for bb in range(2):
        qs = max(int(nonpad[bb]) - 3, 0)
        for h in range(4):
            for i in range(3):
                assert np.array_equal(y[bb, h, i], vf[bb, h // 2, qs + i])
    bw, _ = oracle.bias(nonpad, 3, 40, dt, causal=True, window=8)
    vp = v.copy()
    nan = np.float32(np.nan) if dt == "f32" else np.uint16(0x7FC0)
    for bb in range(2):  # every slot before the first row's window (query 0 at nonpad - 3)
        vp[bb, :, :max(int(nonpad[bb]) - 3 - 8 + 1, 0)] = nan
    y0 = oracle.attention(q, k, v, bw, nonpad, scale, softcap=0.05)
    yp = oracle.attention(q, k, vp, bw, nonpad, scale, softcap=0.05)
    assert np.isfinite(yp).all() and np.array_equal(y0, yp)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(16, 24), (24, 8)])
def test_value_head_size_differs_matches_torch_sdpa_fp64(dt, dk, dv):
    rng = np.random.default_rng(21)
    B, Hq, Hkv, S_q, L = 2, 4, 2, 5, 23
    nonpad = np.array([23, 11], np.int64)
    q = _rand((B, Hq, S_q, dk), dt, rng)
    k = _rand((B, Hkv, L, dk), dt, rng)
    v = _rand((B, Hkv, L, dv), dt, rng)
    bias, _ = oracle.bias(nonpad, S_q, L, dt, causal=True, window=7, spans=[[(15, 5)], []])
    scale = np.float32(1.0 / math.sqrt(dk))
    y = oracle.attention(q, k, v, bias, nonpad, scale)
    assert y.shape == (B, Hq, S_q, dv)
    ref, live = _sdpa(q, k, v, bias, nonpad, float(scale), dt)
    assert live.any()
    np.testing.assert_allclose(y[live], ref[live], rtol=0, atol=1e-12)
    assert (y[~live] == 0).all()


def test_value_columns_split_equals_whole():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, S_q, L, dk, dv = 2, 4, 1, 3, 19, 8, 12
    nonpad = np.array([19, 7], np.int64)
    q = _rand((B, Hq, S_q, dk), "bf16", rng)
    k = _rand((B, Hkv, L, dk), "bf16", rng)
    v = _rand((B, Hkv, L, dv), "bf16", rng)
    bias, _ = oracle.bias(nonpad, S_q, L, "bf16", causal=True, window=5)
    scale = np.float32(0.3)
    whole = oracle.attention(q, k, v, bias, nonpad, scale)
    left = oracle.attention(q, k, np.ascontiguousarray(v[..., :5]), bias, nonpad, scale)
    right = oracle.attention(q, k, np.ascontiguousarray(v[..., 5:]), bias, nonpad, scale)
    assert np.array_equal(whole, np.concatenate([left, right], axis=-1))
