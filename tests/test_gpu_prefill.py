"""GPU parity of the tcgen05 prefill kernel against the fp64 oracle.

Shapes beyond the five workloads: every supported head dim (64, 128, 256),
query groups of 1, 2, 4 and 8 heads, ragged query tails (S_q not a multiple of
the 128-row tile), ragged key tails (max_seq not a multiple of the 64-key
tile), a non-causal layer with a dense extra term, image spans, and a chunk
just above the decode kernel's size.  Each runs in all three bias modes
(materialised, fused in registers, none) with the prefill kernel forced, and
the kernel that ran is checked by name.
"""
import numpy as np
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import TOL, max_err, oracle_path, run_gpu

pytestmark = pytest.mark.gpu

PRE = "attn_prefill_tcgen05"

EXTRA_PREFILL = [
    wl.Workload("pf_d64_g4_ragged", 201, B=2, Hq=8, Hkv=2, D=64, S_q=200, max_seq=1000,
                dtype=torch.bfloat16, causal=True, window=90, nonpad_range=(200, 1000)),
    wl.Workload("pf_d128_g1_noncausal_extra", 202, B=3, Hq=4, Hkv=4, D=128, S_q=130, max_seq=520,
                dtype=torch.bfloat16, causal=False, window=0, nonpad_range=(130, 520), extra=True),
    wl.Workload("pf_d256_g8_spans", 203, B=2, Hq=16, Hkv=2, D=256, S_q=160, max_seq=1024,
                dtype=torch.bfloat16, causal=True, window=64, nonpad_fixed=900, n_spans=2,
                span_len=40, span_start_range=(740, 860)),
    wl.Workload("pf_d128_g2_sq9", 204, B=2, Hq=2, Hkv=1, D=128, S_q=9, max_seq=256,
                dtype=torch.bfloat16, causal=True, nonpad_range=(9, 256)),
    wl.Workload("pf_d64_g2_long_garbage", 205, B=1, Hq=4, Hkv=2, D=64, S_q=384, max_seq=2048,
                dtype=torch.bfloat16, causal=True, window=500, nonpad_fixed=1500,
                garbage_sigma=10.0),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from biased_gqa_attention_gb300 import build
    build.build()


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
@pytest.mark.parametrize("w", EXTRA_PREFILL + [wl.small(wl.C3), wl.small(wl.C5)], ids=lambda w: w.name)
def test_prefill_kernel_forced(w, mode):
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL)
    assert g["kernel"].startswith(PRE)
    o = oracle_path(inp, mode=mode)
    err = max_err(g["y"], o["y"])
    assert err <= TOL[w.dtype], err


@pytest.mark.parametrize("mode", ["fused", "none"])
def test_prefill_key_tail_not_a_multiple_of_8(mode):
    """max_seq = 777: the cache views need no 16-byte bias rows without a bias."""
    w = wl.Workload("pf_d64_maxseq777", 206, B=2, Hq=4, Hkv=2, D=64, S_q=100, max_seq=777,
                    dtype=torch.bfloat16, causal=True, window=300, nonpad_range=(100, 777))
    inp = wl.make_inputs(w, "cuda")
    g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL)
    assert g["kernel"].startswith(PRE)
    o = oracle_path(inp, mode=mode)
    assert max_err(g["y"], o["y"]) <= TOL[w.dtype]


@pytest.mark.parametrize("w", [wl.C3, wl.C5, wl.small(wl.C3), wl.small(wl.C5)], ids=lambda w: w.name)
def test_prefill_workloads_pick_the_prefill_kernel(w):
    inp = wl.make_inputs(w, "cuda")
    assert run_gpu(inp, mode="bias")["kernel"].startswith(PRE)
    assert run_gpu(inp, mode="fused")["kernel"].startswith(PRE)


@pytest.mark.parametrize("mode", ["bias", "fused"])
@pytest.mark.parametrize("w", [wl.C3, wl.small(wl.C3), EXTRA_PREFILL[0]], ids=lambda w: w.name)
def test_prefill_huge_values_under_masked_slots_are_invisible(w, mode):
    """Slots before every row's window are masked for the whole query chunk:
    finite extremes there (K overflowing the scores, V overflowing P V) must
    leave the output bit for bit unchanged."""
    inp = wl.make_inputs(w, "cuda")
    clean = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL)
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    for b in range(w.B):
        q_start = int(inp.nonpad[b]) - w.S_q
        lo = max(q_start - w.window + 1, 0)
        k[b, :, :lo] = 3.0e38
        v[b, :, :lo] = -3.0e38
    dirty = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL, k_cache=k, v_cache=v)
    assert torch.equal(clean["y"].view(torch.int16), dirty["y"].view(torch.int16))


@pytest.mark.parametrize("mode", ["bias", "fused", "none"])
def test_prefill_poison_beyond_nonpad_is_bitwise_invisible(mode):
    w = EXTRA_PREFILL[2]
    clean = run_gpu(wl.make_inputs(w, "cuda"), mode=mode, algo=ek.ALGO_PREFILL)
    dirty = run_gpu(wl.make_inputs(w, "cuda", poison=True), mode=mode, algo=ek.ALGO_PREFILL)
    assert torch.equal(clean["y"].view(torch.int16), dirty["y"].view(torch.int16))


def test_prefill_empty_batch_negative_offset_and_unreachable_rows():
    """nonpad = 0 (all rows zero), nonpad < S_q (clamped start), and explicit
    query starts before slot 0 (causal rows with nothing to attend)."""
    w = wl.Workload("pf_edges", 207, B=3, Hq=4, Hkv=2, D=128, S_q=140, max_seq=512,
                    dtype=torch.bfloat16, causal=True, window=0, nonpad_fixed=300)
    inp = wl.make_inputs(w, "cuda")
    inp.nonpad = torch.tensor([0, 60, 300], dtype=torch.int64, device="cuda")
    inp.write_idx = torch.tensor([0, 0, 160], dtype=torch.int64, device="cuda")
    for mode in ("bias", "fused", "none"):
        g = run_gpu(inp, mode=mode, algo=ek.ALGO_PREFILL, scatter=False)
        o = oracle_path(inp, mode=mode, scatter=False)
        assert g["kernel"].startswith(PRE)
        assert (g["y"][0] == 0).all()
        assert max_err(g["y"], o["y"]) <= TOL[w.dtype]
    qs = torch.tensor([-5, -100, 100], dtype=torch.int64, device="cuda")
    spec = ek.BiasSpec(causal=True, window=0, q_start=qs)
    y = torch.empty_like(inp.q)
    with ek.use_algo(ek.ALGO_PREFILL):
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, fused=spec)
    assert (y[0] == 0).all()
    assert (y[1, :, :100] == 0).all() and (y[1, :, 100:] != 0).any()  # positions -100 .. 39
    bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device="cuda")
    ek.build_static_cache_bias(bias, spec, inp.nonpad)
    y2 = torch.empty_like(inp.q)
    with ek.use_algo(ek.ALGO_PREFILL):
        ek.attention_ext_kv(y2, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, bias=bias)
    assert torch.equal((y == 0), (y2 == 0))
    assert (y - y2).abs().max().item() <= TOL[w.dtype]


def test_prefill_bad_nonpad_sets_the_status_flag():
    w = EXTRA_PREFILL[0]
    inp = wl.make_inputs(w, "cuda")
    inp.nonpad = inp.nonpad.clone()
    inp.nonpad[1] = w.max_seq + 1
    st = ek.new_status()
    y = torch.empty_like(inp.q)
    with ek.use_algo(ek.ALGO_PREFILL):
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale, status=st)
    assert ek.extkv_read_status(st) == ek.EXTKV_ERR_DEVICE
    assert (y[1] == 0).all()


def test_prefill_full_c3_sampled_rows_in_every_mode():
    w = wl.C3
    inp = wl.make_inputs(w, "cuda")
    from gpu_path import sample_rows
    rows = sample_rows(w, 192)
    for mode in ("bias", "fused", "none"):
        g = run_gpu(inp, mode=mode)
        assert g["kernel"].startswith(PRE)
        o = oracle_path(inp, rows=rows, mode=mode)
        assert max_err(g["y"], o["y"], rows) <= TOL[w.dtype]


def test_prefill_bias_with_mask_only_and_dense_tiles_interleaved():
    """A materialised bias whose 128-key tiles alternate between values 0 /
    sentinel only (the kernel reads the plan's row bits) and other values (it
    reads the bias): the term blocks of the dense tiles must pair with the
    right tiles.  Also a NaN and a -0.0 inside mask-only tiles (NaN is masked,
    -0.0 adds nothing), and a finite very negative value that stays unmasked.
    The bias is built by the oracle and edited on the host."""
    from helpers import from_raw, raw
    import oracle
    w = wl.Workload("pf_mixed_tiles", 208, B=2, Hq=4, Hkv=2, D=128, S_q=200, max_seq=1280,
                    dtype=torch.bfloat16, causal=True, window=700, nonpad_range=(900, 1280))
    inp = wl.make_inputs(w, "cuda")
    nonpad = raw(inp.nonpad)
    bias, bad = oracle.bias(nonpad, w.S_q, w.max_seq, "bf16", causal=True, window=w.window)
    assert bad == 0
    b16 = bias.copy()
    rng = np.random.default_rng(5)
    lowest = 0xFF7F
    for t in (1, 3, 6):  # dense tiles: random values on the allowed slots
        blk = b16[:, :, :, t * 128:(t + 1) * 128]
        live = blk != lowest
        vals = (rng.standard_normal(blk.shape) * 2).astype(np.float32)
        bits = ((vals.view(np.uint32) + 0x7FFF + ((vals.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
        blk[live] = bits[live]
    b16[0, 0, 150, 2 * 128 + 5] = 0x7FC1   # NaN in a mask-only tile
    b16[1, 0, 10, 4 * 128 + 9] = 0x8000    # -0.0
    b16[1, 0, 199, 5 * 128 + 77] = 0xFF70  # about -3.2e38: finite, not masked
    y = torch.empty_like(inp.q)
    with ek.use_algo(ek.ALGO_PREFILL):
        ek.attention_ext_kv(y, inp.q, inp.k_cache, inp.v_cache, inp.nonpad, w.scale,
                            bias=from_raw(b16, torch.bfloat16).cuda())
        assert ek.extkv_last_kernel().startswith(PRE)
    ref = oracle.attention(raw(inp.q), raw(inp.k_cache), raw(inp.v_cache), b16, nonpad, np.float32(w.scale))
    assert max_err(y, ref) <= TOL[w.dtype]
