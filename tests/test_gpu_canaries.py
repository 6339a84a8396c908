"""Writes stay inside their buffers: every output, the workspace, the status
word and the bias buffer are views into larger allocations whose guard
regions hold a fixed byte pattern, and the caches must come back bit for bit
as they were except for the new rows at write_idx ("ONNX Domain Attention
(Opset 23/24) CUDA Patterns", section 11: the external cache is updated only
at the write positions).  Each kernel family runs once with the guards in
place: the decode kernel (materialised bias; fused specification with the
extra term), the single-SM prefill kernel with and without key splits, the
prefill on CTA pairs, the SIMT kernel in fp32, and the bias builder.
"""
import pytest
import torch

from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from gpu_path import spec_of

GUARD = 8192  # bytes on each side (keeps every view 256-byte aligned)
PATTERN = 0xA5

PAIR_SHAPE = wl.Workload("canary_pair", 323, B=2, Hq=8, Hkv=4, D=256, S_q=700, max_seq=2048,
                         dtype=torch.bfloat16, causal=True, window=500, nonpad_fixed=1900)


class Guarded:
    """A tensor view of ``nbytes`` bytes in the middle of a pattern-filled allocation."""

    def __init__(self, shape, dtype, device="cuda"):
        n = 1
        for d in shape:
            n *= d
        self.nbytes = n * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.view = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape) if n else \
            torch.empty(shape, dtype=dtype, device=device)

    def guards_intact(self) -> bool:
        torch.cuda.synchronize()
        head, tail = self.raw[:GUARD], self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _expected_caches(inp):
    """The caches after the scatter, by indexing on the device (a bit copy)."""
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    S = inp.k_new.shape[2]
    for b in range(inp.w.B):
        s = int(inp.write_idx[b])
        k[b, :, s:s + S] = inp.k_new[b]
        v[b, :, s:s + S] = inp.v_new[b]
    return k, v


CASES = [
    ("decode_bias", wl.small(wl.C2), "bias", ek.ALGO_DECODE_STREAMK),
    ("decode_fused_extra", wl.small(wl.C4).replace(extra=True), "fused", ek.ALGO_DECODE_STREAMK),
    ("decode_cluster_bias", wl.small(wl.C2), "bias", ek.ALGO_DECODE_CLUSTER),
    ("decode_cluster_fused_extra", wl.small(wl.C4).replace(extra=True), "fused", ek.ALGO_DECODE_CLUSTER),
    ("prefill_bias", wl.small(wl.C3), "bias", ek.ALGO_PREFILL),
    ("prefill_splits_extra", wl.small(wl.C5), "fused", ek.ALGO_PREFILL),
    ("prefill_pair", PAIR_SHAPE, "bias", ek.ALGO_PREFILL_PAIR),
    ("generic_f32", wl.C1_PREFILL, "bias", ek.ALGO_GENERIC),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,w,mode,algo", CASES, ids=[c[0] for c in CASES])
def test_attention_with_scatter_writes_only_its_outputs(name, w, mode, algo):
    inp = wl.make_inputs(w, "cuda")
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    k_exp, v_exp = _expected_caches(inp)
    spec = spec_of(inp)
    bias = None
    if mode == "bias":
        gb = Guarded((w.B, 1, w.S_q, w.max_seq), w.dtype)
        ek.build_static_cache_bias(gb.view, spec, inp.nonpad)
        assert gb.guards_intact(), "the bias builder wrote outside the bias"
        bias = gb.view
    y = Guarded((w.B, w.Hq, w.S_q, w.dv), w.dtype)
    nws = ek.attention_ext_kv_workspace_size(w.B, w.Hq, w.Hkv, w.S_q, w.max_seq, w.D, w.dtype)
    ws = Guarded((nws,), torch.uint8)
    st = Guarded((4,), torch.int32)
    st.view.zero_()
    with ek.use_algo(algo):
        ek.attention_ext_kv_scatter(y.view, inp.q, k, v, inp.k_new, inp.v_new, inp.write_idx, inp.nonpad,
                                    w.scale, bias=bias, fused=spec if mode == "fused" else None,
                                    workspace=ws.view if nws else None, status=st.view)
        kernel = ek.extkv_last_kernel()
    assert ek.extkv_read_status(st.view) == ek.EXTKV_OK, ek.extkv_last_error()
    assert y.guards_intact(), f"{kernel} wrote outside Y"
    assert ws.guards_intact(), f"{kernel} wrote outside its workspace"
    assert st.guards_intact(), f"{kernel} wrote outside the status word"
    # the caches: the new rows and nothing else
    assert torch.equal(k.view(torch.int16) if k.dtype == torch.bfloat16 else k.view(torch.int32),
                       k_exp.view(torch.int16) if k.dtype == torch.bfloat16 else k_exp.view(torch.int32))
    assert torch.equal(v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32),
                       v_exp.view(torch.int16) if v.dtype == torch.bfloat16 else v_exp.view(torch.int32))
    assert torch.isfinite(y.view.float()).all()
    if algo == ek.ALGO_PREFILL_PAIR:
        assert kernel == "attn_prefill_tcgen05_pair"
