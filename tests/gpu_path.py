"""Runs one workload through the CUDA path (C ABI via the binding) and through
the oracle, on identical inputs.  Used by the GPU parity tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from biased_gqa_attention_gb300 import extkv as ek
from biased_gqa_attention_gb300 import workloads as wl
from helpers import dt_name, raw

TOL = {torch.float32: 1e-5, torch.bfloat16: 1.5e-2}


def spec_of(inp: wl.Inputs) -> ek.BiasSpec:
    w = inp.w
    return ek.BiasSpec(causal=w.causal, window=w.window, span_offsets=inp.span_offsets,
                       spans=inp.span_table, extra=inp.extra)


def run_gpu(inp: wl.Inputs, mode: str = "bias", algo: int = ek.ALGO_AUTO, scatter: bool = True,
            k_cache=None, v_cache=None, softcap: float = 0.0):
    """mode: 'bias' (materialised), 'fused' (in-register spec) or 'none'.  A
    workload whose value head size differs from D attends its caches as they
    are (no scatter: the new rows of K and V have different sizes)."""
    w = inp.w
    assert not (scatter and w.dv != w.D), "no scatter with two head sizes"
    k = (inp.k_cache if k_cache is None else k_cache).clone()
    v = (inp.v_cache if v_cache is None else v_cache).clone()
    st = ek.new_status()
    if scatter:
        ek.ext_kv_scatter(k, v, inp.k_new, inp.v_new, inp.write_idx, status=st)
    spec = spec_of(inp)
    bias = None
    if mode == "bias":
        bias = torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device=inp.q.device)
        ek.build_static_cache_bias(bias, spec, inp.nonpad, status=st)
    y = torch.empty((w.B, w.Hq, w.S_q, w.dv), dtype=w.dtype, device=inp.q.device)
    with ek.use_algo(algo):
        ek.attention_ext_kv(y, inp.q, k, v, inp.nonpad, w.scale, bias=bias,
                            fused=spec if mode == "fused" else None, status=st, softcap=softcap)
        kernel = ek.extkv_last_kernel()
    code = ek.extkv_read_status(st)
    assert code == ek.EXTKV_OK, ek.extkv_last_error()
    return dict(k=k, v=v, bias=bias, y=y, kernel=kernel)


def oracle_path(inp: wl.Inputs, rows=None, mode: str = "bias", scatter: bool = True,
                k_cache=None, v_cache=None, softcap: float = 0.0):
    """The oracle on host copies of the same inputs: scatter, bias, attention.
    ``k_cache``/``v_cache`` optionally replace the workload's caches with numpy
    arrays the oracle produced earlier (never with GPU results)."""
    w = inp.w
    dt = dt_name(w.dtype)
    kc = raw(inp.k_cache) if k_cache is None else np.array(k_cache, copy=True)
    vc = raw(inp.v_cache) if v_cache is None else np.array(v_cache, copy=True)
    if scatter:
        assert oracle.scatter(kc, vc, raw(inp.k_new), raw(inp.v_new), raw(inp.write_idx)) == 0
    nonpad = raw(inp.nonpad)
    spans = inp.spans if any(len(s) for s in inp.spans) else None
    extra = raw(inp.extra) if inp.extra is not None else None
    bias, bad = oracle.bias(nonpad, w.S_q, w.max_seq, dt, causal=w.causal, window=w.window,
                            spans=spans, extra=extra)
    assert bad == 0
    y = oracle.attention(raw(inp.q), kc, vc, bias if mode != "none" else None, nonpad,
                         np.float32(w.scale), rows=rows, softcap=softcap)
    return dict(k=kc, v=vc, bias=bias, y=y)


def max_err(y_gpu: torch.Tensor, y_ref: np.ndarray, rows=None) -> float:
    g = y_gpu.detach().to(torch.float64).cpu().numpy()
    if rows is not None:
        g = g.reshape(-1, g.shape[-1])[rows]
    assert np.isfinite(g).all(), "non-finite GPU output"
    return float(np.abs(g - y_ref).max()) if g.size else 0.0


def sample_rows(w: wl.Workload, n: int, seed: int = 0) -> np.ndarray:
    """Rows to check at full size: first, last, every batch's first/last row,
    plus seeded random rows."""
    total = w.B * w.Hq * w.S_q
    if total <= n:
        return np.arange(total, dtype=np.int64)
    rng = np.random.default_rng(seed)
    fixed = {0, total - 1}
    for b in range(w.B):
        fixed.add(b * w.Hq * w.S_q)
        fixed.add((b + 1) * w.Hq * w.S_q - 1)
    extra = rng.choice(total, size=max(0, n - len(fixed)), replace=False)
    return np.array(sorted(fixed | set(extra.tolist())), dtype=np.int64)
