"""Every kernel family on the library built with EXTKV_CHECKED (device bounds
checks that flag EXTKV_DEV_BOUNDS and skip the access), against the oracle.
Run as its own process by tests/test_gpu_checked.py, so that this library,
not libextkv.so, is the one loaded.  Any flag in a call's status word fails
that call (run_gpu reads the status); prints "checked ok <calls>" at the end."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import torch  # noqa: E402

from biased_gqa_attention_gb300 import build  # noqa: E402
from biased_gqa_attention_gb300 import extkv as ek  # noqa: E402

lib = ek.load(build.build(checked=True))
assert os.path.basename(lib._name) == "libextkv_checked.so", lib._name

from biased_gqa_attention_gb300 import workloads as wl  # noqa: E402
from gpu_path import TOL, max_err, oracle_path, run_gpu  # noqa: E402

B1 = wl.Workload("chk_b1", 601, B=1, Hq=16, Hkv=8, D=256, S_q=1, max_seq=2048, dtype=torch.bfloat16,
                 causal=True, window=0, nonpad_fixed=2000)
RG = wl.Workload("chk_rg", 602, B=3, Hq=32, Hkv=2, D=128, S_q=1, max_seq=1024, dtype=torch.bfloat16,
                 causal=True, window=300, nonpad_range=(1, 1024))
MIXED = wl.Workload("chk_dk128_dv256", 603, B=2, Hq=8, Hkv=4, D=128, Dv=256, S_q=1, max_seq=512,
                    dtype=torch.bfloat16, causal=True, window=100, nonpad_range=(1, 512))
PACKED = wl.Workload("chk_packed", 604, B=2, Hq=16, Hkv=2, D=128, S_q=3, max_seq=512, dtype=torch.bfloat16,
                     causal=True, window=200, nonpad_range=(3, 512))
PAIR = wl.Workload("chk_pair", 605, B=2, Hq=8, Hkv=4, D=256, S_q=700, max_seq=2048, dtype=torch.bfloat16,
                   causal=True, window=500, nonpad_fixed=1900)

CASES = [
    (wl.small(wl.C2), ek.ALGO_DECODE_CLUSTER, ("bias", "fused", "none")),
    (B1, ek.ALGO_DECODE_CLUSTER, ("bias", "fused")),            # several clusters per unit + merge
    (wl.small(wl.C2), ek.ALGO_DECODE_STREAMK, ("bias", "fused", "none")),
    (wl.small(wl.C4).replace(extra=True), ek.ALGO_DECODE_STREAMK, ("bias", "fused")),
    (RG, ek.ALGO_DECODE_STREAMK, ("bias", "fused")),            # row groups
    (RG, ek.ALGO_DECODE_CLUSTER, ("bias", "fused")),
    (MIXED, ek.ALGO_DECODE, ("bias", "fused")),                 # two head sizes (no scatter)
    (wl.small(wl.C3), ek.ALGO_PREFILL, ("bias", "fused")),      # spans, a window
    (wl.small(wl.C5), ek.ALGO_PREFILL, ("bias", "fused")),      # key splits + merge, extra term
    (PACKED, ek.ALGO_PREFILL, ("bias", "fused")),               # packed query rows
    (PAIR, ek.ALGO_PREFILL_PAIR, ("bias",)),                    # CTA pairs
    (wl.C1_PREFILL, ek.ALGO_AUTO, ("bias", "fused")),           # fp32: the generic kernel
    (wl.small(wl.C2), ek.ALGO_GENERIC, ("bias",)),
]

calls = 0
for w, algo, modes in CASES:
    inp = wl.make_inputs(w, "cuda")
    scatter = w.dv == w.D
    for mode in modes:
        g = run_gpu(inp, mode=mode, algo=algo, scatter=scatter)  # asserts the status word is clean
        o = oracle_path(inp, mode=mode, scatter=scatter)
        err = max_err(g["y"], o["y"])
        assert err <= TOL[w.dtype], f"{w.name} {mode} {g['kernel']}: {err}"
        calls += 1
        print(f"{w.name} {mode} {g['kernel']}: ok", flush=True)

# the scatter fused into the attention call, on both decode kernels
for algo in (ek.ALGO_DECODE_CLUSTER, ek.ALGO_DECODE_STREAMK):
    w = wl.small(wl.C2)
    inp = wl.make_inputs(w, "cuda")
    ref = run_gpu(inp, mode="bias", algo=algo)
    k, v = inp.k_cache.clone(), inp.v_cache.clone()
    y = torch.empty_like(inp.q)
    st = ek.new_status()
    with ek.use_algo(algo):
        ek.attention_ext_kv_scatter(y, inp.q, k, v, inp.k_new, inp.v_new, inp.write_idx, inp.nonpad, w.scale,
                                    bias=ref["bias"], status=st)
    assert ek.extkv_read_status(st) == ek.EXTKV_OK, ek.extkv_last_error()
    assert torch.equal(y.view(torch.int16), ref["y"].view(torch.int16))
    assert torch.equal(k.view(torch.int16), ref["k"].view(torch.int16))
    calls += 1
    print(f"fused scatter {ek.extkv_last_kernel()}: ok", flush=True)

print(f"checked ok {calls}")
