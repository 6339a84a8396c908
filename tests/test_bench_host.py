"""Host-side logic of bench.py (CPU only): the algorithmic-work accounting and
the multi-rank timing reduction (world size 2 over gloo)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
import oracle
from biased_gqa_attention_gb300 import workloads as wl

LOW = {"f32": 0xFF7FFFFF, "bf16": 0xFF7F}


@pytest.mark.parametrize("w", [wl.C1_PREFILL, wl.C2, wl.C3, wl.small(wl.C3), wl.C4,
                               wl.small(wl.C5)], ids=lambda w: w.name)
def test_allowed_counts_match_the_oracle_bias(w):
    nonpad, _, spans = wl.structure(w)
    dt = "f32" if w.dtype == torch.float32 else "bf16"
    b, _ = oracle.bias(nonpad.numpy(), w.S_q, w.max_seq, dt, causal=w.causal, window=w.window,
                       spans=spans if any(spans) else None)
    bits = b.view(np.uint32) if dt == "f32" else b
    counts = (bits != LOW[dt]).sum(axis=-1)[:, 0, :]
    assert (bench.allowed_counts(w, nonpad.numpy(), spans) == counts).all()


def test_c2_step_bytes_close_to_expected():
    nonpad, _, spans = wl.structure(wl.C2)
    ab, _ = bench.attention_work(wl.C2, nonpad.numpy(), spans, "bias")
    kv = sum(min(int(n), 1024) for n in nonpad) * 8 * 256 * 2 * 2
    assert ab == kv + 2 * 8 * 16 * 256 * 2 + int(nonpad.sum()) * 2


def test_c3_flops_closed_form():
    nonpad, _, spans = wl.structure(wl.C3)
    _, f = bench.attention_work(wl.C3, nonpad.numpy(), spans, "bias")
    assert f == 4 * 256 * 16 * (2048 * 1024 + 3 * sum(255 - k for k in range(256)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, local, wsz = bench.dist_env()
    bench.dist_init(wsz, "gloo")
    t = 1.0 + rank  # rank 1 is the slowest
    tmax = bench.reduce_max(t, wsz)
    bench.barrier(wsz)
    v = bench.whole_job_value(100.0, wsz, tmax)
    q.put((r, local, wsz, tmax, v))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, local, world, tmax, v) in enumerate(res):
        assert (rank, local, world) == (r, r, 2)
        assert tmax == 2.0
        assert v == pytest.approx(100.0 * 2 / 2.0)


def test_reference_arm_reports_the_same_config_as_ours(capsys):
    """bench.py --impl reference (the oracle on the host cores) prints one JSON
    line whose config is the dict the repo's arm builds for the same workload."""
    import json
    import bench
    w = wl.C1_DECODE
    bench.main(["--impl", "reference", "--workload", w.name, "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    nonpad, _, spans = wl.structure(w)
    sb = bench.step_bytes(w, nonpad.numpy(), spans, "bias")
    assert line["impl"] == "reference"
    assert line["config"] == bench.step_config(w, "bias", 1, True, sb)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
