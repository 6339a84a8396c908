#!/usr/bin/env python
"""Benchmark of the external-KV biased GQA attention hot path on GB300.

One step = the whole hot path over one batch of the decode workload
(B=8, Hq=16, Hkv=8, D=256, S_q=1, max_seq=4096, nonpad ~ U[512,4096], causal +
sliding window 1024, bf16): TensorScatter of the new K/V rows, the
(B,1,S_q,max_seq) bias build, and attention over the static cache.

Prints ONE JSON line (rank 0).  `value` is whole-job algorithmic GB/s with the
inputs resident in HBM (for a prefill workload given with --workload: the
attention's algorithmic TFLOP/s); `e2e` is the same metric through the public
API with pinned host inputs copied in and the output copied out every step.
The `roofline` object covers the attention kernel (the dominant one);
`secondary` adds the other workloads' attention calls (prefill in TFLOP/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica (weak scaling: independent
batches, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from biased_gqa_attention_gb300 import workloads as wl  # noqa: E402

METRIC = "ext-KV biased GQA attn: decode HBM GB/s, prefill TFLOP/s (% of GB300 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# distributed plumbing (host logic; covered by a gloo test on CPU)

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, local, world


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------------------------
# algorithmic work (what the method must move or compute; no skipped work is
# counted and no redundant work is credited)

def allowed_counts(w: wl.Workload, nonpad: np.ndarray, spans) -> np.ndarray:
    """|U| per (b, i): allowed keys of each query row, from the workload's
    causal / window / span structure (the definition of the bias)."""
    out = np.zeros((w.B, w.S_q), np.int64)
    for b in range(w.B):
        npb = int(nonpad[b])
        qs = max(npb - w.S_q, 0)
        p = qs + np.arange(w.S_q, dtype=np.int64)
        band_lo = p - w.window + 1 if w.window > 0 else np.full_like(p, -(1 << 40))
        band_hi = p + 1 if w.causal else np.full_like(p, 1 << 40)
        lo = np.clip(band_lo, 0, npb)
        hi = np.clip(band_hi, 0, npb)
        cnt = np.maximum(hi - lo, 0)
        for (s, L) in spans[b]:
            inside = (p >= s) & (p < s + L)
            s_lo, s_hi = np.clip(s, 0, npb), np.clip(s + L, 0, npb)
            extra = np.maximum(s_hi - np.maximum(s_lo, hi), 0) + np.maximum(np.minimum(s_hi, lo) - s_lo, 0)
            cnt = np.where(inside, cnt + extra, cnt)
        out[b] = cnt
    return out


def attention_work(w: wl.Workload, nonpad: np.ndarray, spans, mode: str):
    """(bytes, flops) of one attention call.

    Decode: K and V rows of every allowed slot once per KV head (the group's
    query heads share them), Q in, Y out, and, with a materialised bias, the
    bias row over the valid slots.  Prefill flops: 4*D per (query head, allowed
    key) pair (QK^T and PV)."""
    es = 4 if w.dtype == torch.float32 else 2
    U = allowed_counts(w, nonpad, spans)
    if w.S_q == 1:
        kv = int(U[:, 0].sum()) * w.Hkv * w.D * es * 2
    else:
        kv = 0
        for b in range(w.B):  # union of the rows' key sets, read once
            kv += min(int(nonpad[b]), int(U[b].max()) + w.S_q) * w.Hkv * w.D * es * 2
    qy = 2 * w.B * w.Hq * w.S_q * w.D * es
    bias = int(nonpad.sum()) * w.S_q * es if mode == "bias" else 0
    extra = int(U.sum()) * es if (w.extra and mode == "fused") else 0
    flops = 4.0 * w.D * w.Hq * float(U.sum())
    return kv + qy + bias + extra, flops


def step_bytes(w: wl.Workload, nonpad: np.ndarray, spans, mode: str) -> int:
    es = 4 if w.dtype == torch.float32 else 2
    scatter = 2 * 2 * w.B * w.Hkv * w.S_q * w.D * es  # K and V, read + write
    bias = w.B * w.S_q * w.max_seq * es if mode == "bias" else 0
    if mode == "bias" and w.extra:
        bias *= 2
    attn, _ = attention_work(w, nonpad, spans, mode)
    return scatter + bias + attn


def step_work(w: wl.Workload, nonpad: np.ndarray, spans, mode: str):
    """(amount, scale, unit) of the metric for one step: algorithmic GB/s of
    the whole step for decode, the attention's algorithmic TFLOP/s for a
    prefill chunk (the tensor-bound part; the scatter and the bias build are
    byte-bound and reported in their own kernels' shares)."""
    if w.S_q > 1:
        _, flops = attention_work(w, nonpad, spans, mode)
        return flops, 1e12, "TFLOP/s"
    return step_bytes(w, nonpad, spans, mode), 1e9, "GB/s"


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.bus = None
        try:
            props = torch.cuda.get_device_properties(device)
            dom = getattr(props, "pci_domain_id", 0)
            self.bus = f"{dom:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
        except Exception:
            pass
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            if self.bus and parts[0].upper() not in (self.bus.upper(), self.bus.upper()[4:]):
                if not parts[0].upper().endswith(self.bus.upper()[-12:]):
                    continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm

def _rotation(touched_bytes: int, device) -> int:
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    # enough distinct input sets that the bytes touched between two uses of
    # one set exceed twice the L2 size
    return max(2, math.ceil(2 * l2 / max(touched_bytes, 1)) + 1)


class Decoder:
    """Device-resident state for one workload: R rotating input sets.

    A step is the scatter of the new rows, the bias build (materialised mode)
    and the attention: by default the bias build and attention_ext_kv_scatter
    (the scatter fused into the attention call), or, with fused_step=False, the
    three separate calls."""

    def __init__(self, w: wl.Workload, device, mode: str, sets: int, fused_step: bool = True):
        from biased_gqa_attention_gb300 import extkv as ek
        self.ek, self.w, self.mode, self.device = ek, w, mode, device
        self.fused_step = fused_step
        base = wl.make_inputs(w, device)
        self.base = base
        self.sets = []
        for r in range(sets):
            s = dict(q=base.q.clone(), k_new=base.k_new.clone(), v_new=base.v_new.clone(),
                     k=base.k_cache.clone(), v=base.v_cache.clone(), write_idx=base.write_idx.clone(),
                     nonpad=base.nonpad.clone(), y=torch.empty_like(base.q),
                     bias=torch.empty((w.B, 1, w.S_q, w.max_seq), dtype=w.dtype, device=device),
                     extra=None if base.extra is None else base.extra.clone())
            s["spec"] = ek.BiasSpec(causal=w.causal, window=w.window, span_offsets=base.span_offsets,
                                    spans=base.span_table, extra=s["extra"])
            self.sets.append(s)
        self.status = ek.new_status(device)
        self.workspace = ek.new_workspace(base.q, base.k_cache)
        # The sets were drawn and copied on the current stream, and their blocks
        # may be ones the caching allocator took back from the generator's
        # temporaries with writes still queued there; the steps run on another
        # stream, so nothing of that work may still be pending when they start.
        torch.cuda.synchronize(device)

    def scatter(self, r):
        s = self.sets[r]
        self.ek.ext_kv_scatter(s["k"], s["v"], s["k_new"], s["v_new"], s["write_idx"], status=self.status)

    def bias(self, r, stream=None):
        s = self.sets[r]
        self.ek.build_static_cache_bias(s["bias"], s["spec"], s["nonpad"], status=self.status, stream=stream)

    def attention(self, r):
        s = self.sets[r]
        self.ek.attention_ext_kv(s["y"], s["q"], s["k"], s["v"], s["nonpad"], self.w.scale,
                                 bias=s["bias"] if self.mode == "bias" else None,
                                 fused=s["spec"] if self.mode == "fused" else None,
                                 workspace=self.workspace, status=self.status)

    def attention_scatter(self, r, stream=None):
        s = self.sets[r]
        self.ek.attention_ext_kv_scatter(s["y"], s["q"], s["k"], s["v"], s["k_new"], s["v_new"], s["write_idx"],
                                         s["nonpad"], self.w.scale,
                                         bias=s["bias"] if self.mode == "bias" else None,
                                         fused=s["spec"] if self.mode == "fused" else None,
                                         workspace=self.workspace, status=self.status, stream=stream)

    def recorded_step(self, r):
        """The step's library calls for set r recorded once (extkv_step_*):
        one launch starts them all again.  The calls ran eagerly before, so
        their first-use setup is outside the recording."""
        if not self.fused_step:
            raise ValueError("recorded steps cover the fused step")
        with self.ek.StepRecorder() as rec:
            if self.mode == "bias":
                self.bias(r, stream=rec.stream)
            self.attention_scatter(r, stream=rec.stream)
        return rec.step

    def prepared_step(self, r):
        """The step's calls with their arguments marshalled once
        (extkv.prepare_*): what a caller repeating the step over the same
        buffers issues."""
        s, ek = self.sets[r], self.ek
        calls = []
        if not self.fused_step:
            raise ValueError("prepared steps cover the fused step")
        if self.mode == "bias":
            calls.append(ek.prepare_build_static_cache_bias(s["bias"], s["spec"], s["nonpad"], status=self.status))
        calls.append(ek.prepare_attention_ext_kv_scatter(
            s["y"], s["q"], s["k"], s["v"], s["k_new"], s["v_new"], s["write_idx"], s["nonpad"], self.w.scale,
            bias=s["bias"] if self.mode == "bias" else None, fused=s["spec"] if self.mode == "fused" else None,
            workspace=self.workspace, status=self.status))
        return calls

    def step(self, r):
        if not self.fused_step:
            self.scatter(r)
        if self.mode == "bias":
            self.bias(r)
        if self.fused_step:
            self.attention_scatter(r)
        else:
            self.attention(r)

    def kernels_per_step(self):
        # (scatter,) bias build, and what the attention call reported launching
        # (which counts a scatter kernel it ran ahead of an unfused path)
        return (0 if self.fused_step else 1) + (1 if self.mode == "bias" else 0) + self.ek.extkv_last_launches()


def step_config(w: wl.Workload, mode: str, world: int, fused_step: bool, sb: int) -> dict:
    """The workload and the step, as both arms report them (the same dict)."""
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "S_q": w.S_q,
            "max_seq": w.max_seq, "window": w.window, "bias_mode": mode,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "rotating input sets, >2x L2 touched between reuses of one set",
            "step": ("build_static_cache_bias + attention_ext_kv_scatter (the scatter fused into "
                     "the attention call)" if fused_step else
                     "ext_kv_scatter + build_static_cache_bias + attention_ext_kv"),
            "step_algorithmic_bytes": sb}


def time_graph(dec: Decoder, K: int, W: int, stream):
    """Warm-up W eager steps, capture K steps and replay them once untimed
    (graph upload).  Nothing but the steps' own kernels is captured: an event
    record between two kernels ends the programmatic overlap of the second
    with the first and would be timed as part of the step."""
    R = len(dec.sets)
    with torch.cuda.stream(stream):
        for i in range(W):
            dec.step(i % R)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(K):
            dec.step(k % R)
    g.replay()
    torch.cuda.synchronize()
    return g


def median_replay_ms(g, stream, replays: int = 5) -> float:
    """Median over `replays` replays of a captured graph (after one untimed
    upload replay), CUDA events on the launching stream around each."""
    times = []
    with torch.cuda.stream(stream):
        g.replay()  # upload
        for _ in range(replays):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            g.replay()
            t1.record()
            t1.synchronize()
            times.append(t0.elapsed_time(t1))
    return float(np.median(times))


def time_attention_calls(dec: Decoder, K: int, stream) -> float:
    """The step's attention call alone, max(K, 50) times back to back over the
    same rotating input sets (each set's bias is already built), captured in a
    CUDA graph; the median of 5 replays.  Returns ms per call."""
    R = len(dec.sets)
    n = max(K, 50)
    call = dec.attention_scatter if dec.fused_step else dec.attention
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(n):
            call(k % R)
    return median_replay_ms(g, stream) / n


def run_ours(args, rank, local, world):
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    from biased_gqa_attention_gb300 import build as bld
    bld.build()
    from biased_gqa_attention_gb300 import extkv as ek

    w = wl.BY_NAME[args.workload]
    nonpad, _, spans = wl.structure(w)
    nonpad = nonpad.numpy()
    sb = step_bytes(w, nonpad, spans, args.mode)
    amount, scale, unit = step_work(w, nonpad, spans, args.mode)
    prefill = w.S_q > 1
    attn_b, attn_f = attention_work(w, nonpad, spans, args.mode)
    fused_step = not args.unfused_step
    if fused_step:  # the attention call also moves the new rows (read + write, K and V)
        attn_b += 2 * 2 * w.B * w.Hkv * w.S_q * w.D * (4 if w.dtype == torch.float32 else 2)
    R = _rotation(sb, device)
    dec = Decoder(w, device, args.mode, R, fused_step=fused_step)
    stream = torch.cuda.Stream(device)
    K, W = args.steps, args.warmup

    g = time_graph(dec, K, W, stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # keep the GPU busy on the same graph for ~1 s so clock samples land under load
        tl = time.time()
        while time.time() - tl < args.clock_load_s:
            g.replay()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t0.record()
            g.replay()
            t1.record()
        torch.cuda.synchronize()
        barrier(world)
        # the dominant call on its own, under the same clocks
        attn_avg_ms = time_attention_calls(dec, K, stream)
    ms_total = t0.elapsed_time(t1)
    ms_max = reduce_max(ms_total, world, device)
    ms_per_step = ms_max / K
    value = whole_job_value(amount * K, world, ms_max / 1e3) / scale

    # status after the timed region: no device-side error may hide in the numbers
    assert ek.extkv_read_status(dec.status) == ek.EXTKV_OK, ek.extkv_last_error()
    kernel = ek.extkv_last_kernel()
    traffic = args.traffic if args.traffic is not None else NCU_TRAFFIC.get((w.name, args.mode, kernel))

    # e2e: the public API with pinned host buffers, copies inside the timed region
    e2e = run_e2e(dec, K, W, world, device)

    peaks, peak_src = read_peaks()
    roof = None
    if attn_avg_ms and prefill:
        achieved = attn_f / (attn_avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
                "kernel": kernel, "launch_us": round(attn_avg_ms * 1e3, 3),
                "algorithmic_flops": attn_f, "peak_source": peak_src}
    elif attn_avg_ms:
        achieved = attn_b / (attn_avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": kernel, "launch_us": round(attn_avg_ms * 1e3, 3),
                "algorithmic_bytes": attn_b, "peak_source": peak_src}

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) values, nonpad ~ U[512,4096]; no dataset)",
        "config": step_config(w, args.mode, world, fused_step, sb),
        "rotation_sets": R,
        "timing": ("CUDA graph of K steps, CUDA events on the launching stream around one replay; "
                   "roofline: a CUDA graph of max(K, 50) attention calls over the same sets, median of 5 "
                   "replays"),
        "gpu_launches": K * dec.kernels_per_step(),
        "roofline": roof,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, dec.base, args.mode, amount, scale, unit, args.cpu_seconds)
    if not args.no_secondary:
        out["secondary"] = secondary(args, device, peaks, peak_src)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _packed(tensors: dict, buf: torch.Tensor) -> dict:
    """Views of ``buf`` (uint8) holding each tensor of ``tensors`` at a
    256-byte-aligned offset, in the tensors' shapes and dtypes."""
    views, off = {}, 0
    for k, t in tensors.items():
        n = t.numel() * t.element_size()
        views[k] = buf[off:off + n].view(t.dtype).view(t.shape)
        off += (n + 255) & ~255
    return views


def _packed_bytes(tensors: dict) -> int:
    return sum((t.numel() * t.element_size() + 255) & ~255 for t in tensors.values())


def run_e2e(dec: Decoder, K: int, W: int, world: int, device):
    """The step through the public API with its inputs in pinned host memory:
    every step copies them to the device (one copy: the inputs are packed in
    one buffer, as a caller staging a step's inputs would), runs the step and
    reads the output back."""
    w = dec.w
    keys = ("q", "k_new", "v_new", "write_idx", "nonpad")
    s = dec.sets[0]
    nbytes = _packed_bytes({k: s[k] for k in keys})
    host_buf = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host = _packed({k: s[k] for k in keys}, host_buf)
    for k, t in host.items():
        t.copy_(s[k].cpu())
    # each rotation set's inputs become views of one device buffer
    dev_bufs = []
    for d in dec.sets:
        b = torch.empty(nbytes, dtype=torch.uint8, device=device)
        views = _packed({k: d[k] for k in keys}, b)
        for k in keys:
            views[k].copy_(d[k])
            d[k] = views[k]
        dev_bufs.append(b)
    # the buffers were filled on the current stream; the copy streams below
    # write them next, and an event nobody has recorded yet orders nothing
    torch.cuda.synchronize(device)
    R = len(dec.sets)
    y_hosts = [torch.empty(s["y"].shape, dtype=s["y"].dtype, pin_memory=True) for _ in range(R)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_hosts[0].numel() * y_hosts[0].element_size()
    compute = torch.cuda.current_stream(device)
    handle = compute.cuda_stream
    # the copies run on streams of their own, so that step k's output copy and
    # step k+1's input copy overlap the neighbouring steps' kernels; events keep
    # each input set's buffers from being overwritten while a step still uses them
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(R)]    # set r's inputs landed
    ev_done = [torch.cuda.Event() for _ in range(R)]  # set r's step finished (inputs free, output final)
    ev_read = [torch.cuda.Event() for _ in range(R)]  # set r's output copied out

    def timed(recorded: bool) -> float:
        # the library calls of each set, prepared or recorded once (the copies stay per step)
        if recorded:
            calls = [[dec.recorded_step(r)] for r in range(R)]
            calls = [[(lambda st=c[0]: st(handle))] for c in calls]
        else:
            calls = [dec.prepared_step(r) for r in range(R)]

        def one(r):
            # torch.cuda.set_stream rather than the stream context manager: the
            # latter costs ~6 us of host time per use on this host
            up.wait_event(ev_done[r])
            torch.cuda.set_stream(up)
            dev_bufs[r].copy_(host_buf, non_blocking=True)
            ev_in[r].record(up)
            compute.wait_event(ev_in[r])
            compute.wait_event(ev_read[r])
            torch.cuda.set_stream(compute)
            for c in calls[r]:
                c()
            ev_done[r].record(compute)
            down.wait_event(ev_done[r])
            torch.cuda.set_stream(down)
            y_hosts[r].copy_(dec.sets[r]["y"], non_blocking=True)
            ev_read[r].record(down)
            torch.cuda.set_stream(compute)

        for i in range(W):
            one(i % R)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for k in range(K):
            one(k % R)
        torch.cuda.synchronize()
        return reduce_max(time.perf_counter() - t0, world, device)

    sec_calls = timed(False)
    sec = timed(True)
    assert dec.ek.extkv_read_status(dec.status) == dec.ek.EXTKV_OK, dec.ek.extkv_last_error()
    # the last output of every set the loop ran reached its pinned host buffer
    for r in range(min(R, max(W, K))):
        assert torch.equal(y_hosts[r], dec.sets[r]["y"].cpu()), "an output copy did not land"
    nonpad, _, spans = wl.structure(w)
    amount, scale, unit = step_work(w, nonpad.numpy(), spans, dec.mode)
    return {"value": round(whole_job_value(amount * K, world, sec) / scale, 2), "unit": unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(sec * 1e3 / K, 4),
            "ms_per_step_prepared_calls": round(sec_calls * 1e3 / K, 4),
            "timing": "host wall clock around K steps, each: the inputs' copy from pinned host memory (a copy "
                      "stream), the step's library calls recorded once per input set (extkv_step_*: one "
                      "launch per step), the output's copy back (another copy stream), ordered by events "
                      "so that copies overlap the neighbouring steps' kernels; ms_per_step_prepared_calls: "
                      "the same with the calls issued one by one (extkv.prepare_*)"}


def secondary(args, device, peaks, peak_src):
    """The other workloads' attention calls, each timed alone: a CUDA graph of
    n calls over rotating input sets (no host launch overhead in the number),
    CUDA events on the launching stream around one replay."""
    from biased_gqa_attention_gb300 import extkv as ek
    res = {}
    stream = torch.cuda.Stream(device)
    # C3-C5, two decode steps outside the decode kernel's shapes (the cost of
    # the fallback to the prefill kernel), then C2 and C3 in the other bias mode
    other = "fused" if args.mode == "bias" else "bias"
    runs = [(w, args.mode) for w in (wl.C3, wl.C4, wl.C5, *wl.CLIFFS)] + [(wl.C2, other), (wl.C3, other)]
    for w, mode in runs:
        key = w.name if mode == args.mode else f"{w.name}@{mode}"
        nonpad, _, spans = wl.structure(w)
        nonpad = nonpad.numpy()
        ab, af = attention_work(w, nonpad, spans, mode)
        touched = ab if w.S_q == 1 else ab + w.B * w.S_q * w.max_seq * 2
        R = min(_rotation(touched, device), 6)
        dec = Decoder(w, device, mode, R)
        with torch.cuda.stream(stream):
            for r in range(R):
                dec.scatter(r)
                if mode == "bias":
                    dec.bias(r)
            for i in range(3):
                dec.attention(i % R)
        torch.cuda.synchronize()
        n = 50
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                dec.attention(i % R)
        ms = median_replay_ms(g, stream) / n
        assert ek.extkv_read_status(dec.status) == ek.EXTKV_OK, ek.extkv_last_error()
        if w.S_q == 1:
            ach = ab / (ms / 1e3) / 1e9
            res[key] = {"bound": "hbm", "achieved": round(ach, 1), "unit": "GB/s",
                           "peak": peaks["hbm_gbs"], "frac": round(ach / peaks["hbm_gbs"], 4),
                           "launch_us": round(ms * 1e3, 2), "kernel": ek.extkv_last_kernel(),
                           "launches": ek.extkv_last_launches(), "algorithmic_bytes": ab}
        else:
            ach = af / (ms / 1e3) / 1e12
            res[key] = {"bound": "tensor", "achieved": round(ach, 2), "unit": "TFLOP/s",
                           "peak": peaks["bf16_tflops"], "frac": round(ach / peaks["bf16_tflops"], 4),
                           "launch_us": round(ms * 1e3, 2), "kernel": ek.extkv_last_kernel(),
                           "launches": ek.extkv_last_launches(), "algorithmic_flops": af}
        res[key]["peak_source"] = peak_src
        res[key]["timing"] = f"CUDA graph of {n} attention calls over {R} rotating input sets, median of 5 replays"
        del dec, g
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)

def _oracle_inputs(w: wl.Workload, base):
    """Host copies of one input set in the oracle's raw element types."""
    def raw(t):
        t = t.detach().contiguous().cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16).copy()
        return t.numpy().copy()
    return {k: (None if getattr(base, k) is None else raw(getattr(base, k)))
            for k in ("q", "k_new", "v_new", "k_cache", "v_cache", "write_idx", "nonpad", "extra")}


def oracle_step(w: wl.Workload, h, spans, mode: str):
    import oracle
    dt = "f32" if w.dtype == torch.float32 else "bf16"
    oracle.scatter(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], h["write_idx"])
    b = None
    if mode in ("bias", "fused"):
        b, _ = oracle.bias(h["nonpad"], w.S_q, w.max_seq, dt, causal=w.causal, window=w.window,
                           spans=spans if any(spans) else None, extra=h["extra"])
    return oracle.attention(h["q"], h["k_cache"], h["v_cache"], b, h["nonpad"], np.float32(w.scale))


def cpu_baseline(w, base, mode, amount, scale, unit, seconds):
    import oracle
    _, _, spans = wl.structure(w)
    h = _oracle_inputs(w, base)
    oracle_step(w, h, spans, mode)  # warm-up (also builds the oracle library)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(w, h, spans, mode)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": round(amount * n / el / scale, 6), "unit": unit, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"{n} full steps of {w.name} (scatter + bias + attention over "
            f"all rows), {el:.1f} s, fp64, OpenMP over query rows"}


def run_reference(args, rank, local, world):
    """The oracle as it stands, on the host cores, for the same workload and metric."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.BY_NAME[args.workload]
    base = wl.make_inputs(w, "cpu")
    nonpad, _, spans = wl.structure(w)
    sb = step_bytes(w, nonpad.numpy(), spans, args.mode)
    amount, scale, unit = step_work(w, nonpad.numpy(), spans, args.mode)
    h = _oracle_inputs(w, base)
    for _ in range(args.warmup):
        oracle_step(w, h, spans, args.mode)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, h, spans, args.mode)
    el = time.perf_counter() - t0
    value = amount * args.steps / el / scale
    out = {"metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) values; no dataset)", "impl": "reference",
           "config": step_config(w, args.mode, world, not args.unfused_step, sb),
           "timing": "host wall clock around the oracle's steps, one input set",
           "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": f"{args.steps} full steps of {w.name}"},
           "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant kernel, per
# (workload, mode, the name extkv_last_kernel() reports), from an ncu capture of the kernel as
# committed (the capture's summary under profiles/ names the template).  A call that runs another
# kernel finds no entry (traffic null); a change to a kernel makes its entry stale: drop it.
NCU_TRAFFIC = {
    # attn_decode_cluster_kernel<256, 256, 3, 1, 0> (the step's call, with the fused scatter)
    ("decode_b8_hq16_hkv8_d256_w1024", "bias", "attn_decode_cluster_scatter"): 65.22e6,
    # attn_prefill_kernel<256, 256, 1, 0>
    ("prefill_s2048_hq16_hkv8_d256_w1024_spans", "bias", "attn_prefill_tcgen05"): 43.00e6,
}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.C2.name, choices=sorted(wl.BY_NAME))
    ap.add_argument("--mode", choices=["bias", "fused"], default="bias")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--unfused-step", action="store_true",
                    help="time the step as three calls (ext_kv_scatter, bias build, attention_ext_kv)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--clock-load-s", type=float, default=1.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel (default: the committed capture "
                         "for this workload and mode, if any)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, local, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, local, world)
    else:
        run_ours(args, rank, local, world)


if __name__ == "__main__":
    main()
