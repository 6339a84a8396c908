"""Seeded synthetic workloads for biased GQA attention over a static KV cache.

This module only draws inputs; it holds none of the method's arithmetic.  Both
the CUDA path's tests/bench and the oracle receive exactly the tensors drawn
here.

Recipe (the same for every workload):
  * Structure (nonpad_kv_seqlen, write offsets, image spans) is drawn with a
    CPU ``torch.Generator`` seeded ``1000 + config_id``, so it is identical on
    every machine and device.
  * Values are drawn N(0, 1) in fp32 with a generator on the target device,
    seeded the same, then cast to the element type with round-to-nearest-even.
    Draw order: q, k_new, v_new, past K cache, past V cache, garbage K, garbage
    V, extra.  Garbage (slots at or beyond nonpad) is N(0, sigma^2) with the
    workload's sigma, or NaN in the poisoned variant.
  * scale = 1/sqrt(D).  Masked bias entries hold the element type's lowest
    finite value; the bias itself is built by the library/oracle, not here.

Workload shapes follow the Gemma-4-like decoder layers the pages discuss
("Skill: Attention Optimization": sliding-window local layers, head_dim 512
global layers, KV-shared layers; mobius issue #366: vision-block overlay).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    B: int
    Hq: int
    Hkv: int
    D: int
    S_q: int
    max_seq: int
    dtype: torch.dtype
    causal: bool = True
    window: int = 0  # <= 0: no sliding window
    # nonpad / write offsets
    nonpad_fixed: Optional[int] = None     # every batch has this nonpad
    nonpad_range: Optional[Tuple[int, int]] = None  # uniform inclusive range
    offset_range: Optional[Tuple[int, int]] = None  # write offset range; nonpad = offset + S_q
    # bidirectional image spans: count, length, allowed start range (inclusive)
    n_spans: int = 0
    span_len: int = 0
    span_start_range: Optional[Tuple[int, int]] = None
    extra: bool = False          # dense additive term on allowed slots
    garbage_sigma: float = 1.0   # N(0, sigma^2) beyond nonpad
    kv_shared: bool = False      # a second call attends the borrowed cache
    Dv: Optional[int] = None     # value head size when it differs from D (the q/k head size)
    description: str = ""

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def dv(self) -> int:
        return self.D if self.Dv is None else self.Dv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  C1's two steps are two workloads sharing one cache.
C1_PREFILL = Workload(
    "tiny_f32_prefill", 1, B=1, Hq=4, Hkv=2, D=64, S_q=16, max_seq=64, dtype=torch.float32,
    causal=True, nonpad_fixed=16,
    description="fp32 prefill: 16 tokens scattered at slots 0-15, nonpad=16, causal bias")
C1_DECODE = Workload(
    "tiny_f32_decode", 1, B=1, Hq=4, Hkv=2, D=64, S_q=1, max_seq=64, dtype=torch.float32,
    causal=True, nonpad_fixed=17,
    description="fp32 decode: one token at slot 16, nonpad=17, causal bias")
C2 = Workload(
    "decode_b8_hq16_hkv8_d256_w1024", 2, B=8, Hq=16, Hkv=8, D=256, S_q=1, max_seq=4096,
    dtype=torch.bfloat16, causal=True, window=1024, nonpad_range=(512, 4096),
    description="bf16 decode, new token at nonpad-1, causal + sliding window 1024")
C3 = Workload(
    "prefill_s2048_hq16_hkv8_d256_w1024_spans", 3, B=1, Hq=16, Hkv=8, D=256, S_q=2048,
    max_seq=8192, dtype=torch.bfloat16, causal=True, window=1024, nonpad_fixed=4096,
    n_spans=3, span_len=256, span_start_range=(2048, 4096 - 256),
    description="bf16 prefill chunk at slots 2048-4095, causal + window 1024 + 3 image spans")
C4 = Workload(
    "decode_b32_hq16_hkv2_d512", 4, B=32, Hq=16, Hkv=2, D=512, S_q=1, max_seq=8192,
    dtype=torch.bfloat16, causal=True, nonpad_range=(1, 8192), garbage_sigma=10.0,
    description="bf16 global-layer decode, group 8, head_dim 512, causal + padding")
C5 = Workload(
    "prefill_s128_hq8_hkv4_d128_w4096_extra_kvshared", 5, B=4, Hq=8, Hkv=4, D=128, S_q=128,
    max_seq=16384, dtype=torch.bfloat16, causal=True, window=4096, offset_range=(0, 16000),
    extra=True, kv_shared=True,
    description="bf16 prefill at random offsets, causal + window 4096 + dense term, then KV-shared")

ALL = [C1_PREFILL, C1_DECODE, C2, C3, C4, C5]

# Decode steps at the edges of the decode kernel's shapes, measured and tested
# beside the five workloads: 512 batches (larger than its default shared-memory
# tables, sized per call), and 16 query heads per KV head (more than the 8 query
# rows of a decode unit: such steps run on the prefill kernel).
DECODE_B512 = Workload(
    "decode_b512_hq16_hkv8_d256_w1024", 6, B=512, Hq=16, Hkv=8, D=256, S_q=1, max_seq=4096,
    dtype=torch.bfloat16, causal=True, window=1024, nonpad_range=(512, 4096),
    description="C2 at 512 batches (per-call tables larger than the default 256 batches)")
DECODE_G16 = Workload(
    "decode_b8_hq32_hkv2_d128_w1024", 7, B=8, Hq=32, Hkv=2, D=128, S_q=1, max_seq=4096,
    dtype=torch.bfloat16, causal=True, window=1024, nonpad_range=(512, 4096),
    description="decode with 16 query heads per KV head (beyond the decode kernel's 8 rows per unit)")
CLIFFS = [DECODE_B512, DECODE_G16]

BY_NAME = {w.name: w for w in ALL + CLIFFS}


def small(w: Workload) -> Workload:
    """A smaller workload of the same structure (group size, mask kinds,
    ragged tails) that the oracle finishes in well under a second."""
    if w.config_id == 1:
        return w
    if w.config_id == 2:
        return w.replace(name=w.name + "_small", B=3, max_seq=1000, window=200, nonpad_range=(130, 1000))
    if w.config_id == 3:
        return w.replace(name=w.name + "_small", Hq=4, Hkv=2, S_q=300, max_seq=1200, window=150,
                         nonpad_fixed=700, n_spans=2, span_len=70, span_start_range=(400, 630))
    if w.config_id == 4:
        return w.replace(name=w.name + "_small", B=4, max_seq=1000, nonpad_range=(1, 1000))
    if w.config_id == 5:
        return w.replace(name=w.name + "_small", B=3, S_q=77, max_seq=1200, window=300,
                         offset_range=(0, 1100))
    if w.config_id == 6:  # still beyond 256 batches
        return w.replace(name=w.name + "_small", B=300, max_seq=512, window=200, nonpad_range=(1, 512))
    if w.config_id == 7:
        return w.replace(name=w.name + "_small", B=3, max_seq=1000, window=200, nonpad_range=(130, 1000))
    raise ValueError(w)


@dataclasses.dataclass
class Inputs:
    w: Workload
    q: torch.Tensor          # (B,Hq,S_q,D)
    k_new: torch.Tensor      # (B,Hkv,S_new,D)
    v_new: torch.Tensor
    k_cache: torch.Tensor    # (B,Hkv,max_seq,D), before the scatter
    v_cache: torch.Tensor
    write_idx: torch.Tensor  # (B,) int64
    nonpad: torch.Tensor     # (B,) int64
    spans: List[List[Tuple[int, int]]]
    span_offsets: Optional[torch.Tensor]  # (B+1,) int64 or None
    span_table: Optional[torch.Tensor]    # (n,2) int64 or None
    extra: Optional[torch.Tensor]         # (B,1,S_q,max_seq) or None

    @property
    def S_new(self) -> int:
        return self.k_new.shape[2]


def structure(w: Workload):
    gen = torch.Generator(device="cpu").manual_seed(1000 + w.config_id)
    B, S_q = w.B, w.S_q
    if w.nonpad_fixed is not None:
        nonpad = torch.full((B,), w.nonpad_fixed, dtype=torch.int64)
    elif w.nonpad_range is not None:
        lo, hi = w.nonpad_range
        nonpad = torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64)
    else:
        lo, hi = w.offset_range
        nonpad = torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64) + S_q
    # the new rows are the last S_q valid slots: [nonpad - S_q, nonpad)
    write_idx = nonpad - S_q
    spans: List[List[Tuple[int, int]]] = [[] for _ in range(B)]
    if w.n_spans:
        lo, hi = w.span_start_range
        for b in range(B):
            tries = 0
            while len(spans[b]) < w.n_spans:
                tries += 1
                if tries > 100000:  # the spans drawn so far leave no room for another
                    raise ValueError(f"{w.name}: cannot place {w.n_spans} disjoint spans of {w.span_len} "
                                     f"with starts in [{lo}, {hi}]")
                s = int(torch.randint(lo, hi + 1, (1,), generator=gen))
                if all(s + w.span_len <= t or t + w.span_len <= s for t, _ in spans[b]):
                    spans[b].append((s, w.span_len))
            spans[b].sort()
    return nonpad, write_idx, spans


def make_inputs(w: Workload, device="cpu", poison: bool = False) -> Inputs:
    """Draw one seeded instance of ``w`` on ``device``.

    ``poison`` fills every slot at or beyond nonpad of both caches with NaN
    (the pages' poison-V tests: such slots must never reach the output).
    """
    device = torch.device(device)
    nonpad, write_idx, spans = structure(w)
    gen = torch.Generator(device=device).manual_seed(1000 + w.config_id)

    def draw(shape, sigma=1.0):
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        return x.to(w.dtype)

    B, Hq, Hkv, D, S_q, L, Dv = w.B, w.Hq, w.Hkv, w.D, w.S_q, w.max_seq, w.dv
    q = draw((B, Hq, S_q, D))
    k_new = draw((B, Hkv, S_q, D))
    v_new = draw((B, Hkv, S_q, Dv))
    k_cache = draw((B, Hkv, L, D))
    v_cache = draw((B, Hkv, L, Dv))
    gk = draw((B, Hkv, L, D), w.garbage_sigma)
    gv = draw((B, Hkv, L, Dv), w.garbage_sigma)
    beyond = (torch.arange(L, device=device)[None, :] >= nonpad.to(device)[:, None])  # (B,L)
    sel = beyond[:, None, :, None]
    if poison:
        gk.fill_(float("nan"))
        gv.fill_(float("nan"))
    k_cache = torch.where(sel, gk, k_cache).contiguous()
    v_cache = torch.where(sel, gv, v_cache).contiguous()
    del gk, gv
    extra = draw((B, 1, S_q, L)) if w.extra else None
    if w.n_spans:
        offs = [0]
        flat = []
        for lst in spans:
            flat.extend(lst)
            offs.append(len(flat))
        span_offsets = torch.tensor(offs, dtype=torch.int64, device=device)
        span_table = torch.tensor(flat, dtype=torch.int64, device=device).reshape(-1, 2)
    else:
        span_offsets = span_table = None
    return Inputs(w, q, k_new, v_new, k_cache, v_cache, write_idx.to(device), nonpad.to(device),
                  spans, span_offsets, span_table, extra)


def c1_chain(device="cpu"):
    """The tiny fp32 case: one cache shared by the prefill step and the decode
    step that follows it (decode token drawn after the prefill tensors)."""
    pre = make_inputs(C1_PREFILL, device)
    gen = torch.Generator(device=torch.device(device)).manual_seed(1000 + 1 + 7919)
    dec_q = torch.randn((1, 4, 1, 64), generator=gen, device=device)
    dec_k = torch.randn((1, 2, 1, 64), generator=gen, device=device)
    dec_v = torch.randn((1, 2, 1, 64), generator=gen, device=device)
    dec = Inputs(C1_DECODE, dec_q, dec_k, dec_v, None, None,
                 torch.tensor([16], dtype=torch.int64, device=device),
                 torch.tensor([17], dtype=torch.int64, device=device),
                 [[]], None, None, None)
    return pre, dec
