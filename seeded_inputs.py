"""Seeded synthetic inputs for scaled dot-product attention.

This module only draws random numbers and names workload shapes. It holds none
of the attention arithmetic, so both the CUDA path and the fp64 oracle can be
fed from it without sharing any of the method.

Input model: every tensor is i.i.d. N(0, 1), drawn in fp32 on the CPU from a
``torch.Generator`` with a fixed seed and rounded to bf16 (round-to-nearest-even).
That is the footnote-4 model of "Attention Is All You Need" §3.2.1 (query and
key components independent with mean 0 and variance 1). The pages measure on
WMT 2014 EN-DE / EN-FR batches (§5.1, roughly 25000 source + 25000 target
tokens per batch); no dataset is used here, the shapes below stand in for them:
base model h=8, d_k=d_v=64 (§3.2.2), big model h=16 with d_model=1024
(Table 3 "big" row), and the Table 3 (A) head shapes (h, d_k) = (4, 128) and
(16, 32). 96 sequences x 256 tokens ~ 24.6k tokens matches the batch size.
"""
from __future__ import annotations

import dataclasses
import functools
import math
from typing import Dict, Iterator, List, Optional, Tuple

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "normal_bf16",
    "workload_inputs",
    "ragged_workloads",
    "kv_lengths",
    "DECODE_WORKLOADS",
    "PROJ_WORKLOADS",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: B sequences x h heads, n queries, m keys."""

    name: str
    B: int
    h: int
    n: int
    m: int
    d_k: int
    d_v: int
    causal: bool
    cfg: int  # seed family: Q=1000+cfg, K=2000+cfg, V=3000+cfg, dO=4000+cfg
    q_mult: float = 1.0  # power-of-two multiplier applied before the bf16 cast
    # key padding: 0 = none; else sequence b has kv_len[b] real keys, drawn
    # uniformly from [kv_len_min, m] (seed 5000+cfg), see kv_lengths()
    kv_len_min: int = 0
    # restricted self-attention (§4, Table 1): query i sees keys
    # i - window[0] .. i + window[1] (-1: open side); None = no window
    window: Optional[Tuple[int, int]] = None

    @property
    def heads(self) -> int:
        return self.B * self.h

    @property
    def default_scale(self) -> float:
        # 1/sqrt(d_k): the scale named in §3.2.1 (uses d_k, not d_v)
        return 1.0 / math.sqrt(self.d_k)

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs: 4*B*h*n*m*d_k, halved when causal.

        With key padding (non-causal only) m is replaced by each sequence's
        real key count: 4*h*n*d_k*sum_b kv_len[b]. With a window the count is
        4*d_k per visible (query, key) pair, the pairs counted exactly.
        """
        lens = kv_lengths(self)
        if self.window is not None:
            per_seq = [visible_pairs(self.n, self.m, self.causal, self.window, L)
                       for L in (lens if lens is not None else [self.m] * self.B)]
            return 4.0 * self.h * self.d_k * float(sum(per_seq))
        if lens is not None:
            if self.causal:
                raise ValueError("padded workloads are non-causal")
            return 4.0 * self.h * self.n * self.d_k * float(sum(lens))
        f = 4.0 * self.B * self.h * self.n * self.m * self.d_k
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """Algorithmic backward FLOPs: 2.5x the forward count (five GEMMs)."""
        return 2.5 * self.fwd_flops()


def _wl(name, B, h, n, m, d, causal, cfg, q_mult=1.0, kv_len_min=0, window=None) -> Workload:
    return Workload(name, B, h, n, m, d, d, causal, cfg, q_mult, kv_len_min, window)


@functools.lru_cache(maxsize=None)
def visible_pairs(n: int, m: int, causal: bool, window, mb: int) -> int:
    """Number of (query, key) pairs with key j visible to query i: j < mb,
    j <= i when causal, i - window[0] <= j <= i + window[1] (negative: open)."""
    total = 0
    wl, wr = window if window is not None else (-1, -1)
    for i in range(n):
        hi = mb
        if causal:
            hi = min(hi, i + 1)
        if wr >= 0:
            hi = min(hi, i + wr + 1)
        lo = max(0, i - wl) if wl >= 0 else 0
        total += max(0, hi - lo)
    return total


def _build_table() -> Dict[str, Workload]:
    t: List[Workload] = [
        _wl("tiny", 2, 2, 16, 16, 64, False, 1),
        _wl("tiny_causal", 2, 2, 16, 16, 64, True, 1),
        _wl("encoder", 96, 8, 256, 256, 64, False, 2),
        _wl("encoder_sat", 96, 8, 256, 256, 64, False, 2, q_mult=4.0),
        _wl("decoder", 96, 8, 256, 256, 64, True, 3),
        _wl("cross", 48, 16, 256, 320, 64, False, 4),
        _wl("cross_h4_d128", 48, 4, 256, 320, 128, False, 4),
        _wl("cross_h16_d32", 48, 16, 256, 320, 32, False, 4),
        # variable-length batch (§5.1 batches sentences of similar length;
        # <pad> keys of Figure 3): real key counts uniform in [128, 256]
        _wl("encoder_kpad", 96, 8, 256, 256, 64, False, 6, kv_len_min=128),
    ]
    for n in (1024, 4096, 16384):
        for d in (64, 128):
            for causal in (False, True):
                tag = "c" if causal else "nc"
                t.append(_wl(f"long_n{n}_d{d}_{tag}", 4, 16, n, n, d, causal, 5))
    # restricted self-attention (§4, Table 1: a neighbourhood of size r around
    # each position): r = 257 centred, and causal local attention over the
    # 256 previous positions, on the long-sequence shape
    t.append(_wl("long_n16384_d64_band257", 4, 16, 16384, 16384, 64, False, 9, window=(128, 128)))
    t.append(_wl("long_n16384_d64_local256", 4, 16, 16384, 16384, 64, True, 9, window=(256, -1)))
    return {w.name: w for w in t}


WORKLOADS: Dict[str, Workload] = _build_table()


# One incremental decoding step (§3: one output symbol per step) over a
# key/value cache: (B sequences, h heads, n new positions, m cached positions,
# d). B = 64 stands for a batch of 16 sentences with beam 4 (§6.1 beam size);
# n = 4 for four positions per step; the big model's h = 16 heads of d = 64.
DECODE_WORKLOADS: Dict[str, Tuple[int, int, int, int, int]] = {
    "decode_b64_h16_n1_m4096_d64": (64, 16, 1, 4096, 64),
    "decode_b64_h16_n4_m4096_d64": (64, 16, 4, 4096, 64),
    "decode_b16_h16_n1_m16384_d128": (16, 16, 1, 16384, 128),
}


# The projections around eq. (1) (§3.2.2): (B, n query tokens, m key tokens,
# d_model, h, d). The base model's encoder self-attention batch and the big
# model's encoder-decoder attention (queries from 256 decoder tokens, keys and
# values from 320 encoder tokens).
PROJ_WORKLOADS: Dict[str, Tuple[int, int, int, int, int, int]] = {
    "proj_base_self_b96_n256": (96, 256, 256, 512, 8, 64),
    "proj_big_cross_b48_n256_m320": (48, 256, 320, 1024, 16, 64),
}


def normal_bf16(shape, seed: int, mult: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """i.i.d. N(0,1) drawn in fp32 from ``seed``, times ``mult``, rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    x = x.to(torch.bfloat16)
    return x if device == "cpu" else x.to(device)


def workload_inputs(w: Workload, with_grad: bool = False, device: str = "cpu",
                    heads: Optional[int] = None):
    """Q, K, V (and dO) for workload ``w`` in the [B, h, S, d] layout, bf16.

    ``heads`` (optional) truncates the batch to the first ``heads`` (b, h)
    pairs of a [1, heads, S, d] view; the values are the same bytes as the
    corresponding heads of the full tensors only when heads == B*h, so it is
    meant for bounded CPU samples, not for parity against full runs.
    """
    B, h = (w.B, w.h) if heads is None else (1, heads)
    q = normal_bf16((B, h, w.n, w.d_k), 1000 + w.cfg, w.q_mult, device)
    k = normal_bf16((B, h, w.m, w.d_k), 2000 + w.cfg, 1.0, device)
    v = normal_bf16((B, h, w.m, w.d_v), 3000 + w.cfg, 1.0, device)
    if not with_grad:
        return q, k, v
    do = normal_bf16((B, h, w.n, w.d_v), 4000 + w.cfg, 1.0, device)
    return q, k, v, do


def ragged_workloads() -> Iterator[Workload]:
    """Small shapes that are not tile multiples: ragged tails, n != m, m = 1."""
    cases = [
        (1, 1, 1, 1, 64, False), (1, 1, 1, 1, 64, True),
        (1, 2, 17, 17, 64, True), (2, 1, 127, 129, 64, False),
        (1, 3, 129, 127, 64, True), (1, 2, 320, 320, 64, True),
        (2, 2, 200, 77, 32, False), (1, 2, 130, 300, 128, False),
        (1, 1, 255, 257, 128, True), (1, 1, 64, 1, 32, False),
        (3, 1, 300, 300, 32, True), (1, 1, 5, 400, 64, False),
        # whole 128-key tiles, non-causal (the persistent forward): a partial
        # second query tile, a query block whose second tile is empty, and a
        # long ragged key sequence
        (2, 3, 200, 256, 64, False), (1, 2, 130, 128, 32, False),
        (1, 1, 384, 1024, 64, False), (1, 2, 100, 1100, 64, False),
    ]
    for i, (B, h, n, m, d, c) in enumerate(cases):
        yield _wl(f"ragged{i}_B{B}h{h}n{n}m{m}d{d}{'c' if c else ''}", B, h, n, m, d, c, 50 + i)


def kv_lengths(w: Workload) -> Optional[List[int]]:
    """Real keys per sequence of a padded workload (None: no key padding)."""
    if w.kv_len_min <= 0:
        return None
    g = torch.Generator(device="cpu")
    g.manual_seed(5000 + w.cfg)
    return torch.randint(w.kv_len_min, w.m + 1, (w.B,), generator=g).tolist()
