"""The seeded inputs shared by the oracle and the GPU path (no GPU needed).

They carry none of the method's arithmetic; these tests hold them to the recipe:
every tensor i.i.d. N(0,1) (the model of §3.2.1 footnote 4) drawn in fp32 from
its own seed (Q 1000 + c, K 2000 + c, V 3000 + c, dO 4000 + c for configuration
c) and rounded to bf16; the saturation variant's Q exactly four times the
encoder's; the workload table equal to the five configurations; the FLOP
convention 4 B h n m d_k (halved when causal, backward 2.5 times that).
"""
import math

import torch

from seeded_inputs import (WORKLOADS, Workload, kv_lengths, normal_bf16, visible_pairs,
                           workload_inputs)


def test_inputs_are_deterministic_and_seeded_per_tensor():
    w = Workload("t", 2, 3, 40, 24, 64, 64, False, 9)
    a = workload_inputs(w, with_grad=True)
    b = workload_inputs(w, with_grad=True)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    q, k, v, do = a
    assert torch.equal(q, normal_bf16((2, 3, 40, 64), 1009))
    assert torch.equal(k, normal_bf16((2, 3, 24, 64), 2009))
    assert torch.equal(v, normal_bf16((2, 3, 24, 64), 3009))
    assert torch.equal(do, normal_bf16((2, 3, 40, 64), 4009))
    # four different seeds: no two tensors share their draws
    assert not torch.equal(q[..., :24, :], do[..., :24, :])
    assert not torch.equal(k, v)


def test_draws_are_standard_normal_rounded_to_bf16():
    x = normal_bf16((1 << 20,), 123)
    f = x.double()
    assert abs(f.mean().item()) < 5e-3
    assert abs(f.std().item() - 1.0) < 5e-3
    # the values are exactly what bf16 rounding of the fp32 draw gives
    g = torch.Generator().manual_seed(123)
    ref = torch.randn((1 << 20,), generator=g, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(x, ref)


def test_saturation_variant_is_four_times_the_encoder_queries():
    enc, sat = WORKLOADS["encoder"], WORKLOADS["encoder_sat"]
    assert sat.q_mult == 4.0 and (sat.B, sat.h, sat.n, sat.m, sat.d_k, sat.cfg) == \
        (enc.B, enc.h, enc.n, enc.m, enc.d_k, enc.cfg)
    shape = (1, 2, enc.n, enc.d_k)
    q = normal_bf16(shape, 1000 + enc.cfg)
    q4 = normal_bf16(shape, 1000 + sat.cfg, sat.q_mult)
    # x 4 is a power of two: exact before and after the bf16 rounding
    assert torch.equal(q4.float(), 4.0 * q.float())


def test_workload_table_matches_the_configurations():
    def shape(name):
        w = WORKLOADS[name]
        return (w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal)

    assert shape("tiny") == (2, 2, 16, 16, 64, 64, False)
    assert shape("tiny_causal") == (2, 2, 16, 16, 64, 64, True)
    assert shape("encoder") == (96, 8, 256, 256, 64, 64, False)
    assert shape("decoder") == (96, 8, 256, 256, 64, 64, True)
    assert shape("cross") == (48, 16, 256, 320, 64, 64, False)
    assert shape("cross_h4_d128") == (48, 4, 256, 320, 128, 128, False)
    assert shape("cross_h16_d32") == (48, 16, 256, 320, 32, 32, False)
    for n in (1024, 4096, 16384):
        for d in (64, 128):
            for tag, causal in (("nc", False), ("c", True)):
                assert shape(f"long_n{n}_d{d}_{tag}") == (4, 16, n, n, d, d, causal)
    # d_model = h * d_k: 512 for the base model, 1024 for the big one, 512 for the variants
    assert WORKLOADS["encoder"].h * WORKLOADS["encoder"].d_k == 512
    assert WORKLOADS["cross"].h * WORKLOADS["cross"].d_k == 1024
    assert WORKLOADS["cross_h4_d128"].h * 128 == 512 and WORKLOADS["cross_h16_d32"].h * 32 == 512


def test_flop_convention():
    enc = WORKLOADS["encoder"]
    assert enc.fwd_flops() == 4.0 * 96 * 8 * 256 * 256 * 64 == 12884901888.0
    assert WORKLOADS["decoder"].fwd_flops() == enc.fwd_flops() / 2
    assert enc.bwd_flops() == 2.5 * enc.fwd_flops()
    assert WORKLOADS["cross"].fwd_flops() == 4.0 * 48 * 16 * 256 * 320 * 64
    assert enc.default_scale == 1.0 / math.sqrt(64)


def test_visible_pairs_brute_force():
    """The pair count behind the windowed and padded FLOP figures, against a
    double loop over (i, j) on small sizes."""
    for n, m in ((7, 7), (9, 5), (5, 12)):
        for causal in (False, True):
            for window in (None, (2, 1), (3, -1), (-1, 0)):
                for mb in (0, 1, m // 2, m):
                    wl, wr = window if window is not None else (-1, -1)
                    ref = sum(1 for i in range(n) for j in range(m)
                              if j < mb and (not causal or j <= i)
                              and (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr))
                    assert visible_pairs(n, m, causal, window, mb) == ref, (n, m, causal, window, mb)
    # causal n = m: the lower triangle with its diagonal
    assert visible_pairs(256, 256, True, None, 256) == 256 * 257 // 2


def test_padded_lengths_are_seeded_and_in_range():
    w = WORKLOADS["encoder_kpad"]
    lens = kv_lengths(w)
    assert lens == kv_lengths(w) and len(lens) == w.B
    assert all(w.kv_len_min <= L <= w.m for L in lens)
    assert len(set(lens)) > 1
    assert kv_lengths(WORKLOADS["encoder"]) is None
    # the padded FLOP count uses the real keys
    assert w.fwd_flops() == 4.0 * w.h * w.n * w.d_k * sum(lens)
