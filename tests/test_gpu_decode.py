"""Incremental decoding (one step over a key/value cache) on the GPU against the
fp64 oracle.

"Attention Is All You Need" §3: the decoder emits one symbol at a time; each
step attends to the positions produced so far, itself included. Sequence b has
L_b cached positions; its n newest are the queries, query i seeing keys
j <= L_b - n + i. The cases cover one query and sixteen, d = 32, 64, 128, long
caches split over many CTAs, ragged and empty caches, fewer cached positions
than queries, a cache of one position, and a negative scale; and the
benchmark's decoding steps at full size, sampled by head.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import DECODE_WORKLOADS, normal_bf16
from tests.parity_utils import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # (B, h, n, m, d, kv_len, scale multiplier)
    (4, 8, 1, 4096, 64, None, 1.0),             # long cache, one query, many chunks
    (3, 2, 4, 1000, 64, [1000, 517, 3], 1.0),   # ragged; the last has fewer positions than queries
    (2, 4, 16, 300, 128, None, 1.0),            # sixteen queries, d = 128
    (2, 2, 8, 100, 32, [100, 64], 1.0),         # d = 32, two chunks or fewer
    (1, 1, 1, 1, 64, None, 1.0),                # a cache of one position
    (2, 3, 2, 777, 64, [0, 777], 1.0),          # an empty cache: the empty sum
    (2, 2, 3, 2500, 64, [2500, 1999], -0.5),    # a negative scale
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_matches_oracle(case):
    B, h, n, m, d, lens, mult = CASES[case]
    q = normal_bf16((B, h, n, d), 2100 + case)
    k = normal_bf16((B, h, m, d), 2200 + case)
    v = normal_bf16((B, h, m, d), 2300 + case)
    scale = mult / np.sqrt(d)
    kvl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = A.attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), kv_len=kvl, scale=scale)
    assert A.attn_get_device_status() == A.ATTN_OK
    ro, rlse = oracle.decode(q, k, v, scale, kv_len=lens)
    empty = np.isneginf(rlse)
    lse64 = lse.cpu().double().numpy()
    assert np.array_equal(np.isneginf(lse64), empty)
    assert (o.cpu().double().numpy()[empty] == 0).all()
    assert_close("O", o.cpu(), ro)
    assert_close("lse", np.where(empty, 0.0, lse64), np.where(empty, 0.0, rlse))


def test_decode_equals_causal_forward_rows():
    """The decoding step of the last n positions and the causal forward over the
    whole sequence agree (both against the oracle's causal rows)."""
    B, h, S, n, d = 2, 4, 640, 4, 64
    q = normal_bf16((B, h, S, d), 2400)
    k = normal_bf16((B, h, S, d), 2401)
    v = normal_bf16((B, h, S, d), 2402)
    o_step, l_step = A.attn_decode(q[:, :, S - n:].contiguous().to(DEV), k.to(DEV), v.to(DEV))
    o_full, l_full = A.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    ro, rlse = oracle.fwd(q, k, v, True, 1 / np.sqrt(d), rows=list(range(S - n, S)))
    assert_close("O step", o_step.cpu(), ro[:, :, S - n:])
    assert_close("O full", o_full[:, :, S - n:].cpu(), ro[:, :, S - n:])
    assert_close("lse step", l_step.cpu(), rlse[:, :, S - n:])


def test_decode_argument_checks():
    q = torch.zeros(1, 1, 17, 64, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 1, 32, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(A.AttnError):
        A.attn_decode(q, k, k)  # n > 16
    q = torch.zeros(1, 1, 1, 64, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(4, dtype=torch.float32, device=DEV)
    with pytest.raises(A.AttnError):
        A.attn_decode(q, k, k, workspace=ws)  # workspace too small


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_full_size_sampled(name):
    """The benchmark's decoding steps at their full sizes (the whole batch in one
    call, as timed): eight heads spread over the batch, first and last included,
    against the oracle's step on those heads."""
    B, h, n, m, d = DECODE_WORKLOADS[name]
    q = normal_bf16((B, h, n, d), 2500)
    k = normal_bf16((B, h, m, d), 2501)
    v = normal_bf16((B, h, m, d), 2502)
    scale = 1 / np.sqrt(d)
    o, lse = A.attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale)
    assert A.attn_get_device_status() == A.ATTN_OK
    o, lse = o.cpu(), lse.cpu()
    for bh in sorted(set(np.linspace(0, B * h - 1, 8).round().astype(int).tolist())):
        b, hh = divmod(bh, h)
        sl = (slice(b, b + 1), slice(hh, hh + 1))
        ro, rlse = oracle.decode(q[sl], k[sl], v[sl], scale)
        assert_close(f"{name} O head {bh}", o[sl], ro)
        assert_close(f"{name} lse head {bh}", lse[sl], rlse)
