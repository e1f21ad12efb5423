"""Restricted self-attention (a window of keys around each query) on the GPU
against the fp64 oracle.

"Attention Is All You Need" §4 and Table 1: each output position attends to
a neighbourhood of size r around it, cost O(r n d). Query i sees key j iff
i - left <= j <= i + right (a negative side is open), on top of the causal
mask and key padding. The cases cover every kernel that runs: the per-item
forward with 64- and 128-key tiles, d = 32, 64, 128, the whole-head and the
general backward, causal local attention, one open side, a window of one
position, key padding with an empty sequence, and rows whose window misses
every key (n > m: the empty sum).
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import Workload, workload_inputs
from tests.parity_utils import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # (B, h, n, m, d, causal, (left, right), kv_len)
    (2, 2, 256, 256, 64, False, (64, 64), None),         # 64-key tiles, whole-head bwd
    (1, 2, 700, 700, 64, False, (100, 37), None),        # 128-key tiles, general bwd, ragged
    (1, 2, 300, 300, 128, True, (50, -1), None),         # causal local, d = 128
    (2, 2, 256, 200, 32, False, (10, 300), None),        # n > m: rows past m + 10 see nothing
    (2, 1, 256, 512, 64, False, (0, 0), None),           # one position: O_i = v_i
    (3, 2, 200, 256, 64, False, (30, 30), [256, 100, 0]),  # key padding, an empty sequence
    (1, 1, 1100, 1100, 64, True, (200, 0), None),        # long causal local, ragged
    (1, 1, 64, 1000, 64, False, (-1, 500), None),        # open left side, whole-head bwd, m >> n
]


def _run(q, k, v, do, causal, scale, window, lens):
    kvl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = A.attn_fwd(qd, kd, vd, causal=causal, scale=scale, kv_len=kvl, window=window)
    dq, dk, dv = A.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, kv_len=kvl, window=window)
    assert A.attn_get_device_status() == A.ATTN_OK
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_window_matches_oracle(case):
    B, h, n, m, d, causal, window, lens = CASES[case]
    w = Workload(f"win{case}", B, h, n, m, d, d, causal, 110 + case)
    q, k, v, do = workload_inputs(w, with_grad=True)
    scale = w.default_scale
    o, lse, dq, dk, dv = _run(q, k, v, do, causal, scale, window, lens)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(q, k, v, do, causal, scale, kv_len=lens, window=window)
    empty = np.isneginf(rlse)
    lse64 = lse.double().numpy()
    # rows without a visible key: lse = -inf and O = 0 exactly
    assert np.array_equal(np.isneginf(lse64), empty)
    assert (o.double().numpy()[empty] == 0).all()
    assert_close("O", o, ro)
    assert_close("lse", np.where(empty, 0.0, lse64), np.where(empty, 0.0, rlse))
    # the rows at a window's edges see few keys: gradients there are held to the
    # documented exception for differences of few large terms
    ex = "few_term_cancellation"
    assert_close("dQ", dq, rdq, allow=ex)
    assert_close("dK", dk, rdk, allow=ex)
    assert_close("dV", dv, rdv, allow=ex)


def test_window_covering_everything_equals_no_window_bitwise():
    """A window wider than the sequence takes the per-item kernel but must give
    the very bytes of the unwindowed call whenever that call takes it too
    (causal, so both run the same kernel)."""
    w = Workload("winall", 2, 2, 300, 300, 64, 64, True, 130)
    q, k, v, do = (t.to(DEV) for t in workload_inputs(w, with_grad=True))
    o0, l0 = A.attn_fwd(q, k, v, causal=True)
    o1, l1 = A.attn_fwd(q, k, v, causal=True, window=(300, 300))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    g0 = A.attn_bwd(q, k, v, o0, l0, do, causal=True)
    g1 = A.attn_bwd(q, k, v, o1, l1, do, causal=True, window=(400, 5000))
    for a, b in zip(g0, g1):
        assert torch.equal(a, b)
    assert A.attn_get_device_status() == A.ATTN_OK


def test_keys_outside_every_window_are_never_read():
    """Bitwise: keys and values that no query's window reaches do not change any result."""
    w = Workload("winout", 1, 2, 256, 1024, 64, 64, False, 131)
    q, k, v, do = workload_inputs(w, with_grad=True)
    window = (20, 20)  # queries 0..255 reach keys 0..275 only
    o0, l0, dq0, dk0, dv0 = _run(q, k, v, do, False, w.default_scale, window, None)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 384:] = 30.0
    v2[:, :, 384:] = -5.0
    o1, l1, dq1, dk1, dv1 = _run(q, k2, v2, do, False, w.default_scale, window, None)
    assert torch.equal(o0, o1) and torch.equal(l0, l1) and torch.equal(dq0, dq1)
    assert torch.equal(dk0[:, :, :384], dk1[:, :, :384]) and torch.equal(dv0[:, :, :384], dv1[:, :, :384])
    assert (dk1[:, :, 276:] == 0).all() and (dv1[:, :, 276:] == 0).all()
