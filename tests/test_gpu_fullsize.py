"""Full-size parity for every configuration of the workload list, in the launch
configuration the benchmark times (one attn_fwd + one attn_bwd over the whole batch).

The oracle computes sampled outputs one by one: forward rows and dQ rows of
sampled queries, dK / dV rows of sampled keys (these need a full forward of
their head). Sequences of 4096 and more rows are sampled deeper: 8 heads, both
rows at every 128-row tile boundary, the last tile and a uniform sample (at
least 256 query rows), and 64 key rows. Properties that hold at any size are
checked on every head.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import WORKLOADS, workload_inputs
from tests.parity_utils import assert_close, to64
from tests.test_gpu_parity import invariant_bounds

pytestmark = pytest.mark.gpu

FULL = ["tiny", "tiny_causal", "encoder", "encoder_sat", "decoder", "cross", "cross_h4_d128",
        "cross_h16_d32"] + [f"long_n{n}_d{d}_{c}" for n in (1024, 4096, 16384) for d in (64, 128)
                            for c in ("nc", "c")]


def _sample(size, extra, rng, boundaries=False):
    """Tile-boundary rows plus a uniform sample; returns (rows, positions of the uniform part)."""
    edge = {0, 1, 127, 128, 129, 255, 256, size - 2, size - 1}
    if boundaries:  # both rows at every 128-row tile boundary, and the whole last partial tile's ends
        edge |= {b + o for b in range(128, size, 128) for o in (-1, 0)}
        edge |= {(size - 1) // 128 * 128}
    uni = set(rng.choice(size, size=min(size, extra), replace=False).tolist())
    rows = sorted(i for i in edge | uni if 0 <= i < size)
    return rows, [p for p, i in enumerate(rows) if i in uni]


def _exception(w, tensor):
    """The documented exception a tensor of this workload is held to (None: the plain bound)."""
    if tensor not in ("dQ", "dK", "dV"):
        return None
    if w.q_mult != 1.0:
        return "saturated_softmax_backward"
    if w.causal:
        return "few_term_cancellation"
    return None


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name):
    w = WORKLOADS[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    q, k, v, do = workload_inputs(w, with_grad=True)
    qd, kd, vd, dod = (t.to("cuda") for t in (q, k, v, do))
    scale = w.default_scale
    o, lse = A.attn_fwd(qd, kd, vd, causal=w.causal, scale=scale)
    dq, dk, dv = A.attn_bwd(qd, kd, vd, o, lse, dod, causal=w.causal, scale=scale)
    assert A.attn_get_device_status() == A.ATTN_OK

    H = w.heads
    deep = w.n >= 4096
    if deep:
        heads = sorted(set(np.linspace(0, H - 1, 8).round().astype(int).tolist()))
        key_heads = heads
        n_uni, k_uni = 256, 64
    else:
        heads = sorted({0, H - 1, H // 2})
        key_heads = heads if w.n * w.m <= 4096 * 4096 else [H // 2]
        n_uni, k_uni = 48, 24
    o3, lse3 = o.view(H, w.n, w.d_v), lse.view(H, w.n)
    dq3, dk3, dv3 = dq.view(H, w.n, w.d_k), dk.view(H, w.m, w.d_k), dv.view(H, w.m, w.d_v)
    q3, k3, v3, do3 = (t.view(H, t.shape[2], t.shape[3]) for t in (q, k, v, do))
    for h in heads:
        rows, uni = _sample(w.n, n_uni, rng, boundaries=deep)
        assert not deep or len(rows) >= 256
        ro, rl = oracle.fwd(q3[h], k3[h], v3[h], w.causal, scale, rows=rows)
        assert_close(f"{name} O head {h}", o3[h, rows], ro[rows], rel_rows=uni)
        assert_close(f"{name} lse head {h}", lse3[h, rows][None], rl[rows][None], rel_rows=None)
        krows, kuni = _sample(w.m, k_uni, rng) if h in key_heads else ([], [])
        rdq, rdk, rdv = oracle.bwd_rows(q3[h], k3[h], v3[h], do3[h], w.causal, scale, rows, krows)
        assert_close(f"{name} dQ head {h}", dq3[h, rows], rdq, rel_rows=uni, allow=_exception(w, "dQ"))
        if krows:
            assert_close(f"{name} dK head {h}", dk3[h, krows], rdk, rel_rows=kuni, allow=_exception(w, "dK"))
            assert_close(f"{name} dV head {h}", dv3[h, krows], rdv, rel_rows=kuni, allow=_exception(w, "dV"))

    # invariants on every head: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, within the
    # rounding budget of bf16 arithmetic
    dkk, dvv = to64(dk3), to64(dv3)
    tol_k, tol_v = invariant_bounds(to64(q3), to64(v3), to64(do3), dkk, dvv, scale)
    assert (np.abs(dkk.sum(axis=1)) <= tol_k).all(), name
    assert (np.abs(dvv.sum(axis=1) - to64(do3).sum(axis=1)) <= tol_v).all(), name
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
