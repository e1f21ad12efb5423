"""Full-size parity for every configuration of the workload list, in the launch
configuration the benchmark times (one attn_fwd + one attn_bwd over the whole batch).

The oracle computes sampled outputs one by one: forward rows and dQ rows of
sampled queries, dK / dV rows of sampled keys (these need a full forward of
their head). Properties that hold at any size are checked on every head.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import WORKLOADS, workload_inputs
from tests.parity_utils import assert_close, d_term_bounds, to64
from tests.test_gpu_parity import invariant_bounds

pytestmark = pytest.mark.gpu

FULL = ["tiny", "tiny_causal", "encoder", "encoder_sat", "decoder", "cross", "cross_h4_d128",
        "cross_h16_d32"] + [f"long_n{n}_d{d}_{c}" for n in (1024, 4096, 16384) for d in (64, 128)
                            for c in ("nc", "c")]


def _sample(size, extra, rng):
    """Tile-boundary rows plus a uniform sample; returns (rows, positions of the uniform part)."""
    edge = {0, 1, 127, 128, 129, 255, 256, size - 2, size - 1}
    uni = set(rng.choice(size, size=min(size, extra), replace=False).tolist())
    rows = sorted(i for i in edge | uni if 0 <= i < size)
    return rows, [p for p, i in enumerate(rows) if i in uni]


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
    heads = sorted({0, H - 1, H // 2})
    key_heads = heads if w.n * w.m <= 4096 * 4096 else [H // 2]
    o3, lse3 = o.view(H, w.n, w.d_v), lse.view(H, w.n)
    dq3, dk3, dv3 = dq.view(H, w.n, w.d_k), dk.view(H, w.m, w.d_k), dv.view(H, w.m, w.d_v)
    q3, k3, v3, do3 = (t.view(H, t.shape[2], t.shape[3]) for t in (q, k, v, do))
    for h in heads:
        rows, uni = _sample(w.n, 48, rng)
        ro, rl = oracle.fwd(q3[h], k3[h], v3[h], w.causal, scale, rows=rows)
        assert_close(f"O head {h}", o3[h, rows], ro[rows], rel_rows=uni)
        assert_close(f"lse head {h}", lse3[h, rows][None], rl[rows][None], rel_rows=None)
        krows, kuni = _sample(w.m, 24, rng) if h in key_heads else ([], [])
        rdq, rdk, rdv = oracle.bwd_rows(q3[h], k3[h], v3[h], do3[h], w.causal, scale, rows, krows)
        bq, bk = d_term_bounds(q3[h], k3[h], v3[h], do3[h], w.causal, scale, rows, krows)
        # the saturated Q x 4 variant: D_i from the bf16 O dominates the small gradients
        rel = 1e-2 if w.q_mult != 1.0 else 5e-3
        assert_close(f"dQ head {h}", dq3[h, rows], rdq, grad=True, rel_rows=uni, extra=bq, rel_l2=rel)
        if krows:
            assert_close(f"dK head {h}", dk3[h, krows], rdk, grad=True, rel_rows=kuni, extra=bk,
                         rel_l2=rel)
            assert_close(f"dV head {h}", dv3[h, krows], rdv, grad=True, rel_rows=kuni, rel_l2=rel)

    # invariants on every head: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, within the
    # rounding budget of bf16 arithmetic
    dkk, dvv = to64(dk3), to64(dv3)
    tol_k, tol_v = invariant_bounds(to64(q3), to64(v3), to64(do3), dkk, dvv, scale)
    assert (np.abs(dkk.sum(axis=1)) <= tol_k).all(), name
    assert (np.abs(dvv.sum(axis=1) - to64(do3).sum(axis=1)) <= tol_v).all(), name
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
