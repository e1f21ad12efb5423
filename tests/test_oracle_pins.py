"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test ties the oracle to something the pages print, a closed form, an
invariant of eq. (1), brute-force finite differences, or an independent
library routine. A plausible slip in the oracle (a dropped scale, a wrong
mask index, a transposed operand, a sign error in the backward) fails at
least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from seeded_inputs import normal_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _half_unit(printed: str) -> float:
    """Half a unit in the last printed digit ("4.0" -> 0.05, "66" -> 0.5)."""
    if "." in printed:
        return 0.5 * 10.0 ** (-len(printed.split(".")[1]))
    return 0.5


def _read_rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- printed values

def test_worked_example_scores_and_weights():
    """The 2-d example of the close-reading page (query "它" over seven keys).

    Scores q.k/sqrt(2) and weights must match the printed values to the
    printed precision.
    """
    rows = _read_rows("worked_example_2d.txt")
    q = np.array([[float(rows[0][1]), float(rows[0][2])]])
    assert rows[1][0] == "scale_denominator_sqrt"
    scale = 1.0 / math.sqrt(float(rows[1][1]))
    keys = rows[2:]
    K = np.array([[float(r[1]), float(r[2])] for r in keys])
    S, P = oracle.weights(q, K, causal=False, scale=scale)
    for j, r in enumerate(keys):
        assert abs(S[0, j] - float(r[3])) <= _half_unit(r[3]) + 1e-12, (r, S[0, j])
        assert abs(100.0 * P[0, j] - float(r[4])) <= _half_unit(r[4]) + 1e-12, (r, P[0, j])
    # the printed weights are those of one softmax row: they add up to 100 %
    assert abs(P.sum() - 1.0) < 1e-15


def test_saturation_example_weights_and_derivative():
    """Scores 8 and 0 at d_k=64: weights ~0.9997, derivative ~0.0003; /8: 0.73/0.27, ~0.20.

    The derivative p(1-p) of the softmax weight with respect to its own score
    is read off the oracle's backward: with v_a = 1, v_b = 0 (d_v = 1) the
    output is O = p_a, and with dO = 1 and k_b = 0 the query gradient is
    dQ = scale * dS_a * k_a, where dS_a = dO/ds_a = p_a (1 - p_a).
    """
    for r in _read_rows("saturation.txt"):
        dk, sa, sb, scale = int(r[0]), float(r[1]), float(r[2]), float(r[3])
        wa, wb, dp, tol_w, tol_dp = map(float, r[4:9])
        assert sb == 0.0
        q = np.zeros((1, dk))
        q[0, 0] = sa                      # q . k_a = sa with k_a = e_0
        K = np.zeros((2, dk))
        K[0, 0] = 1.0                     # k_b = 0 gives q . k_b = 0
        S, P = oracle.weights(q, K, causal=False, scale=scale)
        assert S[0, 0] == pytest.approx(sa * scale, abs=1e-15)
        assert abs(P[0, 0] - wa) <= tol_w
        assert abs(P[0, 1] - wb) <= tol_w
        V = np.array([[1.0], [0.0]])
        dO = np.ones((1, 1))
        dQ, dK, dV, O, lse = oracle.bwd(q, K, V, dO, causal=False, scale=scale)
        assert O[0, 0] == pytest.approx(P[0, 0], rel=1e-15)
        deriv = dQ[0, 0] / scale          # = dS_a
        assert abs(deriv - dp) <= tol_dp
        assert deriv == pytest.approx(P[0, 0] * (1 - P[0, 0]), rel=1e-9)


def test_footnote4_score_statistics():
    """Footnote 4 of §3.2.1: for independent N(0,1) components q.k has mean 0, variance d_k.

    Checked statistically on the oracle's unscaled scores (scale = 1), and the
    variance returns to ~1 after the 1/sqrt(d_k) scale.
    """
    dk = 64
    q = normal_bf16((256, dk), 7).double().numpy()
    k = normal_bf16((256, dk), 8).double().numpy()
    S1, _ = oracle.weights(q, k, causal=False, scale=1.0)
    S8, _ = oracle.weights(q, k, causal=False, scale=1.0 / math.sqrt(dk))
    assert abs(S1.mean()) < 0.25
    assert S1.var() == pytest.approx(dk, rel=0.05)
    assert S8.var() == pytest.approx(1.0, rel=0.05)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_masked_weights_are_zero(causal):
    """Each softmax row sums to 100 %; illegal connections (j > i) weigh exactly 0 (§3.2.3)."""
    n, m, dk = 37, 53, 16
    q = normal_bf16((n, dk), 11).double().numpy() * 3
    k = normal_bf16((m, dk), 12).double().numpy()
    S, P = oracle.weights(q, k, causal=causal, scale=0.25)
    assert np.all(np.abs(P.sum(axis=1) - 1.0) < 1e-14)
    for i in range(n):
        for j in range(m):
            if causal and j > i:
                assert P[i, j] == 0.0 and S[i, j] == -np.inf
            else:
                assert P[i, j] > 0.0 and np.isfinite(S[i, j])
    # the diagonal is included: query i always sees key i ("including that position")
    if causal:
        assert all(P[i, i] > 0 for i in range(min(n, m)))


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_give_mean_of_values(causal):
    """Q = 0 (or scale = 0) makes every visible score equal: O_i = mean of the visible v_j.

    lse_i is then ln(number of visible keys): ln m, or ln(i+1) when causal.
    """
    B, h, n, m, d = 1, 2, 9, 7, 8
    v = normal_bf16((B, h, m, d), 13).double().numpy()
    k = normal_bf16((B, h, m, d), 14).double().numpy()
    for q, scale in ((np.zeros((B, h, n, d)), 0.125),
                     (normal_bf16((B, h, n, d), 15).double().numpy(), 0.0)):
        O, lse = oracle.fwd(q, k, v, causal, scale)
        for i in range(n):
            vis = min(i + 1, m) if causal else m
            np.testing.assert_allclose(O[:, :, i], v[:, :, :vis].mean(axis=2), rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[:, :, i], math.log(vis), rtol=0, atol=1e-14)


def test_permutation_equivariance():
    """O is a weighted sum over key/value pairs: permuting them jointly changes nothing.

    Permuting the queries permutes the output rows (non-causal).
    """
    B, h, n, m, d = 2, 2, 11, 13, 8
    q = normal_bf16((B, h, n, d), 21).double().numpy()
    k = normal_bf16((B, h, m, d), 22).double().numpy()
    v = normal_bf16((B, h, m, d), 23).double().numpy()
    O, lse = oracle.fwd(q, k, v, False, 0.3)
    perm = np.random.default_rng(0).permutation(m)
    O2, lse2 = oracle.fwd(q, k[:, :, perm], v[:, :, perm], False, 0.3)
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)
    qperm = np.random.default_rng(1).permutation(n)
    O3, lse3 = oracle.fwd(q[:, :, qperm], k, v, False, 0.3)
    assert np.array_equal(O3, O[:, :, qperm]) and np.array_equal(lse3, lse[:, :, qperm])


def test_single_key_closed_form():
    """m = 1: the only weight is 1, so O = v_0, lse = s_00, and every gradient of q and k is 0."""
    B, h, n, d = 1, 3, 5, 16
    q = normal_bf16((B, h, n, d), 31).double().numpy()
    k = normal_bf16((B, h, 1, d), 32).double().numpy()
    v = normal_bf16((B, h, 1, d), 33).double().numpy()
    dO = normal_bf16((B, h, n, d), 34).double().numpy()
    for causal in (False, True):
        O, lse = oracle.fwd(q, k, v, causal, 0.25)
        np.testing.assert_array_equal(O, np.broadcast_to(v, O.shape))
        s00 = 0.25 * np.einsum("bhnd,bhd->bhn", q, k[:, :, 0])
        np.testing.assert_allclose(lse, s00, rtol=1e-15, atol=1e-15)
        dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, causal, 0.25)
        assert np.all(dQ == 0.0) and np.all(dK == 0.0)
        np.testing.assert_allclose(dV[:, :, 0], dO.sum(axis=2), rtol=1e-14, atol=1e-14)


def test_causal_prefix_invariance():
    """Causal row i depends only on keys/values 0..i: changing later ones leaves it unchanged."""
    B, h, n, d = 1, 2, 12, 8
    q = normal_bf16((B, h, n, d), 41).double().numpy()
    k = normal_bf16((B, h, n, d), 42).double().numpy()
    v = normal_bf16((B, h, n, d), 43).double().numpy()
    O, lse = oracle.fwd(q, k, v, True, 0.35)
    for i in range(n):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] = 1000.0
        v2[:, :, i + 1:] = -1000.0
        O2, lse2 = oracle.fwd(q, k2, v2, True, 0.35)
        assert np.array_equal(O2[:, :, : i + 1], O[:, :, : i + 1])
        assert np.array_equal(lse2[:, :, : i + 1], lse[:, :, : i + 1])
    # row 0 sees only key 0: O_0 = v_0, lse_0 = s_00
    np.testing.assert_array_equal(O[:, :, 0], v[:, :, 0])


def test_row_subset_matches_full():
    B, h, n, m, d = 2, 1, 20, 9, 4
    q = normal_bf16((B, h, n, d), 51).double().numpy()
    k = normal_bf16((B, h, m, d), 52).double().numpy()
    v = normal_bf16((B, h, m, 6), 53).double().numpy()
    O, lse = oracle.fwd(q, k, v, True, 0.5)
    rows = [0, 3, 19]
    Os, lses = oracle.fwd(q, k, v, True, 0.5, rows=rows)
    np.testing.assert_array_equal(Os[:, :, rows], O[:, :, rows])
    np.testing.assert_array_equal(lses[:, :, rows], lse[:, :, rows])
    assert np.isnan(Os[:, :, 1]).all()


# ---------------------------------------------------------------- backward

def _loss(q, k, v, dO, causal, scale):
    O, _ = oracle.fwd(q, k, v, causal, scale)
    return float((dO * O).sum())


@pytest.mark.parametrize("causal,n,m,dk,dv", [(False, 4, 6, 3, 2), (True, 6, 6, 4, 4),
                                              (True, 5, 3, 2, 3), (False, 1, 5, 4, 1)])
def test_backward_matches_central_differences(causal, n, m, dk, dv):
    """dQ, dK, dV agree with fp64 central differences of L = sum(dO * O)."""
    rng = np.random.default_rng(n * 100 + m)
    q = rng.standard_normal((1, 1, n, dk))
    k = rng.standard_normal((1, 1, m, dk))
    v = rng.standard_normal((1, 1, m, dv))
    dO = rng.standard_normal((1, 1, n, dv))
    scale = 0.7
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, causal, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], dO, causal, scale)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], dO, causal, scale)) / (2 * eps)
        err = np.abs(num - g).max()
        assert err <= 1e-8 * max(1.0, np.abs(g).max()), (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_invariants(causal):
    """sum_j dK_j = 0 (rows of dS sum to 0) and sum_j dV_j = sum_i dO_i (rows of P sum to 1)."""
    B, h, n, m, d = 2, 2, 24, 24, 16
    q = normal_bf16((B, h, n, d), 61).double().numpy()
    k = normal_bf16((B, h, m, d), 62).double().numpy()
    v = normal_bf16((B, h, m, d), 63).double().numpy()
    dO = normal_bf16((B, h, n, d), 64).double().numpy()
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, causal, 0.25)
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(dV.sum(axis=2), dO.sum(axis=2), atol=1e-12)


# ---------------------------------------------------------------- library special case

@pytest.mark.parametrize("causal,n,m,dk,dv", [(False, 7, 5, 8, 8), (True, 9, 9, 16, 16),
                                              (True, 6, 10, 4, 4), (False, 3, 8, 4, 6)])
def test_against_torch_cpu_fp64_library(causal, n, m, dk, dv):
    """torch CPU fp64 scaled_dot_product_attention + autograd as an independent routine.

    torch's is_causal mask is lower-triangular from the top-left corner, the
    same reading of "illegal connections" used here.
    """
    F = torch.nn.functional
    g = torch.Generator().manual_seed(n * 31 + m)
    q = torch.randn(2, 2, n, dk, dtype=torch.float64, generator=g, requires_grad=True)
    k = torch.randn(2, 2, m, dk, dtype=torch.float64, generator=g, requires_grad=True)
    v = torch.randn(2, 2, m, dv, dtype=torch.float64, generator=g, requires_grad=True)
    dO = torch.randn(2, 2, n, dv, dtype=torch.float64, generator=g)
    scale = 1.0 / math.sqrt(dk)
    O_t = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    O_t.backward(dO)
    with torch.no_grad():
        sc = (q @ k.transpose(-1, -2)) * scale
        if causal:
            sc = sc.masked_fill(torch.ones(n, m, dtype=torch.bool).triu(1), float("-inf"))
        lse_t = torch.logsumexp(sc, dim=-1)
    O, lse = oracle.fwd(q.detach(), k.detach(), v.detach(), causal, scale)
    dQ, dK, dV, _, _ = oracle.bwd(q.detach(), k.detach(), v.detach(), dO, causal, scale)
    np.testing.assert_allclose(O, O_t.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_backward_rows_equal_full_backward(causal):
    """The sampled entry point (used at full sizes) returns the same rows as the full backward."""
    n, m, d = 40, 33, 8
    q = normal_bf16((n, d), 71).double().numpy()
    k = normal_bf16((m, d), 72).double().numpy()
    v = normal_bf16((m, d), 73).double().numpy()
    dO = normal_bf16((n, d), 74).double().numpy()
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, causal, 0.3)
    qr, kr = [0, 7, 39], [0, 5, 32]
    sq, sk, sv = oracle.bwd_rows(q, k, v, dO, causal, 0.3, qr, kr)
    np.testing.assert_array_equal(sq, dQ[qr])
    np.testing.assert_array_equal(sk, dK[kr])
    np.testing.assert_array_equal(sv, dV[kr])


# ---------------------------------------------------------------- key padding
#
# Variable-length batches ("Attention Is All You Need" §5.1 batches sentences
# of similar length; the <pad> positions of Figure 3): sequence b has kv_len[b]
# real keys, the first ones, and the padding keys are masked.

def _padding_case(seed=5, B=3, h=2, n=7, m=9, dk=5, dv=4):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, h, n, dk, dtype=torch.float64, generator=g).numpy()
    k = torch.randn(B, h, m, dk, dtype=torch.float64, generator=g).numpy()
    v = torch.randn(B, h, m, dv, dtype=torch.float64, generator=g).numpy()
    dO = torch.randn(B, h, n, dv, dtype=torch.float64, generator=g).numpy()
    return q, k, v, dO


@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_equals_truncation(causal):
    """Padding keys j >= L of a sequence act as if the sequence had only L keys."""
    q, k, v, dO = _padding_case()
    lens = [9, 4, 1]
    scale = 0.4
    O, lse = oracle.fwd(q, k, v, causal, scale, kv_len=lens)
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, causal, scale, kv_len=lens)
    for b, L in enumerate(lens):
        Ob, lb = oracle.fwd(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], causal, scale)
        np.testing.assert_allclose(O[b], Ob[0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[b], lb[0], rtol=1e-13, atol=1e-14)
        gq, gk, gv, _, _ = oracle.bwd(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], dO[b:b + 1],
                                      causal, scale)
        np.testing.assert_allclose(dQ[b], gq[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dK[b, :, :L], gk[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dV[b, :, :L], gv[0], rtol=1e-12, atol=1e-14)
        assert (dK[b, :, L:] == 0).all() and (dV[b, :, L:] == 0).all()


def test_key_padding_against_torch_masked_library():
    """torch CPU fp64 scaled_dot_product_attention with a boolean key mask."""
    F = torch.nn.functional
    q, k, v, dO = (torch.from_numpy(a).requires_grad_(i < 3) for i, a in enumerate(_padding_case(seed=9)))
    lens = [2, 9, 6]
    B, h, n, m = q.shape[0], q.shape[1], q.shape[2], k.shape[2]
    keep = torch.arange(m)[None, :] < torch.tensor(lens)[:, None]       # [B, m]
    mask = keep[:, None, None, :].expand(B, 1, n, m)
    O_t = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.3)
    O_t.backward(dO)
    O, _ = oracle.fwd(q.detach(), k.detach(), v.detach(), False, 0.3, kv_len=lens)
    dQ, dK, dV, _, _ = oracle.bwd(q.detach(), k.detach(), v.detach(), dO, False, 0.3, kv_len=lens)
    np.testing.assert_allclose(O, O_t.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_key_padding_values_do_not_matter():
    """What sits in the padding keys and values cannot change any result."""
    q, k, v, dO = _padding_case(seed=7)
    lens = [5, 9, 3]
    k2, v2 = k.copy(), v.copy()
    for b, L in enumerate(lens):
        k2[b, :, L:] = 1e3
        v2[b, :, L:] = -7.0
    a = oracle.fwd(q, k, v, True, 0.5, kv_len=lens)
    b_ = oracle.fwd(q, k2, v2, True, 0.5, kv_len=lens)
    np.testing.assert_array_equal(a[0], b_[0])
    np.testing.assert_array_equal(a[1], b_[1])
    ga = oracle.bwd(q, k, v, dO, True, 0.5, kv_len=lens)
    gb = oracle.bwd(q, k2, v2, dO, True, 0.5, kv_len=lens)
    np.testing.assert_array_equal(ga[0], gb[0])


def test_key_padding_empty_sequence_is_the_empty_sum():
    """A sequence without real keys: O = 0, lse = -inf, zero gradients (the reading for L = 0)."""
    q, k, v, dO = _padding_case(seed=3)
    lens = [0, 9, 0]
    O, lse = oracle.fwd(q, k, v, False, 0.5, kv_len=lens)
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, False, 0.5, kv_len=lens)
    for b in (0, 2):
        assert (O[b] == 0).all() and np.isneginf(lse[b]).all()
        assert (dQ[b] == 0).all() and (dK[b] == 0).all() and (dV[b] == 0).all()
    assert np.isfinite(O[1]).all() and np.isfinite(lse[1]).all()
    # sampled rows agree with the full backward under padding
    sq, sk, sv = oracle.bwd_rows(q[1, 0], k[1, 0], v[1, 0], dO[1, 0], True, 0.5, [0, 6], [0, 3, 8],
                                 kv_len=4)
    fq, fk, fv, _, _ = oracle.bwd(q[1:2, :1], k[1:2, :1], v[1:2, :1], dO[1:2, :1], True, 0.5, kv_len=[4])
    np.testing.assert_array_equal(sq, fq[0, 0][[0, 6]])
    np.testing.assert_array_equal(sk, fk[0, 0][[0, 3, 8]])
    np.testing.assert_array_equal(sv, fv[0, 0][[0, 3, 8]])


# ---------------------------------------------------------------- restricted self-attention (§4, Table 1)

def _window_case(seed=21, B=2, h=2, n=11, m=11, d=6):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, h, n, d))
    k = rng.standard_normal((B, h, m, d))
    v = rng.standard_normal((B, h, m, d))
    dO = rng.standard_normal((B, h, n, d))
    return q, k, v, dO


def _band(n, m, wl, wr, causal=False, lens=None, B=1):
    """Boolean [B, n, m] mask written out from the definition: i - wl <= j <= i + wr."""
    i = np.arange(n)[:, None]
    j = np.arange(m)[None, :]
    keep = np.ones((n, m), dtype=bool)
    if wl >= 0:
        keep &= j >= i - wl
    if wr >= 0:
        keep &= j <= i + wr
    if causal:
        keep &= j <= i
    keep = np.broadcast_to(keep, (B, n, m)).copy()
    if lens is not None:
        for b, L in enumerate(lens):
            keep[b, :, L:] = False
    return keep


def test_window_wider_than_the_sequence_is_no_window():
    """A window reaching past both ends changes nothing, bit for bit."""
    q, k, v, dO = _window_case()
    for causal in (False, True):
        a = oracle.fwd(q, k, v, causal, 0.5)
        b = oracle.fwd(q, k, v, causal, 0.5, window=(11, 11))
        c = oracle.fwd(q, k, v, causal, 0.5, window=(-1, 40))
        for x in (b, c):
            np.testing.assert_array_equal(a[0], x[0])
            np.testing.assert_array_equal(a[1], x[1])
        ga = oracle.bwd(q, k, v, dO, causal, 0.5)
        gb = oracle.bwd(q, k, v, dO, causal, 0.5, window=(20, 20))
        for x, y in zip(ga[:3], gb[:3]):
            np.testing.assert_array_equal(x, y)


def test_window_of_one_position_returns_own_value():
    """r = 1 (wl = wr = 0): query i sees only key i, so O_i = v_i, lse_i = s_ii,
    dQ = dK = 0 (a single weight of 1 has zero derivative) and dV_i = dO_i."""
    q, k, v, dO = _window_case(seed=5)
    scale = 0.8
    O, lse = oracle.fwd(q, k, v, False, scale, window=(0, 0))
    np.testing.assert_allclose(O, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, scale * (q * k).sum(-1), rtol=1e-14, atol=1e-14)
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, False, scale, window=(0, 0))
    np.testing.assert_allclose(dQ, 0.0, atol=1e-14)
    np.testing.assert_allclose(dK, 0.0, atol=1e-14)
    np.testing.assert_allclose(dV, dO, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("wl,wr,causal,lens", [(2, 3, False, None), (4, -1, False, None), (-1, 1, False, None),
                                               (3, 3, True, None), (2, 5, False, [7, 11])])
def test_window_against_torch_masked_library(wl, wr, causal, lens):
    """torch CPU fp64 scaled_dot_product_attention (+ autograd) with the band written
    out as a boolean mask, asymmetric windows, one open side, causal, key padding."""
    F = torch.nn.functional
    q, k, v, dO = (torch.from_numpy(a).requires_grad_(i < 3) for i, a in enumerate(_window_case(seed=wl + 7)))
    B, h, n, m = q.shape[0], q.shape[1], q.shape[2], k.shape[2]
    mask = torch.from_numpy(_band(n, m, wl, wr, causal, lens, B))[:, None]
    O_t = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.6)
    O_t.backward(dO)
    O, _ = oracle.fwd(q.detach(), k.detach(), v.detach(), causal, 0.6, kv_len=lens, window=(wl, wr))
    dQ, dK, dV, _, _ = oracle.bwd(q.detach(), k.detach(), v.detach(), dO, causal, 0.6, kv_len=lens,
                                  window=(wl, wr))
    np.testing.assert_allclose(O, O_t.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_causal_window_is_the_left_window():
    """The causal mask is the window's right side at 0: (causal, wl, any wr) = (not causal, wl, 0)."""
    q, k, v, dO = _window_case(seed=8)
    a = oracle.bwd(q, k, v, dO, True, 0.4, window=(3, 6))
    b = oracle.bwd(q, k, v, dO, False, 0.4, window=(3, 0))
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_window_rows_without_keys_are_the_empty_sum():
    """n > m: rows whose window lies wholly past the last key see nothing (O = 0,
    lse = -inf) and pass no gradient; the other rows are untouched by them."""
    q, k, v, dO = _window_case(seed=4, n=14, m=6)
    wl, wr = 2, 1
    O, lse = oracle.fwd(q, k, v, False, 0.5, window=(wl, wr))
    empty = np.arange(14) - wl > 5
    assert (O[:, :, empty] == 0).all() and np.isneginf(lse[:, :, empty]).all()
    assert np.isfinite(lse[:, :, ~empty]).all()
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, False, 0.5, window=(wl, wr))
    assert (dQ[:, :, empty] == 0).all()
    dO2 = dO.copy()
    dO2[:, :, empty] = 5.0  # upstream gradient of the empty rows cannot reach K or V
    _, dK2, dV2, _, _ = oracle.bwd(q, k, v, dO2, False, 0.5, window=(wl, wr))
    np.testing.assert_array_equal(dK, dK2)
    np.testing.assert_array_equal(dV, dV2)


def test_window_backward_matches_central_differences():
    """Brute force for the banded backward on a tiny head."""
    rng = np.random.default_rng(77)
    n, m, dk, dv = 6, 7, 3, 2
    q = rng.standard_normal((1, 1, n, dk))
    k = rng.standard_normal((1, 1, m, dk))
    v = rng.standard_normal((1, 1, m, dv))
    dO = rng.standard_normal((1, 1, n, dv))
    win, scale = (1, 2), 0.9
    dQ, dK, dV, _, _ = oracle.bwd(q, k, v, dO, False, scale, window=win)

    def loss(qq, kk, vv):
        O, _ = oracle.fwd(qq, kk, vv, False, scale, window=win)
        return float((dO * O).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            a = {"q": q, "k": k, "v": v}
            b = dict(a)
            a[name], b[name] = xp, xm
            num[idx] = (loss(a["q"], a["k"], a["v"]) - loss(b["q"], b["k"], b["v"])) / (2 * eps)
        assert np.abs(num - g).max() <= 1e-8 * max(1.0, np.abs(g).max()), name


def test_window_sampled_rows_match_full_backward():
    q, k, v, dO = _window_case(seed=12, B=1, h=1, n=13, m=13)
    win = (2, 4)
    sq, sk, sv = oracle.bwd_rows(q[0, 0], k[0, 0], v[0, 0], dO[0, 0], False, 0.5, [0, 7, 12], [1, 6, 12],
                                 kv_len=10, window=win)
    fq, fk, fv, _, _ = oracle.bwd(q, k, v, dO, False, 0.5, kv_len=[10], window=win)
    np.testing.assert_array_equal(sq, fq[0, 0][[0, 7, 12]])
    np.testing.assert_array_equal(sk, fk[0, 0][[1, 6, 12]])
    np.testing.assert_array_equal(sv, fv[0, 0][[1, 6, 12]])


# ---------------------------------------------------------------- incremental decoding (§3)

@pytest.mark.parametrize("n,lens", [(1, None), (4, None), (3, [9, 17, 4]), (5, [2, 17, 0])])
def test_decode_step_equals_last_rows_of_full_causal_pass(n, lens):
    """A decoding step over the cache gives exactly the last n rows of the decoder's
    causal self-attention over the whole sequence (the reason a cache works): the
    n newest queries attend to everything cached up to and including themselves."""
    rng = np.random.default_rng(n + 31)
    B, h, m, d = 3, 2, 17, 5
    q_full = rng.standard_normal((B, h, m, d))
    k = rng.standard_normal((B, h, m, d))
    v = rng.standard_normal((B, h, m, d))
    Ls = [m] * B if lens is None else lens
    q_new = np.zeros((B, h, n, d))
    for b, L in enumerate(Ls):
        for i in range(n):
            pos = L - n + i
            if pos >= 0:
                q_new[b, :, i] = q_full[b, :, pos]
    O, lse = oracle.decode(q_new, k, v, 0.45, kv_len=lens)
    for b, L in enumerate(Ls):
        if L == 0:
            assert (O[b] == 0).all() and np.isneginf(lse[b]).all()
            continue
        Of, lf = oracle.fwd(q_full[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L], True, 0.45)
        for i in range(n):
            pos = L - n + i
            if pos < 0:
                assert (O[b, :, i] == 0).all() and np.isneginf(lse[b, :, i]).all()
            else:
                np.testing.assert_allclose(O[b, :, i], Of[0, :, pos], rtol=1e-13, atol=1e-14)
                np.testing.assert_allclose(lse[b, :, i], lf[0, :, pos], rtol=1e-13, atol=1e-14)


def test_decode_against_torch_with_bottom_right_mask():
    """torch fp64 SDPA with the cache mask written out: query i of n sees key j iff j <= L - n + i, j < L."""
    F = torch.nn.functional
    rng = np.random.default_rng(5)
    B, h, n, m, d = 2, 3, 4, 13, 8
    q = torch.from_numpy(rng.standard_normal((B, h, n, d)))
    k = torch.from_numpy(rng.standard_normal((B, h, m, d)))
    v = torch.from_numpy(rng.standard_normal((B, h, m, d)))
    lens = [13, 7]
    mask = torch.zeros(B, 1, n, m, dtype=torch.bool)
    for b, L in enumerate(lens):
        for i in range(n):
            mask[b, 0, i, : L - n + i + 1] = True
    ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.3)
    O, _ = oracle.decode(q, k, v, 0.3, kv_len=lens)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- multi-head projections (§3.2.2)

def test_multi_head_shapes_and_weight_count_of_the_close_reading():
    """The close reading's walk-through: a 10-token sentence, d_model 512, h = 8 heads of 64:
    each head projects 10 x 512 to 10 x 64, weights are 10 x 10, the heads concatenate back to
    10 x 512, and the sublayer holds four 512 x 512 matrices = 1,048,576 weights."""
    rng = np.random.default_rng(0)
    h, d, dm = 8, 64, 512
    x = rng.standard_normal((1, 10, dm))
    w_qkv = rng.standard_normal((dm, 3 * h * d)) / np.sqrt(dm)
    w_o = rng.standard_normal((h * d, dm)) / np.sqrt(dm)
    q, k, v = oracle.project_qkv(x, x, w_qkv, h, d)
    assert q.shape == k.shape == v.shape == (1, h, 10, d)
    S, P = oracle.weights(q[0, 0], k[0, 0], False, 1 / 8)
    assert P.shape == (10, 10)
    y = oracle.multi_head(x, x, w_qkv, w_o, h, d)
    assert y.shape == (1, 10, dm)
    assert w_qkv.size + w_o.size == 1_048_576


@pytest.mark.parametrize("causal,n,m", [(False, 7, 7), (True, 9, 9), (False, 5, 11)])
def test_multi_head_against_torch_library(causal, n, m):
    """torch fp64 multi_head_attention_forward (no biases, no dropout) as an independent routine;
    its in_proj_weight [3E, E] is the transpose of the pages' [d_model, 3 h d] orientation."""
    F = torch.nn.functional
    rng = np.random.default_rng(n * 7 + m)
    h, d = 4, 8
    E = h * d
    xq = rng.standard_normal((2, n, E))
    xkv = xq if n == m else rng.standard_normal((2, m, E))  # self- or cross-attention
    w_qkv = rng.standard_normal((E, 3 * E)) / np.sqrt(E)
    w_o = rng.standard_normal((E, E)) / np.sqrt(E)
    mask = None
    if causal:
        mask = torch.triu(torch.full((n, m), float("-inf"), dtype=torch.float64), diagonal=1)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    ref, _ = F.multi_head_attention_forward(
        t(xq).transpose(0, 1), t(xkv).transpose(0, 1), t(xkv).transpose(0, 1), E, h,
        in_proj_weight=t(w_qkv.T), in_proj_bias=None, bias_k=None, bias_v=None, add_zero_attn=False,
        dropout_p=0.0, out_proj_weight=t(w_o.T), out_proj_bias=None, training=False,
        need_weights=False, attn_mask=mask)
    y = oracle.multi_head(xq, xkv, w_qkv, w_o, h, d, causal=causal)
    np.testing.assert_allclose(y, ref.transpose(0, 1).numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- projection gradients (§3.2.2, differentiated)

def _proj_case(seed, B=2, n=5, m=7, h=2, d=4, dm=8):
    rng = np.random.default_rng(seed)
    xq = rng.standard_normal((B, n, dm))
    xkv = rng.standard_normal((B, m, dm))
    w_qkv = rng.standard_normal((dm, 3 * h * d))
    w_o = rng.standard_normal((h * d, dm))
    gq = rng.standard_normal((B, h, n, d))
    gk = rng.standard_normal((B, h, m, d))
    gv = rng.standard_normal((B, h, m, d))
    o = rng.standard_normal((B, h, n, d))
    gy = rng.standard_normal((B, n, dm))
    return xq, xkv, w_qkv, w_o, gq, gk, gv, o, gy


def test_projection_gradients_match_finite_differences():
    """For L = <dq, Q> + <dk, K> + <dv, V> (and <dy, Y>) the oracle's gradients are the derivatives
    of its own forward projections: a central difference along a random direction of (x, W) equals
    <grad, direction> (the maps are linear, so only rounding separates the two)."""
    xq, xkv, w_qkv, w_o, gq, gk, gv, o, gy = _proj_case(11)
    h, d = gq.shape[1], gq.shape[3]
    rng = np.random.default_rng(12)
    ux, uk, uw = (rng.standard_normal(a.shape) for a in (xq, xkv, w_qkv))

    def loss(a, b, w):
        q, k, v = oracle.project_qkv(a, b, w, h, d)
        return float((gq * q).sum() + (gk * k).sum() + (gv * v).sum())

    eps = 1e-3
    fd = (loss(xq + eps * ux, xkv + eps * uk, w_qkv + eps * uw) -
          loss(xq - eps * ux, xkv - eps * uk, w_qkv - eps * uw)) / (2 * eps)
    dxq, dxkv, dw = oracle.project_qkv_bwd(xq, xkv, w_qkv, gq, gk, gv)
    an = float((dxq * ux).sum() + (dxkv * uk).sum() + (dw * uw).sum())
    assert abs(fd - an) <= 1e-8 * max(1.0, abs(an))

    uo, uwo = rng.standard_normal(o.shape), rng.standard_normal(w_o.shape)
    lo = lambda a, w: float((gy * oracle.project_out(a, w)).sum())
    fd = (lo(o + eps * uo, w_o + eps * uwo) - lo(o - eps * uo, w_o - eps * uwo)) / (2 * eps)
    d_o, dwo = oracle.project_out_bwd(o, w_o, gy)
    an = float((d_o * uo).sum() + (dwo * uwo).sum())
    assert abs(fd - an) <= 1e-8 * max(1.0, abs(an))


def test_projection_gradients_against_torch_autograd():
    """torch fp64 autograd of the same products (an independent routine): the head split of
    x W (reshape to heads) and the concatenation Concat(o) W^O, differentiated by the library."""
    xq, xkv, w_qkv, w_o, gq, gk, gv, o, gy = _proj_case(21, B=3, n=6, m=4, h=3, d=2, dm=5)
    B, h, n, d = gq.shape
    m = gk.shape[2]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True)
    Xq, Xkv, W, O, Wo = t(xq), t(xkv), t(w_qkv), t(o), t(w_o)
    hd = h * d
    split = lambda Y, S: Y.reshape(Y.shape[0], S, h, d).transpose(1, 2)
    q, k, v = split(Xq @ W[:, :hd], n), split(Xkv @ W[:, hd:2 * hd], m), split(Xkv @ W[:, 2 * hd:], m)
    y = O.transpose(1, 2).reshape(B, n, hd) @ Wo
    L = (q * torch.from_numpy(gq)).sum() + (k * torch.from_numpy(gk)).sum() + (v * torch.from_numpy(gv)).sum() \
        + (y * torch.from_numpy(gy)).sum()
    L.backward()
    dxq, dxkv, dw = oracle.project_qkv_bwd(xq, xkv, w_qkv, gq, gk, gv)
    d_o, dwo = oracle.project_out_bwd(o, w_o, gy)
    for got, ref in ((dxq, Xq.grad), (dxkv, Xkv.grad), (dw, W.grad), (d_o, O.grad), (dwo, Wo.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)
