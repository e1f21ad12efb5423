"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import WORKLOADS, Workload, normal_bf16, ragged_workloads, workload_inputs
from tests.parity_utils import assert_close, default_scale, errors, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _small(name, B, h, n, m, d, causal, cfg):
    return Workload(name, B, h, n, m, d, d, causal, cfg)


# Shapes of every configuration, shrunk in B*h so the oracle runs in seconds,
# spanning several 128/256-row tiles with ragged tails.
SMALL = [
    WORKLOADS["tiny"], WORKLOADS["tiny_causal"],
    _small("encoder_s", 2, 2, 256, 256, 64, False, 2),
    _small("decoder_s", 2, 2, 256, 256, 64, True, 3),
    _small("cross_s", 1, 3, 256, 320, 64, False, 4),
    _small("cross_h4d128_s", 1, 2, 256, 320, 128, False, 4),
    _small("cross_h16d32_s", 1, 3, 256, 320, 32, False, 4),
    _small("long1024_d64_s", 1, 1, 1024, 1024, 64, False, 5),
    _small("long1024_d64c_s", 1, 1, 1024, 1024, 64, True, 5),
    _small("long1024_d128c_s", 1, 1, 1024, 1024, 128, True, 5),
    _small("long700_d128_s", 1, 1, 700, 700, 128, False, 5),
    # more short items than SMs, so that every persistent CTA runs several in a
    # row: one key tile with a partial second query tile, and two key tiles
    _small("items400_n200_m128_d32", 50, 8, 200, 128, 32, False, 7),
    _small("items320_n256_m256_d64", 40, 8, 256, 256, 64, False, 8),
] + list(ragged_workloads())


def run_fwd(q, k, v, causal, scale):
    o, lse = A.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    assert A.attn_get_device_status() == A.ATTN_OK
    return o, lse


def run_bwd(q, k, v, o, lse, do, causal, scale):
    dq, dk, dv = A.attn_bwd(q.to(DEV), k.to(DEV), v.to(DEV), o, lse, do.to(DEV), causal=causal, scale=scale)
    assert A.attn_get_device_status() == A.ATTN_OK
    return dq, dk, dv


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fwd_bwd_match_oracle(w):
    q, k, v, do = workload_inputs(w, with_grad=True)
    scale = w.default_scale
    o, lse = run_fwd(q, k, v, w.causal, scale)
    dq, dk, dv = run_bwd(q, k, v, o, lse, do, w.causal, scale)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(q, k, v, do, w.causal, scale)
    ex = "few_term_cancellation" if w.causal else None
    assert_close("O", o, ro)
    assert_close("lse", lse, rlse)
    assert_close("dQ", dq, rdq, allow=ex)
    assert_close("dK", dk, rdk, allow=ex)
    assert_close("dV", dv, rdv, allow=ex)


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("mult,first_big", [(4.0, 1), (16.0, 1), (64.0, 1), (64.0, 3), (0.25, 1)])
def test_scores_that_grow_after_the_first_key_tile(d, mult, first_big):
    """Later key tiles with much larger scores than the first (keys scaled by a
    power of two, exact in bf16): the forward that exponentiates later tiles
    against the first tile's row maximum must notice the growth (weights far
    above 1, or infinite for mult = 64) and move to the new maximum; mult < 1
    makes the later tiles' weights vanish instead."""
    n, m = 256, 512
    q = normal_bf16((1, 2, n, d), 1101)
    k = normal_bf16((1, 2, m, d), 1102)
    v = normal_bf16((1, 2, m, d), 1103)
    k[:, :, first_big * 128:, :] *= mult
    scale = default_scale(d)
    o, lse = run_fwd(q, k, v, False, scale)
    ro, rlse = oracle.fwd(q, k, v, False, scale)
    assert_close("O", o, ro)
    assert_close("lse", lse, rlse)


@pytest.mark.parametrize("scale", [0.0, 1.0, -0.2, 0.03])
@pytest.mark.parametrize("causal", [False, True])
def test_scale_values(scale, causal):
    """scale = 0 (equal weights), 1 (unscaled dot product), negative and small.

    At scale = 1 with d_k = 64 the scores have standard deviation 8 and the
    softmax saturates (the case §3.2.1 gives for the 1/sqrt(d_k) scale): the
    gradients become small and their error is set by D_i = dO_i . O_i formed
    from the bf16 O. That backward is held to the documented exception
    "unscaled_scores_backward" (tests/parity_utils.py); causal gradients may use
    "few_term_cancellation"; everything else the plain bound.
    """
    w = _small("s", 1, 2, 200, 200, 64, causal, 7)
    q, k, v, do = workload_inputs(w, with_grad=True)
    o, lse = run_fwd(q, k, v, causal, scale)
    dq, dk, dv = run_bwd(q, k, v, o, lse, do, causal, scale)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(q, k, v, do, causal, scale)
    assert_close("O", o, ro)
    assert_close("lse", lse, rlse)
    sat = "unscaled_scores_backward" if abs(scale) >= 1.0 else ("few_term_cancellation" if causal else None)
    assert_close("dQ", dq, rdq, allow=sat)
    assert_close("dK", dk, rdk, allow=sat)
    assert_close("dV", dv, rdv, allow=sat)


@pytest.mark.parametrize("scale", [0.0, 1.0, -0.2, 0.03])
@pytest.mark.parametrize("m", [256, 640])
def test_scale_values_persistent_forward(scale, m):
    """The same scales through the persistent forward (non-causal, whole 128-key
    tiles): m = 256 takes every tile's maximum, m = 640 exponentiates its later
    tiles against the running reference (scale = 1 saturates the softmax, so the
    scores there often outgrow the first tile's maximum)."""
    w = _small("sp", 1, 2, 256, m, 64, False, 8)
    q, k, v = workload_inputs(w)
    o, lse = run_fwd(q, k, v, False, scale)
    ro, rlse = oracle.fwd(q, k, v, False, scale)
    assert_close("O", o, ro)
    assert_close("lse", lse, rlse)


def test_worked_example_weights_on_gpu():
    """The 2-d example of the close-reading page, zero-padded to d=32, V = identity rows.

    With v_j = e_j the output row is the weight vector itself.
    """
    q2 = [[2.2, 0.0]]
    k2 = [[0.2, 0], [2, 0.4], [0.3, 1.6], [0, 0.2], [1, 0.3], [0.1, 0.5], [0.4, 1.4]]
    q = torch.zeros(1, 1, 1, 32)
    k = torch.zeros(1, 1, 7, 32)
    q[0, 0, :, :2] = torch.tensor(q2)
    k[0, 0, :, :2] = torch.tensor(k2)
    v = torch.zeros(1, 1, 7, 32)
    v[0, 0, torch.arange(7), torch.arange(7)] = 1.0
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    scale = 1 / math.sqrt(2)
    o, lse = run_fwd(q, k, v, False, scale)
    _, P = oracle.weights(q[0, 0], k[0, 0], False, scale)
    w = to64(o)[0, 0, 0, :7]
    np.testing.assert_allclose(w, P[0], atol=2e-3)
    # the printed percentages (4.0 / 66 / 4.7 / 2.9 / 14 / 3.4 / 5.5) to within 0.6 points
    printed = np.array([4.0, 66, 4.7, 2.9, 14, 3.4, 5.5])
    assert np.abs(100 * w - printed).max() < 0.6


def test_causal_prefix_invariance_bitwise():
    """Causal row i ignores keys after i: replacing them leaves O_i and lse_i bit-identical."""
    w = _small("p", 1, 2, 300, 300, 64, True, 8)
    q, k, v = workload_inputs(w)
    o, lse = run_fwd(q, k, v, True, w.default_scale)
    for cut in (0, 5, 127, 128, 129, 255, 256, 299):
        k2, v2 = k.clone(), v.clone()
        k2[:, :, cut + 1:] = 1000.0
        v2[:, :, cut + 1:] = -1000.0
        o2, lse2 = run_fwd(q, k2, v2, True, w.default_scale)
        assert torch.equal(o2[:, :, : cut + 1], o[:, :, : cut + 1]), cut
        assert torch.equal(lse2[:, :, : cut + 1], lse[:, :, : cut + 1]), cut
    # row 0 sees only key 0
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_and_ones(causal):
    """Q = 0: O_i = mean of visible v_j, lse_i = ln(#visible). V = 1: O = 1."""
    w = _small("e", 1, 2, 260, 260, 64, causal, 9)
    _, k, v = workload_inputs(w)
    q = torch.zeros(1, 2, 260, 64, dtype=torch.bfloat16)
    o, lse = run_fwd(q, k, v, causal, 0.125)
    vis = np.minimum(np.arange(260) + 1, 260) if causal else np.full(260, 260)
    vv = to64(v)
    mean = np.cumsum(vv, axis=2) / np.arange(1, 261)[None, None, :, None] if causal else \
        np.broadcast_to(vv.mean(axis=2, keepdims=True), vv.shape)
    assert_close("O", o, mean)
    assert_close("lse", lse, np.broadcast_to(np.log(vis), (1, 2, 260)))
    ones = torch.ones_like(v)
    o1, _ = run_fwd(workload_inputs(w)[0], k, ones, causal, 0.125)
    assert np.abs(to64(o1) - 1.0).max() <= 4e-3


def test_single_key():
    """m = 1: O = v_0 exactly, lse = scale q.k_0, dQ = dK = 0, dV_0 = sum_i dO_i."""
    q = normal_bf16((1, 2, 70, 64), 91)
    k = normal_bf16((1, 2, 1, 64), 92)
    v = normal_bf16((1, 2, 1, 64), 93)
    do = normal_bf16((1, 2, 70, 64), 94)
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, causal, 0.125)
        assert torch.equal(o.cpu(), v.expand(1, 2, 70, 64))
        dq, dk, dv = run_bwd(q, k, v, o, lse, do, causal, 0.125)
        rdq, rdk, rdv, _, rlse = oracle.bwd(q, k, v, do, causal, 0.125)
        assert_close("lse", lse, rlse)
        assert np.abs(to64(dq)).max() < 1e-2 and np.abs(to64(dk)).max() < 1e-2
        assert_close("dV", dv, rdv)


def invariant_bounds(q, v, do, dk, dv, scale):
    """6-sigma bounds for |sum_j dK_j| and |sum_j dV_j - sum_i dO_i| per (head, column).

    In exact arithmetic both are 0. In bf16 arithmetic the deviation is a sum
    of independent roundings of relative size u = 2^-9 (rms u / sqrt(3)):
      dV: bf16 weights P (each row's rounding error weighs at most the row,
          since sum_j P_ij^2 <= 1) times dO_i, plus the output rounding of each dV_j;
      dK: the inconsistency of D_i = dO_i . O_i with the bf16 O (|O_i| is at
          most max_j |v_j|, two roundings) times scale q_i, plus the output
          rounding of each dK_j.
    Only inputs and the GPU's own dK, dV rows enter the bound, never an expected value.
    """
    u = 2.0 ** -9 / math.sqrt(3)
    vmax = np.linalg.norm(v, axis=-1).max(axis=-1)[..., None, None]
    dnorm = np.linalg.norm(do, axis=-1)[..., None]
    tol_v = 6 * u * np.sqrt((do ** 2).sum(axis=-2) + (dv ** 2).sum(axis=-2)) + 1e-3
    tol_k = 6 * u * np.sqrt(((2 * abs(scale) * dnorm * vmax * q) ** 2).sum(axis=-2)
                            + (dk ** 2).sum(axis=-2)) + 1e-3
    return tol_k, tol_v


def test_gradient_invariants_on_gpu():
    """sum_j dK_j ~ 0 and sum_j dV_j ~ sum_i dO_i on the GPU outputs, within the rounding budget."""
    for causal in (False, True):
        w = _small("g", 1, 2, 384, 384, 64, causal, 10)
        q, k, v, do = workload_inputs(w, with_grad=True)
        o, lse = run_fwd(q, k, v, causal, w.default_scale)
        dq, dk, dv = run_bwd(q, k, v, o, lse, do, causal, w.default_scale)
        dkk, dvv = to64(dk), to64(dv)
        tol_k, tol_v = invariant_bounds(to64(q), to64(v), to64(do), dkk, dvv, w.default_scale)
        assert (np.abs(dkk.sum(axis=2)) <= tol_k).all()
        assert (np.abs(dvv.sum(axis=2) - to64(do).sum(axis=2)) <= tol_v).all()


def test_outputs_written_exactly_in_bounds():
    """NaN-filled outputs are fully overwritten, and guard words after each output stay intact."""
    w = _small("c", 1, 3, 200, 77, 64, True, 11)
    q, k, v, do = [t.to(DEV) for t in workload_inputs(w, with_grad=True)]
    G = 4096

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + G,), float("nan"), dtype=dtype, device=DEV)
        buf[n:] = 7.0
        return buf, buf[:n].view(shape)

    ob, o = guarded(q.shape, torch.bfloat16)
    lb, lse = guarded(q.shape[:3], torch.float32)
    A.attn_fwd(q, k, v, causal=True, scale=0.125, out=o, lse=lse)
    qb, dq = guarded(q.shape, torch.bfloat16)
    kb, dk = guarded(k.shape, torch.bfloat16)
    vb, dv = guarded(v.shape, torch.bfloat16)
    A.attn_bwd(q, k, v, o, lse, do, causal=True, scale=0.125, dq=dq, dk=dk, dv=dv)
    assert A.attn_get_device_status() == A.ATTN_OK
    for buf, t in ((ob, o), (lb, lse), (qb, dq), (kb, dk), (vb, dv)):
        assert torch.isfinite(t).all()
        assert (buf[t.numel():] == 7.0).all()


def test_empty_and_degenerate_sizes():
    q = torch.zeros(0, 2, 16, 64, dtype=torch.bfloat16, device=DEV)
    o, lse = A.attn_fwd(q, q, q)
    assert o.shape == (0, 2, 16, 64)
    # n = 0 with keys present: no outputs for O; dK = dV = 0
    q0 = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device=DEV)
    k = normal_bf16((1, 2, 33, 64), 5).to(DEV)
    o0, lse0 = A.attn_fwd(q0, k, k)
    dq, dk, dv = A.attn_bwd(q0, k, k, o0, lse0, q0)
    assert A.attn_get_device_status() == A.ATTN_OK
    assert (dk == 0).all() and (dv == 0).all()


def test_watchdog_reports_timeout_and_gpu_stays_usable():
    """A value tile that never arrives ends in ATTN_ERR_TIMEOUT, not a hang; the next call is fine."""
    w = _small("t", 1, 2, 256, 512, 64, False, 12)
    q, k, v = workload_inputs(w)
    ref_o, ref_lse = oracle.fwd(q, k, v, False, w.default_scale)
    A.attn_set_watchdog_ns(50_000_000)  # 50 ms per wait
    try:
        A.attn_debug_inject(1)
        A.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), scale=w.default_scale)
        assert A.attn_get_device_status() == A.ATTN_ERR_TIMEOUT
        assert A.attn_get_device_status() == A.ATTN_OK  # cleared once read
    finally:
        A.attn_debug_inject(0)
        A.attn_set_watchdog_ns(0)
    o, lse = run_fwd(q, k, v, False, w.default_scale)
    assert_close("O", o, ref_o)
    assert_close("lse", lse, ref_lse)


def test_bad_arguments_on_gpu():
    q = normal_bf16((1, 1, 8, 48), 1).to(DEV)
    with pytest.raises(A.AttnError) as e:
        A.attn_fwd(q, q, q)
    assert e.value.status == A.ATTN_ERR_UNSUPPORTED
    q64 = normal_bf16((1, 1, 8, 64), 1).to(DEV)
    with pytest.raises(A.AttnError) as e:
        A.attn_fwd(q64, q64, q64, scale=float("nan"))
    assert e.value.status == A.ATTN_ERR_INVALID_ARG
