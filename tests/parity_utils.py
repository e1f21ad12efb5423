"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerance (per output tensor, bf16 inputs with fp32 accumulation):
  relative L2:  ||gpu - ref||_2 / ||ref||_2 <= 5e-3 over the tensor (at full
                sizes, over uniformly sampled rows, an unbiased estimate);
  max-abs:      |gpu - ref| <= 1e-2 at every element, with two exemptions
                where bf16 cannot resolve 1e-2:
   (a) every output: the GPU value lies within one bf16 ulp of the fp64
       oracle value. For |ref| >= 4 the bf16 spacing is >= 2^-5, so even the
       correctly rounded oracle value can be 0.0156 away.
   (b) gradients (dQ, dK, dV) only: the error is within two bf16 ulps of the
       largest |ref| in the same row. A gradient row is a sum of products
       that passes through three bf16 roundings of relative size 2^-9 (the
       weights P before P.V, O and hence D_i = dO_i . O_i, and dS before the
       dQ / dK products); their errors scale with the row's terms, not with
       the element, and in rows that see only a few keys (the first rows
       under the causal mask, saturated softmax) the terms cancel, so an
       element near zero can carry an error near 2^-8 of the row scale.
  For dQ and dK the max-abs bound also admits the first-order effect of the
  interface's bf16 O on D_i (``d_term_bounds``): the backward receives O in
  bf16, so D_i moves by up to 2^-8 sum_c |dO_ic||O_ic|, which moves dQ_ic by
  |scale| |dD_i| (P|K|)_ic and dK_jc by |scale| (P^T (|dD| |Q|))_jc. Both are
  computed by the oracle (attention with values |K|; the backward with a
  synthetic upstream gradient), never from the GPU outputs.
"""
import math

import numpy as np
import torch

MAX_ABS = 1e-2
REL_L2 = 5e-3


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def errors(gpu, ref):
    g, r = to64(gpu), to64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values in GPU output"
    d = np.abs(g - r)
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else 0.0
    return float(d.max()) if d.size else 0.0, float(rel)


def ulp_ratio(gpu, ref) -> float:
    """max |gpu - ref| / ulp_bf16(ref): errors in units of bf16 spacing at the oracle value."""
    g, r = to64(gpu), to64(ref)
    if g.size == 0:
        return 0.0
    return float((np.abs(g - r) / bf16_ulp(r)).max())


def d_term_bounds(q, k, v, dO, causal, scale, qrows=None, krows=None, kv_len=None, window=None):
    """Bounds on |dQ| and |dK| errors caused by forming D_i from the bf16 O (see module doc).

    Full heads ([B,h,S,d] tensors) when qrows/krows are None; otherwise ONE head
    ([S,d] tensors) and the bounds of the listed query / key rows; kv_len is
    then that head's real key count (key padding). kv_len (per sequence, full
    heads) and window (left, right) are the masks of the call checked.
    """
    import oracle
    u = 2.0 ** -8
    qa, ka, va, da = to64(q), to64(k), to64(v), to64(dO)
    if qrows is None:
        O, _ = oracle.fwd(qa, ka, va, causal, scale, kv_len=kv_len, window=window)
        PK, _ = oracle.fwd(qa, ka, np.abs(ka), causal, scale, kv_len=kv_len, window=window)
        dD = u * (np.abs(da) * np.abs(O)).sum(axis=-1)
        bq = abs(scale) * dD[..., None] * PK
        # dK bound: P^T (|dD| |q|), i.e. the dV of a backward whose upstream gradient is |dD| |q|
        _, _, PtdDq, _, _ = oracle.bwd(qa, ka, ka, dD[..., None] * np.abs(qa), causal, scale, kv_len=kv_len,
                                       window=window)
        return bq, abs(scale) * PtdDq
    n = qa.shape[0]
    all_rows = list(range(n))
    lens = None if kv_len is None else [kv_len]
    O, _ = oracle.fwd(qa, ka, va, causal, scale, rows=all_rows, kv_len=lens, window=window)
    dD = u * (np.abs(da) * np.abs(O)).sum(axis=-1)
    PK, _ = oracle.fwd(qa, ka, np.abs(ka), causal, scale, rows=list(qrows), kv_len=lens, window=window)
    bq = abs(scale) * dD[list(qrows), None] * PK[list(qrows)]
    bk = None
    if krows is not None and len(krows):
        _, _, PtdDq = oracle.bwd_rows(qa, ka, ka, dD[:, None] * np.abs(qa), causal, scale, [], krows,
                                      kv_len=kv_len, window=window)
        bk = abs(scale) * PtdDq
    return bq, bk


def assert_close(name, gpu, ref, max_abs=MAX_ABS, rel_l2=REL_L2, grad=False, rel_rows=None,
                 extra=None):
    """Check one output tensor; rows are the second-to-last axis.

    grad: apply exemption (b) for gradient tensors.
    rel_rows: indices (along the row axis) of a uniform sample used for the
    relative-L2 estimate; default: all rows given.
    extra: per-element bound added to max_abs (the D-term of ``d_term_bounds``).
    """
    g, r = to64(gpu), to64(ref)
    ma, _ = errors(g, r)
    if rel_rows is not None:
        _, rl = errors(np.take(g, rel_rows, axis=-2), np.take(r, rel_rows, axis=-2))
    else:
        _, rl = errors(g, r)
    # relative L2 is undefined against an all-zero oracle (e.g. dQ with one key);
    # the max-abs bound below still applies there
    if np.any(r != 0):
        assert rl <= rel_l2, f"{name}: rel_l2={rl:.3e} (<= {rel_l2}), max_abs={ma:.3e}"
    if ma > max_abs:
        d = np.abs(g - r)
        bad = d > max_abs
        allowed = bf16_ulp(r)
        if extra is not None:
            allowed = np.maximum(allowed, max_abs + to64(extra))
        if grad and r.ndim >= 1:
            row_max = np.abs(r).max(axis=-1, keepdims=True)
            allowed = np.maximum(allowed, 2.0 * bf16_ulp(np.broadcast_to(row_max, r.shape)))
        ok = d[bad] <= allowed[bad]
        assert ok.all(), (
            f"{name}: max_abs={ma:.3e} > {max_abs} at {int((~ok).sum())} element(s) beyond the "
            f"bf16 exemption (max ulp ratio {ulp_ratio(g, r):.2f})")
    return ma, rl


def default_scale(d):
    return 1.0 / math.sqrt(d)
