"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerance (per output tensor, fixed for bf16 inputs with fp32 accumulation):
  ||gpu - ref||_2 / ||ref||_2 <= 5e-3, and
  max |gpu - ref| <= 1e-2 at every element, except where that bound is below
  bf16's own resolution: an element whose error exceeds 1e-2 passes only if
  the GPU value lies within one bf16 ulp of the fp64 oracle value. For
  |ref| >= 4 the bf16 spacing is >= 2^-5, so even the correctly rounded fp64
  result can be 0.0156 away; no bf16 output can meet 1e-2 there. (Large
  values occur in gradients of rows that see few keys, e.g. dV_0 = sum_i dO_i
  when m = 1, and in the saturated Q x 4 variant.)
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
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g - r)
    return float(d.max()) if d.size else 0.0, float(rel)


def ulp_ratio(gpu, ref) -> float:
    """max |gpu - ref| / ulp_bf16(ref): errors in units of bf16 spacing at the oracle value."""
    g, r = to64(gpu), to64(ref)
    if g.size == 0:
        return 0.0
    return float((np.abs(g - r) / bf16_ulp(r)).max())


def assert_close(name, gpu, ref, max_abs=MAX_ABS, rel_l2=REL_L2):
    g, r = to64(gpu), to64(ref)
    ma, rl = errors(g, r)
    assert rl <= rel_l2, f"{name}: rel_l2={rl:.3e} (<= {rel_l2}), max_abs={ma:.3e}"
    if ma > max_abs:
        d = np.abs(g - r)
        bad = d > max_abs
        within_ulp = d[bad] <= bf16_ulp(r[bad])
        assert within_ulp.all(), (
            f"{name}: max_abs={ma:.3e} > {max_abs} at {int((~within_ulp).sum())} element(s) "
            f"more than one bf16 ulp from the oracle (max ulp ratio {ulp_ratio(g, r):.2f})")
    return ma, rl


def default_scale(d):
    return 1.0 / math.sqrt(d)
