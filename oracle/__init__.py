"""fp64 CPU oracle for scaled dot-product attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library and its Python binding
never import it, and it imports nothing from them.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over heads
and rows). This module only compiles it (``build()``), loads it with ctypes
and converts arrays: bf16 inputs are upcast to fp64 exactly, so the oracle
sees the very bytes the GPU sees.

Functions:
  weights(q, k, causal, scale)             -> (S, P) of one head       (§3.2.1, Fig. 2)
  fwd(q, k, v, causal, scale, rows=None)   -> (O, lse)                 (eq. (1))
  bwd(q, k, v, dO, causal, scale)          -> (dQ, dK, dV, O, lse)     (derivative of eq. (1))
  bwd_rows(q, k, v, dO, causal, scale, qrows, krows) -> sampled rows of one head
  decode(q, k, v, scale, kv_len=None)      -> (O, lse) of one decoding step (§3, KV cache)
  project_qkv / project_out / multi_head   -> the projections around eq. (1) (§3.2.2)

Optional masks on fwd / bwd / bwd_rows: ``kv_len`` (key padding, per
sequence) and ``window=(wl, wr)`` (restricted self-attention, §4 and Table 1:
key j visible to query i only if i - wl <= j <= i + wr; a negative side is
open; None = no window).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (gcc, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
            lib.oracle_attn_weights.argtypes = [dp, dp, L, L, L, I, D, dp, dp]
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, L, I, D, lp, L, lp,
                                            L, L]
            lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                            L, L, L, L, L, L, I, D, lp, L, L]
            lib.oracle_attn_bwd_rows.argtypes = [dp, dp, dp, dp, L, L, L, L, I, D, lp, L, dp,
                                                 lp, L, dp, dp, L, L, L]
            lib.oracle_attn_bwd_rows.restype = ctypes.c_int
            for f in (lib.oracle_attn_weights, lib.oracle_attn_fwd, lib.oracle_attn_bwd):
                f.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact upcast to a C-contiguous float64 numpy array (bf16 -> fp64 is lossless)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as4(a: np.ndarray) -> np.ndarray:
    if a.ndim == 2:
        return a[None, None]
    if a.ndim == 3:
        return a[None]
    if a.ndim != 4:
        raise ValueError("expected a [S,d], [h,S,d] or [B,h,S,d] array")
    return a


def _check(status: int, what: str):
    if status != 0:
        raise RuntimeError(f"oracle {what} failed with status {status}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def weights(q, k, causal: bool, scale: float):
    """Scaled scores S (masked = -inf) and weights P of ONE head, each n x m."""
    Q, K = _f64(q), _f64(k)
    n, dk = Q.shape
    m = K.shape[0]
    S = np.empty((n, m))
    P = np.empty((n, m))
    _check(_load().oracle_attn_weights(_ptr(Q), _ptr(K), n, m, dk, int(causal), float(scale),
                                       _ptr(S), _ptr(P)), "weights")
    return S, P


def _window(window):
    """(wl, wr) as C longs; None -> (-1, -1), no window."""
    if window is None:
        return -1, -1
    wl, wr = window
    return int(wl), int(wr)


def _lens(kv_len, B):
    """Per-sequence real key counts as a C long array (None: no key padding)."""
    if kv_len is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int64).reshape(-1))
    if a.size != B:
        raise ValueError("kv_len needs one entry per sequence")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


def fwd(q, k, v, causal: bool, scale: float, rows: Optional[Sequence[int]] = None, kv_len=None,
        window=None):
    """O (fp64, shape of q with d_v) and lse ([..., n]) by eq. (1).

    With ``rows`` only those query rows are computed; the others are NaN.
    ``kv_len`` (one entry per sequence b): only the first kv_len[b] keys of
    sequence b are real, the rest are padding (masked).
    """
    Q, K, V = _as4(_f64(q)), _as4(_f64(k)), _as4(_f64(v))
    B, h, n, dk = Q.shape
    m, dv = K.shape[2], V.shape[3]
    if K.shape != (B, h, m, dk) or V.shape != (B, h, m, dv):
        raise ValueError("q/k/v shapes disagree")
    O = np.full((B, h, n, dv), np.nan)
    lse = np.full((B, h, n), np.nan)
    r = None
    nr = 0
    if rows is not None:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nr = int(r.size)
    lens, lens_p = _lens(kv_len, B)
    _check(_load().oracle_attn_fwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), B, h, n, m, dk, dv, int(causal),
        float(scale), None if r is None else r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
        nr, lens_p, *_window(window)), "fwd")
    shape_o = tuple(np.shape(q)[:-1]) + (dv,)
    return O.reshape(shape_o), lse.reshape(shape_o[:-1])


def bwd(q, k, v, dO, causal: bool, scale: float, need=("dq", "dk", "dv"), kv_len=None, window=None):
    """dQ, dK, dV of L = sum(dO * O) for O = Attention(q, k, v); also O and lse.

    ``kv_len``: per-sequence real key counts, as in ``fwd``.
    """
    Q, K, V, G = _as4(_f64(q)), _as4(_f64(k)), _as4(_f64(v)), _as4(_f64(dO))
    B, h, n, dk = Q.shape
    m, dv = K.shape[2], V.shape[3]
    if K.shape != (B, h, m, dk) or V.shape != (B, h, m, dv) or G.shape != (B, h, n, dv):
        raise ValueError("q/k/v/dO shapes disagree")
    dQ = np.zeros((B, h, n, dk)) if "dq" in need else None
    dK = np.zeros((B, h, m, dk)) if "dk" in need else None
    dV = np.zeros((B, h, m, dv)) if "dv" in need else None
    O = np.empty((B, h, n, dv))
    lse = np.empty((B, h, n))
    lens, lens_p = _lens(kv_len, B)
    _check(_load().oracle_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(G), _ptr(dQ), _ptr(dK),
                                   _ptr(dV), _ptr(O), _ptr(lse), B, h, n, m, dk, dv,
                                   int(causal), float(scale), lens_p, *_window(window)), "bwd")
    lead_q = tuple(q.shape[:-2])
    lead_k = tuple(k.shape[:-2])

    def shp(a, lead, S, d):
        return None if a is None else a.reshape(lead + (S, d))

    return (shp(dQ, lead_q, n, dk), shp(dK, lead_k, m, dk), shp(dV, lead_k, m, dv),
            O.reshape(lead_q + (n, dv)), lse.reshape(lead_q + (n,)))


def decode(q, k, v, scale: float, kv_len=None):
    """One incremental decoding step (§3: the decoder emits one symbol at a time,
    each step attending to the positions produced so far, itself included).

    q: [B, h, n, d] are the queries of the n newest positions of each sequence,
    k / v: [B, h, m, d] its cached keys and values, of which the first L_b =
    kv_len[b] (all m without kv_len) are real. Query i stands at position
    L_b - n + i and sees keys j <= L_b - n + i: the decoder's causal mask aligned
    to the end of the cache. Written with the masks above, per sequence: key
    padding L_b and the window's right side L_b - n. Returns (O, lse).
    """
    Q, K, V = _as4(_f64(q)), _as4(_f64(k)), _as4(_f64(v))
    B, h, n, _ = Q.shape
    m = K.shape[2]
    lens = [m] * B if kv_len is None else [int(x) for x in np.asarray(kv_len).reshape(-1)]
    if len(lens) != B:
        raise ValueError("kv_len needs one entry per sequence")
    O = np.empty(Q.shape[:3] + (V.shape[3],))
    lse = np.empty(Q.shape[:3])
    for b, L in enumerate(lens):
        L = min(max(L, 0), m)
        if L >= n:
            O[b:b + 1], lse[b:b + 1] = fwd(Q[b:b + 1], K[b:b + 1], V[b:b + 1], False, scale, kv_len=[L],
                                           window=(-1, L - n))
        else:
            # fewer cached positions than new queries: the first n - L queries
            # stand before the cache starts and see nothing (the empty sum)
            i0 = n - L
            O[b, :, :i0] = 0.0
            lse[b, :, :i0] = -np.inf
            if L > 0:
                O[b:b + 1, :, i0:], lse[b:b + 1, :, i0:] = fwd(Q[b:b + 1, :, i0:], K[b:b + 1], V[b:b + 1], True,
                                                               scale, kv_len=[L])
    return O, lse


def project_qkv(x_q, x_kv, w_qkv, h: int, d: int):
    """The multi-head projections of §3.2.2: Q = x_q W^Q, K = x_kv W^K, V = x_kv W^V.

    x_q: [B, n, d_model], x_kv: [B, m, d_model]; w_qkv: [d_model, 3 h d], the
    column blocks W^Q | W^K | W^V, head i's d columns at i d within each (the
    pages' W_i^Q in R^{d_model x d_k}). Returns q [B, h, n, d], k, v [B, h, m, d] (fp64).
    """
    Xq, Xkv, W = _f64(x_q), _f64(x_kv), _f64(w_qkv)
    hd = h * d
    if W.shape != (Xq.shape[-1], 3 * hd):
        raise ValueError("w_qkv must be [d_model, 3 h d]")

    def heads(Y):  # [B, S, h d] -> [B, h, S, d]
        B, S, _ = Y.shape
        return np.ascontiguousarray(Y.reshape(B, S, h, d).transpose(0, 2, 1, 3))

    return heads(Xq @ W[:, :hd]), heads(Xkv @ W[:, hd:2 * hd]), heads(Xkv @ W[:, 2 * hd:])


def project_out(o, w_o):
    """Concat(head_1, ..., head_h) W^O (§3.2.2): o [B, h, n, d], w_o [h d, d_model] -> [B, n, d_model]."""
    O, W = _f64(o), _f64(w_o)
    B, h, n, d = O.shape
    if W.shape[0] != h * d:
        raise ValueError("w_o must be [h d, d_model]")
    return O.transpose(0, 2, 1, 3).reshape(B, n, h * d) @ W


def project_qkv_bwd(x_q, x_kv, w_qkv, dq, dk, dv):
    """Gradients of project_qkv for upstream gradients dq [B, h, n, d], dk, dv [B, h, m, d].

    The projections are linear, y = x W, so dx = dy W^T and dW = sum over the
    batch's tokens of x^T dy, with the head split undone (Concat of the heads'
    columns, §3.2.2). Returns dx_q [B, n, d_model], dx_kv [B, m, d_model] and
    dw_qkv [d_model, 3 h d] (fp64).
    """
    Xq, Xkv, W = _f64(x_q), _f64(x_kv), _f64(w_qkv)
    Gq, Gk, Gv = _f64(dq), _f64(dk), _f64(dv)
    B, h, n, d = Gq.shape
    hd = h * d

    def concat(G):  # [B, h, S, d] -> [B, S, h d]
        b, hh, S, dd = G.shape
        return G.transpose(0, 2, 1, 3).reshape(b, S, hh * dd)

    Cq, Ck, Cv = concat(Gq), concat(Gk), concat(Gv)
    dx_q = Cq @ W[:, :hd].T
    dx_kv = Ck @ W[:, hd:2 * hd].T + Cv @ W[:, 2 * hd:].T
    dw = np.concatenate([np.einsum("bsc,bsj->cj", Xq, Cq), np.einsum("bsc,bsj->cj", Xkv, Ck),
                         np.einsum("bsc,bsj->cj", Xkv, Cv)], axis=1)
    return dx_q, dx_kv, dw


def project_out_bwd(o, w_o, dy):
    """Gradients of project_out for dy [B, n, d_model]: d_o = dy (W^O)^T back in the
    [B, h, n, d] layout, dw_o = sum over tokens of Concat(o)^T dy [h d, d_model] (fp64)."""
    O, W, G = _f64(o), _f64(w_o), _f64(dy)
    B, h, n, d = O.shape
    C = O.transpose(0, 2, 1, 3).reshape(B, n, h * d)
    d_o = (G @ W.T).reshape(B, n, h, d).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(d_o), np.einsum("bsj,bsc->jc", C, G)


def multi_head(x_q, x_kv, w_qkv, w_o, h: int, d: int, causal: bool = False, scale=None):
    """MultiHead(Q, K, V) = Concat(head_1..head_h) W^O, head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V)."""
    q, k, v = project_qkv(x_q, x_kv, w_qkv, h, d)
    O, _ = fwd(q, k, v, causal, 1.0 / np.sqrt(d) if scale is None else scale)
    return project_out(O, w_o)


def bwd_rows(q, k, v, dO, causal: bool, scale: float, qrows=(), krows=(), kv_len=None, window=None):
    """Sampled backward of ONE head: (dQ[qrows], dK[krows], dV[krows]), fp64.

    q, dO: [n, d]; k, v: [m, d]. Key rows cost a full forward of the head.
    ``kv_len``: the head's real key count (None: all m).
    """
    Q, K, V, G = _f64(q), _f64(k), _f64(v), _f64(dO)
    n, dk = Q.shape
    m, dv = K.shape[0], V.shape[1]
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64).reshape(-1))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int64).reshape(-1))
    dQ = np.empty((max(qr.size, 1), dk))
    dK = np.empty((max(kr.size, 1), dk))
    dV = np.empty((max(kr.size, 1), dv))
    lp = ctypes.POINTER(ctypes.c_long)
    _check(_load().oracle_attn_bwd_rows(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(G), n, m, dk, dv, int(causal), float(scale),
        qr.ctypes.data_as(lp), qr.size, _ptr(dQ), kr.ctypes.data_as(lp), kr.size, _ptr(dK),
        _ptr(dV), -1 if kv_len is None else int(kv_len), *_window(window)), "bwd_rows")
    return dQ[: qr.size], dK[: kr.size], dV[: kr.size]
