"""GB300 (sm_103a) multi-head scaled dot-product attention.

Python binding of the C ABI declared in ``include/attn.h``. It only checks and
marshals arguments (torch tensors give device pointers and the current CUDA
stream); every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is not built, calls raise.

    O = softmax(Q K^T * scale) V      ("Attention Is All You Need", §3.2.1 eq. (1))

Tensors are bf16, contiguous, shaped [B, h, S, d] (d fastest); lse is fp32
[B, h, n]. ``scale`` defaults to 1/sqrt(d_k). ``causal`` applies the decoder
mask of §3.2.3 (key j visible to query i iff j <= i).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

from .native_build import LIB_PATH, build  # noqa: F401  (re-exported for __graft_entry__)

__all__ = [
    "AttnError", "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA",
    "ATTN_ERR_TIMEOUT", "load_library", "library_path", "attn_fwd", "attn_bwd",
    "attn_bwd_workspace_bytes", "attn_get_device_status", "attn_status_string",
    "attn_set_watchdog_ns", "attn_debug_inject", "attn_profile_enable", "attn_profile_read",
    "attn_bwd_noalloc", "attn_decode", "attn_decode_workspace_bytes",
    "attn_qkv_projection", "attn_out_projection", "attn_qkv_projection_bwd", "attn_out_projection_bwd",
    "attn_qkv_projection_bwd_workspace_bytes", "attn_out_projection_bwd_workspace_bytes",
    "attn_fwd_bwd_host", "HostStepBuffers", "EXPORTED_SYMBOLS", "KERNEL_KINDS",
]
# attn_fwd / attn_bwd take an optional ``kv_len`` (int32 CUDA tensor [B]: real
# keys per sequence) and an optional ``window`` = (left, right) (restricted
# self-attention: query i sees keys i - left .. i + right, None or a negative
# side = open); with either they call attn_fwd_masked / attn_bwd_masked.

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4

# Every entry point include/attn.h declares.
EXPORTED_SYMBOLS = (
    "attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_get_device_status",
    "attn_status_string", "attn_set_watchdog_ns", "attn_debug_inject", "attn_profile_enable",
    "attn_profile_read", "attn_bwd_noalloc", "attn_fwd_varlen",
    "attn_bwd_varlen", "attn_fwd_masked", "attn_bwd_masked", "attn_decode_workspace_bytes", "attn_decode",
    "attn_qkv_projection", "attn_out_projection", "attn_qkv_projection_bwd_workspace_bytes",
    "attn_qkv_projection_bwd", "attn_out_projection_bwd_workspace_bytes", "attn_out_projection_bwd",
    "attn_fwd_bwd_host",
)

# Kernel kinds of attn_profile_read.
KERNEL_KINDS = {"fwd": 0, "bwd_pre": 1, "bwd_main": 2, "bwd_post": 3, "decode": 4, "decode_merge": 5, "proj": 6}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} ({status})")


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load ``libattn_gb300.so`` (ctypes) and declare every entry point's signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        vp, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        fp = ctypes.POINTER(ctypes.c_float)
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, fp, I, I, I, I, I, I, I, F, vp]
        lib.attn_fwd.restype = I
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, I, I, I, I, I, I, I, F,
                                 vp, SZ, vp]
        lib.attn_bwd.restype = I
        lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, fp, vp, I, I, I, I, I, I, I, F, vp]
        lib.attn_fwd_varlen.restype = I
        lib.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, vp, I, I, I, I, I, I, I, F,
                                        vp, SZ, vp]
        lib.attn_bwd_varlen.restype = I
        lib.attn_fwd_masked.argtypes = [vp, vp, vp, vp, fp, vp, I, I, I, I, I, I, I, I, I, F, vp]
        lib.attn_fwd_masked.restype = I
        lib.attn_bwd_masked.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, vp, I, I, I, I, I, I, I, I, I,
                                        F, vp, SZ, vp]
        lib.attn_bwd_masked.restype = I
        lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.attn_decode_workspace_bytes.restype = SZ
        lib.attn_decode.argtypes = [vp, vp, vp, vp, fp, vp, I, I, I, I, I, I, F, vp, SZ, vp]
        lib.attn_decode.restype = I
        lib.attn_qkv_projection.argtypes = [vp, vp, vp, vp, vp, vp, I, I, I, I, I, I, vp]
        lib.attn_qkv_projection.restype = I
        lib.attn_out_projection.argtypes = [vp, vp, vp, I, I, I, I, I, vp]
        lib.attn_out_projection.restype = I
        lib.attn_qkv_projection_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.attn_qkv_projection_bwd_workspace_bytes.restype = SZ
        lib.attn_qkv_projection_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, I, vp, SZ, vp]
        lib.attn_qkv_projection_bwd.restype = I
        lib.attn_out_projection_bwd_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.attn_out_projection_bwd_workspace_bytes.restype = SZ
        lib.attn_out_projection_bwd.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, vp, SZ, vp]
        lib.attn_out_projection_bwd.restype = I
        lib.attn_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, fp, vp, vp, vp, vp, vp, vp, vp, vp, fp, vp, vp, vp,
                                          vp, SZ, I, I, I, I, I, I, I, F, I, vp]
        lib.attn_fwd_bwd_host.restype = I
        lib.attn_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
        lib.attn_bwd_workspace_bytes.restype = SZ
        lib.attn_get_device_status.argtypes = [vp]
        lib.attn_get_device_status.restype = I
        lib.attn_status_string.argtypes = [I]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_set_watchdog_ns.argtypes = [ctypes.c_ulonglong]
        lib.attn_set_watchdog_ns.restype = I
        lib.attn_debug_inject.argtypes = [I]
        lib.attn_debug_inject.restype = I
        lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, I, I, I, I, I, I, I, F,
                                         vp]
        lib.attn_bwd_noalloc.restype = I
        lib.attn_profile_enable.argtypes = [I]
        lib.attn_profile_enable.restype = I
        lib.attn_profile_read.argtypes = [I, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double)]
        lib.attn_profile_read.restype = I
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_tensor(name, t, shape=None, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _fptr(t):
    return None if t is None else ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_float))


def _vptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_lengths(kv_len, B, device):
    import torch
    if kv_len is None:
        return None
    _check_tensor("kv_len", kv_len, (B,), torch.int32)
    if kv_len.device != device:
        raise ValueError("kv_len must be on the device of q")
    return _vptr(kv_len)


def _window(window):
    """(left, right) as C ints, -1 for an open side; None when there is no window."""
    if window is None:
        return None
    wl, wr = window
    wl = -1 if wl is None or int(wl) < 0 else int(wl)
    wr = -1 if wr is None or int(wr) < 0 else int(wr)
    if wl > 0x7fffffff or wr > 0x7fffffff:
        raise ValueError("window sides must fit in int32")
    return None if (wl < 0 and wr < 0) else (wl, wr)


def attn_fwd(q, k, v, causal: bool = False, scale: Optional[float] = None, out=None, lse=None,
             need_lse: bool = True, stream=None, kv_len=None,
             window=None) -> Tuple["torch.Tensor", Optional["torch.Tensor"]]:
    """O, lse = attention(q, k, v) on the GPU. q [B,h,n,d], k/v [B,h,m,d], bf16.

    kv_len (optional int32 CUDA tensor [B]): real keys per sequence; the keys
    past them are padding and masked.
    window (optional (left, right)): query i sees only keys i - left .. i + right.
    """
    import torch
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, S, d]")
    B, h, n, dk = q.shape
    m, dv = k.shape[2], v.shape[3]
    _check_tensor("q", q, dtype=torch.bfloat16)
    _check_tensor("k", k, (B, h, m, dk), torch.bfloat16)
    _check_tensor("v", v, (B, h, m, dv), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if out is None:
        out = torch.empty((B, h, n, dv), dtype=torch.bfloat16, device=q.device)
    _check_tensor("out", out, (B, h, n, dv), torch.bfloat16)
    if need_lse and lse is None:
        lse = torch.empty((B, h, n), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor("lse", lse, (B, h, n), torch.float32)
    lens = _check_lengths(kv_len, B, q.device)
    win = _window(window)
    if win is not None:
        st = lib.attn_fwd_masked(_vptr(q), _vptr(k), _vptr(v), _vptr(out), _fptr(lse), lens, B, h, n,
                                 m, dk, dv, int(bool(causal)), win[0], win[1], float(scale),
                                 _stream_handle(stream))
    elif lens is None:
        st = lib.attn_fwd(_vptr(q), _vptr(k), _vptr(v), _vptr(out), _fptr(lse), B, h, n, m, dk, dv,
                          int(bool(causal)), float(scale), _stream_handle(stream))
    else:
        st = lib.attn_fwd_varlen(_vptr(q), _vptr(k), _vptr(v), _vptr(out), _fptr(lse), lens, B, h, n,
                                 m, dk, dv, int(bool(causal)), float(scale), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")
    return out, lse


def attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal=False) -> int:
    return int(load_library().attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, int(bool(causal))))


def attn_bwd(q, k, v, o, lse, dO, causal: bool = False, scale: Optional[float] = None,
             dq=None, dk=None, dv=None, workspace=None, stream=None, kv_len=None, window=None):
    """dQ, dK, dV of sum(dO * O) for O = attention(q, k, v), from attn_fwd's O and lse
    (the same causal, kv_len and window as the forward)."""
    import torch
    lib = load_library()
    B, h, n, d_k = q.shape
    m, d_v = k.shape[2], v.shape[3]
    _check_tensor("q", q, dtype=torch.bfloat16)
    _check_tensor("k", k, (B, h, m, d_k), torch.bfloat16)
    _check_tensor("v", v, (B, h, m, d_v), torch.bfloat16)
    _check_tensor("o", o, (B, h, n, d_v), torch.bfloat16)
    _check_tensor("lse", lse, (B, h, n), torch.float32)
    _check_tensor("dO", dO, (B, h, n, d_v), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _check_tensor(name, t, tuple(ref.shape), torch.bfloat16)
    need = attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal)
    if workspace is None and need > 0:
        workspace = torch.empty((need + 15) // 16 * 4, dtype=torch.float32, device=q.device)
    if workspace is not None:
        _check_tensor("workspace", workspace)
    ws_ptr = _vptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lens = _check_lengths(kv_len, B, q.device)
    win = _window(window)
    if win is not None:
        st = lib.attn_bwd_masked(_vptr(q), _vptr(k), _vptr(v), _vptr(o), _fptr(lse), _vptr(dO),
                                 _vptr(dq), _vptr(dk), _vptr(dv), lens, B, h, n, m, d_k, d_v,
                                 int(bool(causal)), win[0], win[1], float(scale), ws_ptr, ws_bytes,
                                 _stream_handle(stream))
    elif lens is None:
        st = lib.attn_bwd(_vptr(q), _vptr(k), _vptr(v), _vptr(o), _fptr(lse), _vptr(dO), _vptr(dq),
                          _vptr(dk), _vptr(dv), B, h, n, m, d_k, d_v, int(bool(causal)), float(scale),
                          ws_ptr, ws_bytes, _stream_handle(stream))
    else:
        st = lib.attn_bwd_varlen(_vptr(q), _vptr(k), _vptr(v), _vptr(o), _fptr(lse), _vptr(dO),
                                 _vptr(dq), _vptr(dk), _vptr(dv), lens, B, h, n, m, d_k, d_v,
                                 int(bool(causal)), float(scale), ws_ptr, ws_bytes,
                                 _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


class HostStepBuffers:
    """Device buffers of attn_fwd_bwd_host for one set of sizes (allocated once,
    reused by every call): q, k, v, dO, o, lse, dq, dk, dv and the workspace."""

    def __init__(self, B, h, n, m, d_k, d_v, causal=False, device=None):
        import torch
        dev = torch.device("cuda") if device is None else torch.device(device)
        bf = torch.bfloat16
        self.shape = (B, h, n, m, d_k, d_v)
        self.q = torch.empty((B, h, n, d_k), dtype=bf, device=dev)
        self.k = torch.empty((B, h, m, d_k), dtype=bf, device=dev)
        self.v = torch.empty((B, h, m, d_v), dtype=bf, device=dev)
        self.dO = torch.empty((B, h, n, d_v), dtype=bf, device=dev)
        self.o = torch.empty((B, h, n, d_v), dtype=bf, device=dev)
        self.lse = torch.empty((B, h, n), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.v)
        need = attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal)
        self.workspace = torch.empty(max(need, 16) // 4 + 4, dtype=torch.float32, device=dev)


def _check_host(name, t, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")


def attn_fwd_bwd_host(q, k, v, dO, causal: bool = False, scale: Optional[float] = None, out=None,
                      buffers: Optional[HostStepBuffers] = None, chunks: int = 0, need_lse: bool = True,
                      stream=None):
    """Forward and backward with HOST inputs and results: q, dO [B,h,n,d], k, v
    [B,h,m,d] bf16 CPU tensors (page-locked for the copies to overlap).

    Returns host tensors (O, lse, dQ, dK, dV) (lse None when need_lse is False);
    ``out`` may give them (same order). ``buffers`` holds the device memory
    (allocated here when None). The copies and kernels are enqueued on
    ``stream``'s device and the call returns without waiting: synchronise the
    stream before reading the results."""
    import torch
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, S, d]")
    B, h, n, d_k = q.shape
    m, d_v = k.shape[2], v.shape[3]
    bf = torch.bfloat16
    for name, t, shp in (("q", q, (B, h, n, d_k)), ("k", k, (B, h, m, d_k)), ("v", v, (B, h, m, d_v)),
                         ("dO", dO, (B, h, n, d_v))):
        _check_host(name, t, shp, bf)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    if buffers is None:
        buffers = HostStepBuffers(B, h, n, m, d_k, d_v, causal)
    if buffers.shape != (B, h, n, m, d_k, d_v):
        raise ValueError(f"buffers are for sizes {buffers.shape}, not {(B, h, n, m, d_k, d_v)}")
    pin = torch.cuda.is_available()
    if out is None:
        out = (torch.empty((B, h, n, d_v), dtype=bf, pin_memory=pin),
               torch.empty((B, h, n), dtype=torch.float32, pin_memory=pin) if need_lse else None,
               torch.empty((B, h, n, d_k), dtype=bf, pin_memory=pin),
               torch.empty((B, h, m, d_k), dtype=bf, pin_memory=pin),
               torch.empty((B, h, m, d_v), dtype=bf, pin_memory=pin))
    ho, hlse, hdq, hdk, hdv = out
    _check_host("out O", ho, (B, h, n, d_v), bf)
    if hlse is not None:
        _check_host("out lse", hlse, (B, h, n), torch.float32)
    _check_host("out dQ", hdq, (B, h, n, d_k), bf)
    _check_host("out dK", hdk, (B, h, m, d_k), bf)
    _check_host("out dV", hdv, (B, h, m, d_v), bf)
    b = buffers
    ws = b.workspace
    st = lib.attn_fwd_bwd_host(_vptr(q), _vptr(k), _vptr(v), _vptr(dO), _vptr(ho), _fptr(hlse), _vptr(hdq),
                               _vptr(hdk), _vptr(hdv), _vptr(b.q), _vptr(b.k), _vptr(b.v), _vptr(b.dO),
                               _vptr(b.o), _fptr(b.lse), _vptr(b.dq), _vptr(b.dk), _vptr(b.dv), _vptr(ws),
                               ws.numel() * ws.element_size(), B, h, n, m, d_k, d_v, int(bool(causal)),
                               float(scale), int(chunks), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_bwd_host")
    return ho, hlse, hdq, hdk, hdv


def attn_decode_workspace_bytes(B, h, n, m, d_k, d_v) -> int:
    return int(load_library().attn_decode_workspace_bytes(B, h, n, m, d_k, d_v))


def attn_decode(q, k, v, kv_len=None, scale: Optional[float] = None, out=None, lse=None,
                need_lse: bool = True, workspace=None, stream=None):
    """One decoding step: q [B,h,n,d] (the n newest positions, n <= 16) against the
    caches k, v [B,h,m,d]; kv_len (optional int32 CUDA [B]) cached positions per
    sequence (default m). Query i sees keys j <= L - n + i. Returns (O, lse)."""
    import torch
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, S, d]")
    B, h, n, dk = q.shape
    m, dv = k.shape[2], v.shape[3]
    _check_tensor("q", q, dtype=torch.bfloat16)
    _check_tensor("k", k, (B, h, m, dk), torch.bfloat16)
    _check_tensor("v", v, (B, h, m, dv), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if out is None:
        out = torch.empty((B, h, n, dv), dtype=torch.bfloat16, device=q.device)
    _check_tensor("out", out, (B, h, n, dv), torch.bfloat16)
    if need_lse and lse is None:
        lse = torch.empty((B, h, n), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor("lse", lse, (B, h, n), torch.float32)
    lens = _check_lengths(kv_len, B, q.device)
    need = attn_decode_workspace_bytes(B, h, n, m, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 16) // 4 + 4, dtype=torch.float32, device=q.device)
    _check_tensor("workspace", workspace)
    st = lib.attn_decode(_vptr(q), _vptr(k), _vptr(v), _vptr(out), _fptr(lse), lens, B, h, n, m, dk, dv,
                         float(scale), _vptr(workspace), workspace.numel() * workspace.element_size(),
                         _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode")
    return out, lse


def attn_qkv_projection(x_q, x_kv, w_qkv, h: int, d: int, q=None, k=None, v=None, stream=None):
    """Q = x_q W^Q, K = x_kv W^K, V = x_kv W^V into [B, h, S, d] (§3.2.2).

    x_q [B, n, d_model], x_kv [B, m, d_model] (the same tensor for
    self-attention), w_qkv [d_model, 3 h d] (W^Q | W^K | W^V), all bf16 CUDA."""
    import torch
    lib = load_library()
    if x_q.dim() != 3 or x_kv.dim() != 3:
        raise ValueError("x_q, x_kv must be [B, S, d_model]")
    B, n, dm = x_q.shape
    m = x_kv.shape[1]
    _check_tensor("x_q", x_q, dtype=torch.bfloat16)
    _check_tensor("x_kv", x_kv, (B, m, dm), torch.bfloat16)
    _check_tensor("w_qkv", w_qkv, (dm, 3 * h * d), torch.bfloat16)
    q = torch.empty((B, h, n, d), dtype=torch.bfloat16, device=x_q.device) if q is None else q
    k = torch.empty((B, h, m, d), dtype=torch.bfloat16, device=x_q.device) if k is None else k
    v = torch.empty((B, h, m, d), dtype=torch.bfloat16, device=x_q.device) if v is None else v
    _check_tensor("q", q, (B, h, n, d), torch.bfloat16)
    _check_tensor("k", k, (B, h, m, d), torch.bfloat16)
    _check_tensor("v", v, (B, h, m, d), torch.bfloat16)
    st = lib.attn_qkv_projection(_vptr(x_q), _vptr(x_kv), _vptr(w_qkv), _vptr(q), _vptr(k), _vptr(v),
                                 B, n, m, dm, h, d, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_qkv_projection")
    return q, k, v


def attn_out_projection(o, w_o, y=None, stream=None):
    """y = Concat(head_1..h) W^O from o [B, h, n, d] and w_o [h d, d_model], bf16 CUDA (§3.2.2)."""
    import torch
    lib = load_library()
    if o.dim() != 4:
        raise ValueError("o must be [B, h, n, d]")
    B, h, n, d = o.shape
    _check_tensor("o", o, dtype=torch.bfloat16)
    if w_o.dim() != 2 or w_o.shape[0] != h * d:
        raise ValueError("w_o must be [h d, d_model]")
    dm = w_o.shape[1]
    _check_tensor("w_o", w_o, (h * d, dm), torch.bfloat16)
    y = torch.empty((B, n, dm), dtype=torch.bfloat16, device=o.device) if y is None else y
    _check_tensor("y", y, (B, n, dm), torch.bfloat16)
    st = lib.attn_out_projection(_vptr(o), _vptr(w_o), _vptr(y), B, n, dm, h, d, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_out_projection")
    return y


def attn_qkv_projection_bwd_workspace_bytes(B, n, m, d_model, h, d) -> int:
    return int(load_library().attn_qkv_projection_bwd_workspace_bytes(B, n, m, d_model, h, d))


def attn_out_projection_bwd_workspace_bytes(B, n, d_model, h, d) -> int:
    return int(load_library().attn_out_projection_bwd_workspace_bytes(B, n, d_model, h, d))


def attn_qkv_projection_bwd(x_q, x_kv, w_qkv, dq, dk, dv, dx_q=None, dx_kv=None, dw_qkv=None, workspace=None,
                            stream=None):
    """Gradients of attn_qkv_projection: dx_q, dx_kv [B, S, d_model] and dw_qkv [d_model, 3 h d]
    from dq [B, h, n, d], dk, dv [B, h, m, d] (bf16 CUDA). Self-attention (x_q is x_kv) with
    dx_kv omitted: dx_q is the whole input gradient and dx_kv is returned as the same tensor."""
    import torch
    lib = load_library()
    if dq.dim() != 4 or dk.dim() != 4:
        raise ValueError("dq, dk, dv must be [B, h, S, d]")
    B, h, n, d = dq.shape
    m = dk.shape[2]
    dm = x_q.shape[2]
    _check_tensor("x_q", x_q, (B, n, dm), torch.bfloat16)
    _check_tensor("x_kv", x_kv, (B, m, dm), torch.bfloat16)
    _check_tensor("w_qkv", w_qkv, (dm, 3 * h * d), torch.bfloat16)
    _check_tensor("dq", dq, (B, h, n, d), torch.bfloat16)
    _check_tensor("dk", dk, (B, h, m, d), torch.bfloat16)
    _check_tensor("dv", dv, (B, h, m, d), torch.bfloat16)
    dev = dq.device
    self_attn = x_q.data_ptr() == x_kv.data_ptr() and n == m
    if dx_q is None:
        dx_q = torch.empty((B, n, dm), dtype=torch.bfloat16, device=dev)
    if dx_kv is None:
        dx_kv = dx_q if self_attn else torch.empty((B, m, dm), dtype=torch.bfloat16, device=dev)
    if dw_qkv is None:
        dw_qkv = torch.empty((dm, 3 * h * d), dtype=torch.bfloat16, device=dev)
    _check_tensor("dx_q", dx_q, (B, n, dm), torch.bfloat16)
    _check_tensor("dx_kv", dx_kv, (B, m, dm), torch.bfloat16)
    _check_tensor("dw_qkv", dw_qkv, (dm, 3 * h * d), torch.bfloat16)
    need = lib.attn_qkv_projection_bwd_workspace_bytes(B, n, m, dm, h, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib.attn_qkv_projection_bwd(_vptr(x_q), _vptr(x_kv), _vptr(w_qkv), _vptr(dq), _vptr(dk), _vptr(dv),
                                     _vptr(dx_q), _vptr(dx_kv), _vptr(dw_qkv), B, n, m, dm, h, d,
                                     _vptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_qkv_projection_bwd")
    return dx_q, dx_kv, dw_qkv


def attn_out_projection_bwd(o, w_o, dy, d_o=None, dw_o=None, workspace=None, stream=None):
    """Gradients of attn_out_projection: d_o [B, h, n, d] (attn_fwd's layout) and
    dw_o [h d, d_model] from dy [B, n, d_model] (bf16 CUDA)."""
    import torch
    lib = load_library()
    if o.dim() != 4:
        raise ValueError("o must be [B, h, n, d]")
    B, h, n, d = o.shape
    dm = w_o.shape[1]
    _check_tensor("o", o, (B, h, n, d), torch.bfloat16)
    _check_tensor("w_o", w_o, (h * d, dm), torch.bfloat16)
    _check_tensor("dy", dy, (B, n, dm), torch.bfloat16)
    dev = o.device
    d_o = torch.empty((B, h, n, d), dtype=torch.bfloat16, device=dev) if d_o is None else d_o
    dw_o = torch.empty((h * d, dm), dtype=torch.bfloat16, device=dev) if dw_o is None else dw_o
    _check_tensor("d_o", d_o, (B, h, n, d), torch.bfloat16)
    _check_tensor("dw_o", dw_o, (h * d, dm), torch.bfloat16)
    need = lib.attn_out_projection_bwd_workspace_bytes(B, n, dm, h, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib.attn_out_projection_bwd(_vptr(o), _vptr(w_o), _vptr(dy), _vptr(d_o), _vptr(dw_o), B, n, dm, h, d,
                                     _vptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_out_projection_bwd")
    return d_o, dw_o


def attn_get_device_status(stream=None) -> int:
    return int(load_library().attn_get_device_status(_stream_handle(stream)))


def attn_set_watchdog_ns(budget_ns: int) -> int:
    return int(load_library().attn_set_watchdog_ns(int(budget_ns)))


def attn_debug_inject(mode: int) -> int:
    return int(load_library().attn_debug_inject(int(mode)))


def attn_profile_enable(on: bool) -> int:
    return int(load_library().attn_profile_enable(int(bool(on))))


def attn_profile_read(kind) -> Tuple[int, float]:
    """(launches, total device ms) of one kernel kind since the last read; clears them."""
    k = KERNEL_KINDS[kind] if isinstance(kind, str) else int(kind)
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    st = load_library().attn_profile_read(k, ctypes.byref(n), ctypes.byref(ms))
    if st != ATTN_OK:
        raise AttnError(st, "attn_profile_read")
    return int(n.value), float(ms.value)


def attn_bwd_noalloc(q, k, v, o, lse, dO, causal: bool = False, scale: Optional[float] = None,
                     dq=None, dk=None, dv=None, stream=None):
    """attn_bwd whose scratch lives in the library's fixed device array (no workspace).

    For callers that cannot allocate device memory at the call site; see
    include/attn.h for the size limit and the one-call-at-a-time rule.
    """
    import torch
    lib = load_library()
    B, h, n, d_k = q.shape
    m, d_v = k.shape[2], v.shape[3]
    _check_tensor("q", q, dtype=torch.bfloat16)
    _check_tensor("k", k, (B, h, m, d_k), torch.bfloat16)
    _check_tensor("v", v, (B, h, m, d_v), torch.bfloat16)
    _check_tensor("o", o, (B, h, n, d_v), torch.bfloat16)
    _check_tensor("lse", lse, (B, h, n), torch.float32)
    _check_tensor("dO", dO, (B, h, n, d_v), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _check_tensor(name, t, tuple(ref.shape), torch.bfloat16)
    st = lib.attn_bwd_noalloc(_vptr(q), _vptr(k), _vptr(v), _vptr(o), _fptr(lse), _vptr(dO),
                              _vptr(dq), _vptr(dk), _vptr(dv), B, h, n, m, d_k, d_v,
                              int(bool(causal)), float(scale), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_noalloc")
    return dq, dk, dv
