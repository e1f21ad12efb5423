"""The C-ABI library builds for sm_103a, loads, exports what include/attn.h declares,
and rejects bad arguments on the host (no GPU needed: no call here reaches CUDA)."""
import ctypes
import os
import re

import pytest

import transformer_scaled_dot_attn_gb300 as A
from transformer_scaled_dot_attn_gb300 import native_build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return A.load_library()


def _declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    assert _declared_functions() == sorted(A.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    # and the exported names really are C symbols (no C++ mangling)
    out = os.popen(f"nm -D --defined-only {A.library_path()}").read()
    for name in _declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_status_strings(lib):
    assert A.attn_status_string(0) == "ATTN_OK"
    assert A.attn_status_string(4) == "ATTN_ERR_TIMEOUT"
    assert A.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(lib, B_=1, h=1, n=8, m=8, dk=64, dv=64, causal=0, scale=0.125, ptrs=(FAKE,) * 4, lse=None):
    vp = [ctypes.c_void_p(p) if p else None for p in ptrs]
    return lib.attn_fwd(vp[0], vp[1], vp[2], vp[3], lse, B_, h, n, m, dk, dv, causal, scale, None)


def test_fwd_argument_checks(lib):
    assert _fwd(lib, B_=-1) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, n=-1) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, m=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, dk=48, dv=48) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, dk=64, dv=32) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, dk=256, dv=256) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, n=256 * 65536) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, ptrs=(FAKE, 0, FAKE, FAKE)) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, ptrs=(FAKE + 8, FAKE, FAKE, FAKE)) == A.ATTN_ERR_INVALID_ARG
    bad_lse = ctypes.cast(ctypes.c_void_p(FAKE + 2), ctypes.POINTER(ctypes.c_float))
    assert _fwd(lib, lse=bad_lse) == A.ATTN_ERR_INVALID_ARG
    # empty batches are a no-op, even with null pointers
    assert _fwd(lib, B_=0, ptrs=(0, 0, 0, 0)) == A.ATTN_OK
    assert _fwd(lib, n=0, ptrs=(0, 0, 0, 0)) == A.ATTN_OK


def test_bwd_argument_checks(lib):
    vp = ctypes.c_void_p
    f = ctypes.cast(vp(FAKE), ctypes.POINTER(ctypes.c_float))

    # n = 300: the general path, which needs a workspace (n <= 256 with d <= 64 needs none)
    def call(n=300, m=8, d=64, ws_bytes=1 << 30, ws=FAKE, dq=FAKE, lse=f, scale=0.125):
        return lib.attn_bwd(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), lse, vp(FAKE), vp(dq) if dq else None,
                            vp(FAKE), vp(FAKE), 1, 1, n, m, d, d, 0, scale, vp(ws) if ws else None,
                            ws_bytes, None)

    assert call(m=0) == A.ATTN_ERR_INVALID_ARG
    assert call(d=96) == A.ATTN_ERR_UNSUPPORTED
    assert call(ws=0) == A.ATTN_ERR_INVALID_ARG
    assert call(dq=0) == A.ATTN_ERR_INVALID_ARG
    assert call(lse=None) == A.ATTN_ERR_INVALID_ARG
    assert call(ws_bytes=16) == A.ATTN_ERR_INVALID_ARG
    assert call(scale=float("nan")) == A.ATTN_ERR_INVALID_ARG


def test_workspace_size(lib):
    # general path: fp32 dQ accumulator + two fp32 per-row statistics, rows padded to 128
    assert A.attn_bwd_workspace_bytes(2, 3, 300, 77, 64, 64) == 2 * 3 * 384 * (64 + 2) * 4
    assert A.attn_bwd_workspace_bytes(2, 3, 200, 77, 128, 128) == 2 * 3 * 256 * (128 + 2) * 4
    assert A.attn_bwd_workspace_bytes(1, 1, 257, 1, 32, 32, True) == 384 * 34 * 4
    # whole-head kernel (n <= 256, d <= 64): no workspace at all
    assert A.attn_bwd_workspace_bytes(2, 3, 200, 77, 64, 64) == 0
    assert A.attn_bwd_workspace_bytes(1, 1, 256, 1, 32, 32, True) == 0
    assert A.attn_bwd_workspace_bytes(0, 3, 200, 77, 64, 64) == 0
    assert A.attn_bwd_workspace_bytes(1, 1, 0, 77, 64, 64) == 0


@pytest.mark.parametrize("n,d,causal", [(300, 64, False), (16384, 128, False), (1000, 32, True), (257, 128, True)])
def test_workspace_is_per_head_scratch(lib, n, d, causal):
    # attn_fwd_bwd_host gives each head chunk the workspace part of its own heads
    # (offset: the bytes of the heads before it), so the size must be the heads
    # times one head's bytes, and one head's bytes a multiple of 16 (TMA alignment)
    one = A.attn_bwd_workspace_bytes(1, 1, n, n, d, d, causal)
    assert one > 0 and one % 16 == 0
    for B, h in ((1, 7), (4, 16), (3, 5)):
        assert A.attn_bwd_workspace_bytes(B, h, n, n, d, d, causal) == B * h * one
        for h0 in range(B * h):
            assert A.attn_bwd_workspace_bytes(h0, 1, n, n, d, d, causal) == h0 * one


def test_debug_hooks(lib):
    assert A.attn_debug_inject(2) == A.ATTN_ERR_INVALID_ARG
    assert A.attn_debug_inject(0) == A.ATTN_OK
    assert A.attn_set_watchdog_ns(0) == A.ATTN_OK


def test_built_for_sm103a():
    """The build command targets sm_103a only (one -gencode, arch=compute_103a,code=sm_103a)."""
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        A.attn_fwd(q, q, q)


def test_varlen_argument_checks(lib):
    """The key-padding entry points refuse a misaligned length array before any launch."""
    vp = ctypes.c_void_p
    f = ctypes.cast(vp(FAKE), ctypes.POINTER(ctypes.c_float))
    st = lib.attn_fwd_varlen(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), f, vp(FAKE + 2), 1, 1, 8, 8, 64, 64,
                             0, 0.125, None)
    assert st == A.ATTN_ERR_INVALID_ARG
    st = lib.attn_bwd_varlen(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), f, vp(FAKE), vp(FAKE), vp(FAKE),
                             vp(FAKE), vp(FAKE + 2), 1, 1, 8, 8, 64, 64, 0, 0.125, vp(FAKE), 1 << 30, None)
    assert st == A.ATTN_ERR_INVALID_ARG
    # the same validation as the unpadded calls applies
    st = lib.attn_fwd_varlen(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), f, vp(FAKE), 1, 1, 8, 8, 48, 48, 0,
                             0.125, None)
    assert st == A.ATTN_ERR_UNSUPPORTED


def test_host_step_argument_checks(lib):
    """attn_fwd_bwd_host refuses bad arguments before it enqueues anything."""
    vp = ctypes.c_void_p
    f = ctypes.cast(vp(FAKE), ctypes.POINTER(ctypes.c_float))

    def call(B_=1, h=2, n=8, m=8, d=64, chunks=0, hq=FAKE, dq=FAKE, q=FAKE, ws=None, ws_bytes=0,
             scale=0.125):
        host = [vp(hq) if hq else None, vp(FAKE), vp(FAKE), vp(FAKE), None, None,
                vp(FAKE), vp(FAKE), vp(FAKE)]
        dev = [vp(q) if q else None, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), f,
               vp(dq) if dq else None, vp(FAKE), vp(FAKE)]
        return lib.attn_fwd_bwd_host(*host, *dev, vp(ws) if ws else None, ws_bytes, B_, h, n, m, d, d, 0,
                                     scale, chunks, None)

    assert call(chunks=-1) == A.ATTN_ERR_INVALID_ARG
    assert call(B_=-1) == A.ATTN_ERR_INVALID_ARG
    assert call(m=0) == A.ATTN_ERR_INVALID_ARG
    assert call(scale=float("nan")) == A.ATTN_ERR_INVALID_ARG
    assert call(d=48) == A.ATTN_ERR_UNSUPPORTED
    assert call(hq=0) == A.ATTN_ERR_INVALID_ARG
    assert call(dq=0) == A.ATTN_ERR_INVALID_ARG
    assert call(q=FAKE + 8) == A.ATTN_ERR_INVALID_ARG
    # n = 300 takes the general backward: it needs the whole batch's workspace
    need = A.attn_bwd_workspace_bytes(1, 2, 300, 8, 64, 64, False)
    assert need > 0
    assert call(n=300) == A.ATTN_ERR_INVALID_ARG
    assert call(n=300, ws=FAKE, ws_bytes=need - 16) == A.ATTN_ERR_INVALID_ARG
    # nothing to compute: OK with null pointers everywhere
    assert lib.attn_fwd_bwd_host(*([None] * 18), None, 0, 0, 4, 8, 8, 64, 64, 0, 0.125, 0, None) == A.ATTN_OK


def test_host_step_binding_checks_host_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="float32|bfloat16"):
        A.attn_fwd_bwd_host(x.float(), x, x, x)
    with pytest.raises(ValueError, match="shape"):
        A.attn_fwd_bwd_host(x, x, x, x[:, :, :2])
