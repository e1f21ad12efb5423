"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory
at the call site (a pooled allocator owns the device memory, or cudaMalloc's
implicit synchronisation is not allowed in the calling loop). Its scratch is a
fixed array inside the library, so it must give what attn_bwd gives with a
caller-provided workspace, call after call, even though every call reuses the
same array and finds the previous call's data in it.

This file is collected last on purpose; it must also pass alone in a fresh process.
"""
import ctypes

import pytest
import torch

import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import Workload, workload_inputs
from tests.parity_utils import assert_close

FAKE = 0x10000  # never dereferenced: the call below is refused before any launch


def test_refuses_sizes_beyond_the_fixed_scratch():
    lib = A.load_library()
    vp = ctypes.c_void_p
    lse = ctypes.cast(vp(FAKE), ctypes.POINTER(ctypes.c_float))
    # 16 heads x 8192 padded rows x (128 + 2) fp32 = 68 MB > 32 MiB
    st = lib.attn_bwd_noalloc(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), lse, vp(FAKE), vp(FAKE),
                              vp(FAKE), vp(FAKE), 1, 16, 8192, 8192, 128, 128, 0, 0.088, None)
    assert st == A.ATTN_ERR_UNSUPPORTED
    # within the limit it gets past the size check (and fails on the fake pointers' alignment)
    st = lib.attn_bwd_noalloc(vp(FAKE + 8), vp(FAKE), vp(FAKE), vp(FAKE), lse, vp(FAKE), vp(FAKE),
                              vp(FAKE), vp(FAKE), 1, 2, 256, 256, 64, 64, 0, 0.125, None)
    assert st == A.ATTN_ERR_INVALID_ARG


@pytest.mark.gpu
def test_matches_the_workspace_backward_on_two_calls_in_a_row():
    cases = [Workload("na", 2, 4, 256, 320, 64, 64, False, 81),
             Workload("nb", 1, 3, 200, 200, 128, 128, True, 82)]
    for w in cases:  # two calls in a row, different sizes: the second finds the first's data
        q, k, v, do = (t.cuda() for t in workload_inputs(w, with_grad=True))
        o, lse = A.attn_fwd(q, k, v, causal=w.causal)
        ref = A.attn_bwd(q, k, v, o, lse, do, causal=w.causal)
        got = A.attn_bwd_noalloc(q, k, v, o, lse, do, causal=w.causal)
        assert A.attn_get_device_status() == A.ATTN_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.isfinite(g).all()
            assert_close(f"{w.name} {name}", g, r, grad=True)
