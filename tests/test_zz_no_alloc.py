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

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import Workload, workload_inputs
from tests.parity_utils import assert_close

FAKE = 0x10000  # never dereferenced: the calls below are refused before any launch
LIMIT = 32 << 20  # bytes of the library's fixed scratch array


def _call(lib, q, B, h, n, d, causal=0):
    vp = ctypes.c_void_p
    lse = ctypes.cast(vp(FAKE), ctypes.POINTER(ctypes.c_float))
    return lib.attn_bwd_noalloc(vp(q), vp(FAKE), vp(FAKE), vp(FAKE), lse, vp(FAKE), vp(FAKE),
                                vp(FAKE), vp(FAKE), B, h, n, n, d, d, causal, 0.088, None)


def test_refuses_sizes_beyond_the_fixed_scratch():
    lib = A.load_library()
    # 16 heads x 8192 padded rows x (128 + 2) fp32 = 68 MB > 32 MiB: refused by the size
    # check, which comes before every pointer check
    assert A.attn_bwd_workspace_bytes(1, 16, 8192, 8192, 128, 128, 0) > LIMIT
    assert _call(lib, FAKE + 8, 1, 16, 8192, 128) == A.ATTN_ERR_UNSUPPORTED
    # 15 heads x 4096 rows x 130 fp32 = 31.9 MB, just under the limit: it passes the size
    # check and is refused only for the misaligned query pointer
    assert A.attn_bwd_workspace_bytes(1, 15, 4096, 4096, 128, 128, 0) <= LIMIT
    assert _call(lib, FAKE + 8, 1, 15, 4096, 128) == A.ATTN_ERR_INVALID_ARG


def _check_against_oracle(w, got, q, k, v, do):
    rq, rk, rv, _, _ = oracle.bwd(q, k, v, do, w.causal, w.default_scale)
    ex = "few_term_cancellation" if w.causal else None  # the documented exception of causal gradients
    for name, g, r in zip(("dQ", "dK", "dV"), got, (rq, rk, rv)):
        assert_close(f"{w.name} {name} vs oracle", g, r, allow=ex)


@pytest.mark.gpu
def test_matches_the_workspace_backward_and_the_oracle_on_calls_in_a_row():
    # every case needs scratch (n > 256 or d = 128 runs the three-launch backward);
    # the second and third calls find the previous call's accumulator and statistics
    # in the array, the third with the first one's shape but other inputs
    cases = [Workload("na", 1, 3, 300, 300, 64, 64, False, 81),
             Workload("nb", 1, 2, 200, 260, 128, 128, True, 82),
             Workload("nc", 1, 3, 300, 300, 64, 64, False, 83)]
    for w in cases:
        assert A.attn_bwd_workspace_bytes(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal) > 0
        q, k, v, do = workload_inputs(w, with_grad=True)
        qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
        o, lse = A.attn_fwd(qd, kd, vd, causal=w.causal)
        ref = A.attn_bwd(qd, kd, vd, o, lse, dod, causal=w.causal)
        got = A.attn_bwd_noalloc(qd, kd, vd, o, lse, dod, causal=w.causal)
        assert A.attn_get_device_status() == A.ATTN_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.isfinite(g).all()
            assert_close(f"{w.name} {name} vs attn_bwd", g, r)
        _check_against_oracle(w, got, q, k, v, do)


@pytest.mark.gpu
def test_largest_accepted_size_runs():
    # scratch of 31.9 MB, just under the 32 MiB array: accepted and equal to attn_bwd
    w = Workload("nmax", 1, 15, 4096, 4096, 128, 128, False, 84)
    assert A.attn_bwd_workspace_bytes(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal) <= LIMIT
    g = torch.Generator(device="cuda").manual_seed(84)
    q, k, v, do = (torch.randn(1, 15, 4096, 128, device="cuda", generator=g).bfloat16() for _ in range(4))
    o, lse = A.attn_fwd(q, k, v)
    ref = A.attn_bwd(q, k, v, o, lse, do)
    got = A.attn_bwd_noalloc(q, k, v, o, lse, do)
    assert A.attn_get_device_status() == A.ATTN_OK
    for name, gg, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_close(f"{w.name} {name} vs attn_bwd", gg, r)
