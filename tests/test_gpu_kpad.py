"""Key padding (variable-length batches) on the GPU against the fp64 oracle.

Sequence b has kv_len[b] real keys; the keys past them are padding and are
masked ("Attention Is All You Need" §5.1 batches similar-length sentences;
the <pad> positions of Figure 3). The cases cover every kernel that runs:
the persistent and per-item forwards, the whole-head and general backwards,
causal and not, lengths 0, 1, m and ragged ones, d = 32, 64, 128.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import WORKLOADS, Workload, kv_lengths, workload_inputs
from tests.parity_utils import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # (B, h, n, m, d, causal, kv_len)
    (4, 2, 256, 256, 64, False, [256, 0, 129, 1]),      # persistent fwd, whole-head bwd
    (4, 2, 200, 256, 64, True, [256, 7, 0, 128]),       # per-item fwd, whole-head bwd, causal
    (3, 2, 130, 300, 32, False, [300, 64, 0]),          # ragged m, d = 32
    (2, 2, 384, 1024, 64, False, [1000, 513]),          # persistent fwd, general bwd
    (3, 2, 256, 512, 32, False, [0, 300, 512]),         # persistent fwd (later tiles speculative)
    (3, 1, 300, 300, 64, True, [300, 150, 1]),          # general bwd, causal
    (2, 2, 200, 320, 128, False, [320, 0]),             # d = 128: per-item fwd, general bwd
]


def _run(q, k, v, do, causal, scale, lens):
    kvl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = A.attn_fwd(qd, kd, vd, causal=causal, scale=scale, kv_len=kvl)
    dq, dk, dv = A.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, kv_len=kvl)
    assert A.attn_get_device_status() == A.ATTN_OK
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_key_padding_matches_oracle(case):
    B, h, n, m, d, causal, lens = CASES[case]
    w = Workload(f"kpad{case}", B, h, n, m, d, d, causal, 70 + case)
    q, k, v, do = workload_inputs(w, with_grad=True)
    scale = w.default_scale
    o, lse, dq, dk, dv = _run(q, k, v, do, causal, scale, lens)
    ro, rl = oracle.fwd(q, k, v, causal, scale, kv_len=lens)
    rdq, rdk, rdv, _, _ = oracle.bwd(q, k, v, do, causal, scale, kv_len=lens)
    for b, L in enumerate(lens):
        if L == 0:
            # the empty sum, exactly
            assert (o[b] == 0).all() and torch.isneginf(lse[b]).all()
            assert (dq[b] == 0).all() and (dk[b] == 0).all() and (dv[b] == 0).all()
            continue
        assert_close(f"O b{b}", o[b], ro[b])
        assert_close(f"lse b{b}", lse[b], rl[b])
        ex = "few_term_cancellation"  # keys of padded sequences that few queries weight
        for hh in range(h):
            assert_close(f"dQ b{b}h{hh}", dq[b, hh], rdq[b, hh], allow=ex)
            assert_close(f"dK b{b}h{hh}", dk[b, hh], rdk[b, hh], allow=ex)
            assert_close(f"dV b{b}h{hh}", dv[b, hh], rdv[b, hh], allow=ex)
        # padding keys get exactly zero gradient
        assert (dk[b, :, L:] == 0).all() and (dv[b, :, L:] == 0).all()


def test_padded_values_do_not_change_any_result():
    """Bitwise: what sits in the padding keys and values is never read into a result."""
    B, h, n, m, d = 3, 2, 256, 256, 64
    w = Workload("kpad_vals", B, h, n, m, d, d, False, 90)
    q, k, v, do = workload_inputs(w, with_grad=True)
    lens = [100, 256, 17]
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate(lens):
        k2[b, :, L:] = 1000.0
        v2[b, :, L:] = -3.0
    for causal in (False, True):
        a = _run(q, k, v, do, causal, 0.125, lens)
        b_ = _run(q, k2, v2, do, causal, 0.125, lens)
        for x, y in zip(a, b_):
            assert torch.equal(x, y)


def test_full_length_equals_no_padding():
    """kv_len = m everywhere gives bit-identical results to the unpadded call."""
    w = WORKLOADS["encoder"]
    B = 8
    q, k, v, do = (t[:B].contiguous().to(DEV) for t in workload_inputs(w, with_grad=True))
    kvl = torch.full((B,), w.m, dtype=torch.int32, device=DEV)
    o1, l1 = A.attn_fwd(q, k, v)
    o2, l2 = A.attn_fwd(q, k, v, kv_len=kvl)
    g1 = A.attn_bwd(q, k, v, o1, l1, do)
    g2 = A.attn_bwd(q, k, v, o2, l2, do, kv_len=kvl)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for x, y in zip(g1, g2):
        assert torch.equal(x, y)


def test_full_size_padded_encoder_sampled():
    """The benchmark's variable-length workload at full size, sampled heads and rows."""
    w = WORKLOADS["encoder_kpad"]
    lens = kv_lengths(w)
    q, k, v, do = workload_inputs(w, with_grad=True)
    o, lse, dq, dk, dv = _run(q, k, v, do, w.causal, w.default_scale, lens)
    rng = np.random.default_rng(11)
    for b in sorted(set([0, w.B - 1] + rng.choice(w.B, 4, replace=False).tolist())):
        L = lens[b]
        hh = int(rng.integers(w.h))
        rows = sorted(set([0, 1, 127, 128, w.n - 1] + rng.choice(w.n, 24, replace=False).tolist()))
        krows = sorted(set([0, L - 1, min(L, w.m - 1)] + rng.choice(w.m, 12, replace=False).tolist()))
        ro, rl = oracle.fwd(q[b, hh], k[b, hh], v[b, hh], False, w.default_scale, rows=rows, kv_len=[L])
        assert_close(f"O b{b}", o[b, hh, rows], ro[rows])
        assert_close(f"lse b{b}", lse[b, hh, rows][None], rl[rows][None])
        rdq, rdk, rdv = oracle.bwd_rows(q[b, hh], k[b, hh], v[b, hh], do[b, hh], False, w.default_scale,
                                       rows, krows, kv_len=L)
        ex = "few_term_cancellation"
        assert_close(f"dQ b{b}", dq[b, hh, rows], rdq, allow=ex)
        assert_close(f"dK b{b}", dk[b, hh, krows], rdk, allow=ex)
        assert_close(f"dV b{b}", dv[b, hh, krows], rdv, allow=ex)


def test_long_causal_padded_forward_sampled_rows():
    """Causal forward with key padding at 8192 query rows, where the persistent
    kernel takes causal work (longest query blocks first, speculative exponentials
    from the third key tile): sampled rows of every sequence against the oracle,
    including rows past a sequence's last real key and the tile edges."""
    B, h, n, d = 3, 2, 8192, 64
    lens = [8192, 5000, 129]
    w = Workload("kpad_long_causal", B, h, n, n, d, d, True, 79)
    q, k, v = workload_inputs(w)
    kvl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = A.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, kv_len=kvl)
    assert A.attn_get_device_status() == A.ATTN_OK
    o, lse = o.cpu(), lse.cpu()
    rng = np.random.default_rng(79)
    rows = sorted({0, 1, 127, 128, 129, 255, 256, 4999, 5000, 5001, n - 129, n - 128, n - 1}
                  | set(rng.choice(n, size=40, replace=False).tolist()))
    ro, rl = oracle.fwd(q, k, v, True, w.default_scale, rows=rows, kv_len=lens)
    for b in range(B):
        assert_close(f"O b{b}", o[b][:, rows], ro[b][:, rows])
        assert_close(f"lse b{b}", lse[b][:, rows][..., None], rl[b][:, rows][..., None])
