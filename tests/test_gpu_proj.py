"""Multi-head projections (§3.2.2) on the GPU against the fp64 oracle.

Q = x_q W^Q, K = x_kv W^K, V = x_kv W^V written into the [B, h, S, d] layout,
and y = Concat(heads) W^O read from it. Each GEMM is checked on the same bf16
inputs as the oracle (fp32 accumulation, one bf16 rounding of the result);
the chained sublayer is checked stage by stage on the GPU's own bf16
intermediates, and end to end with a relative-L2 bound that admits the bf16
roundings of Q, K, V and O between the stages.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import normal_bf16
from tests.parity_utils import assert_close, errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(rows, cols, seed):
    # N(0, 1/rows) so that the projections stay O(1), rounded to bf16
    return normal_bf16((rows, cols), seed, mult=1.0 / np.sqrt(rows))


QKV_CASES = [
    # (B, n, m, d_model, h, d, self-attention)
    (2, 256, 256, 512, 8, 64, True),      # base model, one fused GEMM
    (2, 200, 320, 512, 8, 64, False),     # cross-attention, ragged sequences
    (3, 130, 130, 512, 4, 128, True),     # d = 128
    (1, 77, 300, 1024, 16, 64, False),    # big model width, one short query sequence
]


@pytest.mark.parametrize("case", range(len(QKV_CASES)))
def test_qkv_projection_matches_oracle(case):
    B, n, m, dm, h, d, self_attn = QKV_CASES[case]
    xq = normal_bf16((B, n, dm), 3100 + case)
    xkv = xq if self_attn else normal_bf16((B, m, dm), 3200 + case)
    w = _weights(dm, 3 * h * d, 3300 + case)
    xq_d = xq.to(DEV)
    xkv_d = xq_d if self_attn else xkv.to(DEV)
    q, k, v = A.attn_qkv_projection(xq_d, xkv_d, w.to(DEV), h, d)
    assert A.attn_get_device_status() == A.ATTN_OK
    rq, rk, rv = oracle.project_qkv(xq, xkv, w, h, d)
    assert_close("Q", q.cpu(), rq)
    assert_close("K", k.cpu(), rk)
    assert_close("V", v.cpu(), rv)


OUT_CASES = [
    # (B, n, h, d, d_model)
    (2, 256, 8, 64, 512),
    (3, 200, 4, 128, 512),
    (2, 130, 8, 64, 576),     # a last column tile of 64
    (1, 300, 16, 64, 1024),
]


@pytest.mark.parametrize("case", range(len(OUT_CASES)))
def test_out_projection_matches_oracle(case):
    B, n, h, d, dm = OUT_CASES[case]
    o = normal_bf16((B, h, n, d), 3400 + case)
    w = _weights(h * d, dm, 3500 + case)
    y = A.attn_out_projection(o.to(DEV), w.to(DEV))
    assert A.attn_get_device_status() == A.ATTN_OK
    assert_close("Y", y.cpu(), oracle.project_out(o, w))


@pytest.mark.parametrize("causal", [False, True])
def test_multi_head_sublayer_chain(causal):
    """x -> Q, K, V -> attention -> Concat W^O, all on the GPU."""
    B, n, dm, h, d = 2, 256, 512, 8, 64
    x = normal_bf16((B, n, dm), 3600)
    w = _weights(dm, 3 * h * d, 3601)
    wo = _weights(h * d, dm, 3602)
    xd = x.to(DEV)
    q, k, v = A.attn_qkv_projection(xd, xd, w.to(DEV), h, d)
    o, _ = A.attn_fwd(q, k, v, causal=causal)
    y = A.attn_out_projection(o, wo.to(DEV))
    assert A.attn_get_device_status() == A.ATTN_OK
    # stage by stage on the GPU's own bf16 intermediates
    ro, _ = oracle.fwd(q.cpu(), k.cpu(), v.cpu(), causal, 1 / np.sqrt(d))
    assert_close("O", o.cpu(), ro)
    assert_close("Y", y.cpu(), oracle.project_out(o.cpu(), wo))
    # end to end: Q, K, V and O each pass through one bf16 rounding (2^-9
    # relative) that the fp64 oracle does not make
    _, rel = errors(y.cpu(), oracle.multi_head(x, x, w, wo, h, d, causal=causal))
    assert rel <= 1e-2, rel


def test_projection_argument_checks():
    x = torch.zeros(1, 8, 512, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(512, 3 * 8 * 32, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(A.AttnError):
        A.attn_qkv_projection(x, x, w, 8, 32)  # d = 32: unsupported
    o = torch.zeros(1, 8, 8, 64, dtype=torch.bfloat16, device=DEV)
    wo = torch.zeros(512, 100, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(A.AttnError):
        A.attn_out_projection(o, wo)  # d_model = 100: not a multiple of 64


# ---------------------------------------------------------------- backward (dx = dy W^T, dW = x^T dy)

QKV_BWD_CASES = [
    # (B, n, m, d_model, h, d, self-attention, one input gradient for self-attention)
    (2, 256, 256, 512, 8, 64, True, True),      # base model: dx and dW one GEMM each
    (2, 256, 256, 512, 8, 64, True, False),     # same inputs, dx_q and dx_kv apart
    (2, 200, 320, 512, 8, 64, False, False),    # cross-attention, ragged sequences
    (3, 130, 130, 512, 4, 128, True, True),     # d = 128
    (1, 77, 300, 1024, 16, 64, False, False),   # big model width
    (2, 64, 0, 256, 2, 64, False, False),       # no keys: dW^K = dW^V = 0
]


@pytest.mark.parametrize("case", range(len(QKV_BWD_CASES)))
def test_qkv_projection_bwd_matches_oracle(case):
    B, n, m, dm, h, d, self_attn, fused = QKV_BWD_CASES[case]
    xq = normal_bf16((B, n, dm), 3700 + case)
    xkv = xq if self_attn else normal_bf16((B, m, dm), 3710 + case)
    w = _weights(dm, 3 * h * d, 3720 + case)
    gq = normal_bf16((B, h, n, d), 3730 + case)
    gk = normal_bf16((B, h, m, d), 3740 + case)
    gv = normal_bf16((B, h, m, d), 3750 + case)
    xq_d = xq.to(DEV)
    xkv_d = xq_d if self_attn else xkv.to(DEV)
    dx_kv = None if fused else torch.empty((B, m, dm), dtype=torch.bfloat16, device=DEV)
    dxq, dxkv, dw = A.attn_qkv_projection_bwd(xq_d, xkv_d, w.to(DEV), gq.to(DEV), gk.to(DEV), gv.to(DEV),
                                              dx_kv=dx_kv)
    assert A.attn_get_device_status() == A.ATTN_OK
    rq, rkv, rw = oracle.project_qkv_bwd(xq, xkv, w, gq, gk, gv)
    if self_attn and fused:
        assert dxkv.data_ptr() == dxq.data_ptr()
        assert_close("dx", dxq.cpu(), rq + rkv)
    else:
        if n > 0:
            assert_close("dx_q", dxq.cpu(), rq)
        if m > 0:
            assert_close("dx_kv", dxkv.cpu(), rkv)
    assert_close("dW_qkv", dw.cpu(), rw)
    if m == 0:
        assert not dw[:, h * d:].any()


OUT_BWD_CASES = [
    # (B, n, h, d, d_model)
    (2, 256, 8, 64, 512),
    (3, 200, 4, 128, 512),
    (2, 130, 8, 64, 576),     # a last column tile of 64 (dO reduction and dW^O columns)
    (1, 300, 16, 64, 1024),
]


@pytest.mark.parametrize("case", range(len(OUT_BWD_CASES)))
def test_out_projection_bwd_matches_oracle(case):
    B, n, h, d, dm = OUT_BWD_CASES[case]
    o = normal_bf16((B, h, n, d), 3800 + case)
    w = _weights(h * d, dm, 3810 + case)
    gy = normal_bf16((B, n, dm), 3820 + case)
    d_o, dw = A.attn_out_projection_bwd(o.to(DEV), w.to(DEV), gy.to(DEV))
    assert A.attn_get_device_status() == A.ATTN_OK
    r_o, r_w = oracle.project_out_bwd(o, w, gy)
    assert_close("dO", d_o.cpu(), r_o)
    assert_close("dW_o", dw.cpu(), r_w)


def test_projection_bwd_is_deterministic():
    """The weight gradients add their token splits in a fixed order: two runs agree bit for bit."""
    B, n, h, d, dm = 4, 256, 8, 64, 512
    o = normal_bf16((B, h, n, d), 3900).to(DEV)
    w = _weights(h * d, dm, 3901).to(DEV)
    gy = normal_bf16((B, n, dm), 3902).to(DEV)
    a = A.attn_out_projection_bwd(o, w, gy)[1].clone()
    b = A.attn_out_projection_bwd(o, w, gy)[1]
    assert torch.equal(a, b)


def test_projection_bwd_rejects_a_short_workspace():
    B, n, h, d, dm = 2, 128, 4, 64, 256
    o = normal_bf16((B, h, n, d), 3910).to(DEV)
    w = _weights(h * d, dm, 3911).to(DEV)
    gy = normal_bf16((B, n, dm), 3912).to(DEV)
    need = A.attn_out_projection_bwd_workspace_bytes(B, n, dm, h, d)
    assert need > 0
    short = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(A.AttnError):
        A.attn_out_projection_bwd(o, w, gy, workspace=short)
