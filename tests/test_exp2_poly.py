"""The forward kernel's FMA-pipe exponential 2^x (range reduction + degree-3 polynomial).

CPU: an fp32 emulation of the same arithmetic (numpy rounds every fp32
operation to nearest) bounds the relative error by 2^-13 against exact 2^x,
which pins the coefficients. GPU: the kernel's own function against fp64 2^x
and against the hardware ex2.approx over the working range.
"""
import numpy as np
import pytest
import torch

C = np.array([1.0, 6.932829022e-01, 2.422109544e-01, 5.500893667e-02], dtype=np.float32)
BOUND = 2.0 ** -13


def poly_exp2_f32(x):
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    sh = np.float32(12582912.0)
    t = (x + sh).astype(np.float32)
    f = (x - (t - sh).astype(np.float32)).astype(np.float32)
    # fma emulated in fp64 then rounded once: a*b is exact in fp64 for fp32 operands
    p = (f.astype(np.float64) * C[3] + C[2]).astype(np.float32)
    p = (f.astype(np.float64) * p + C[1]).astype(np.float32)
    p = (f.astype(np.float64) * p + C[0]).astype(np.float32)
    n = (t.view(np.uint32).astype(np.int64) - np.float32(sh).view(np.uint32).astype(np.int64))
    bits = (p.view(np.uint32).astype(np.int64) + (n << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_polynomial_error_bound_cpu():
    x = np.concatenate([np.linspace(-125.0, 9.0, 400001, dtype=np.float32),
                        np.linspace(-1.0, 1.0, 100001, dtype=np.float32)])
    y = poly_exp2_f32(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() <= BOUND, rel.max()


def test_polynomial_is_exact_at_zero():
    assert poly_exp2_f32(np.array([0.0], dtype=np.float32))[0] == 1.0
    assert np.all(poly_exp2_f32(np.arange(-100, 9, dtype=np.float32)) == np.exp2(np.arange(-100, 9)))


def test_polynomial_clamps_far_below():
    y = poly_exp2_f32(np.array([-126.0, -200.0, -1e30], dtype=np.float32))
    assert np.all(y >= 0) and np.all(y <= 2.0 ** -125) and np.all(np.isfinite(y))


@pytest.mark.gpu
def test_polynomial_on_gpu_matches_exp2_and_mufu():
    import transformer_scaled_dot_attn_gb300 as A
    x = torch.cat([torch.linspace(-125.0, 9.0, 400001), torch.linspace(-1.0, 1.0, 100001),
                   torch.tensor([-126.0, -200.0, -1e30])]).float().cuda()
    yp, ym = A.attn_debug_exp2(x)
    xe = x.double()
    exact = torch.exp2(xe)
    body = xe >= -125
    rel_p = ((yp.double() - exact).abs() / exact)[body].max().item()
    rel_m = ((ym.double() - exact).abs() / exact)[body & (xe >= -120)].max().item()
    assert rel_p <= BOUND, rel_p
    assert rel_m <= 2.0 ** -20, rel_m  # the hardware path, for comparison
    # same values as the CPU emulation of the same fp32 arithmetic (to within one
    # fp32 rounding: the emulated fma rounds through fp64 first)
    emu = poly_exp2_f32(x.cpu().numpy()).astype(np.float64)
    got = yp.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - emu) <= 2.0 ** -23 * np.abs(emu) + 1e-44)
    tail = yp[~body]
    assert torch.all(tail >= 0) and torch.all(tail <= 2.0 ** -125)
