"""attn_fwd_bwd_host: the forward + backward step with inputs and results in host
memory (head chunks whose copies overlap the kernels) gives what attn_fwd +
attn_bwd give on device buffers: the forward bit for bit (every head is computed
alone, whatever the chunk), the gradients within the parity tolerance (the
long-sequence backward adds dQ partial sums in no fixed order)."""
import pytest
import torch

import transformer_scaled_dot_attn_gb300 as A
from seeded_inputs import WORKLOADS, Workload, workload_inputs
from tests.parity_utils import assert_close

pytestmark = pytest.mark.gpu

CASES = [
    Workload("hs_encoder", 4, 4, 256, 256, 64, 64, False, 91),   # whole-head backward, no workspace
    Workload("hs_general", 2, 3, 300, 200, 128, 128, True, 92),  # general backward with workspace
    Workload("hs_d32", 3, 2, 130, 320, 32, 32, False, 93),
]


def _pinned(ts):
    return [t.contiguous().pin_memory() for t in ts]


def _device_path(q, k, v, do, causal):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = A.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = A.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("chunks", [0, 1, 5, 1000])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_step_equals_device_path(w, chunks):
    q, k, v, do = workload_inputs(w, with_grad=True)
    ref = _device_path(q, k, v, do, w.causal)
    got = A.attn_fwd_bwd_host(*_pinned((q, k, v, do)), causal=w.causal, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    assert A.attn_get_device_status() == A.ATTN_OK
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    for name, g, r in zip(("dQ", "dK", "dV"), got[2:], ref[2:]):
        assert torch.isfinite(g).all()
        assert_close(f"{w.name} chunks={chunks} {name}", g, r)


def test_host_step_reuses_buffers_across_calls():
    """Two calls in a row on the same device buffers and the same outputs: the
    second returns the second inputs' results, none of the first's."""
    w = CASES[1]
    buf = A.HostStepBuffers(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal)
    out = None
    for cfg in (94, 95):
        wi = Workload(w.name, w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal, cfg)
        q, k, v, do = workload_inputs(wi, with_grad=True)
        out = A.attn_fwd_bwd_host(*_pinned((q, k, v, do)), causal=w.causal, buffers=buf, chunks=2, out=out)
        torch.cuda.current_stream().synchronize()
        ref = _device_path(q, k, v, do, w.causal)
        assert torch.equal(out[0], ref[0]) and torch.equal(out[1], ref[1])
        for name, g, r in zip(("dQ", "dK", "dV"), out[2:], ref[2:]):
            assert_close(f"cfg {cfg} {name}", g, r)


def test_host_step_without_query_rows():
    """n = 0: no forward rows; dK and dV come back as zeros."""
    B, h, m, d = 2, 3, 40, 64
    k = torch.randn(B, h, m, d, generator=torch.Generator().manual_seed(7)).bfloat16()
    v = torch.randn(B, h, m, d, generator=torch.Generator().manual_seed(8)).bfloat16()
    q = torch.empty(B, h, 0, d, dtype=torch.bfloat16)
    out = (torch.empty(B, h, 0, d, dtype=torch.bfloat16), None, torch.empty(B, h, 0, d, dtype=torch.bfloat16),
           torch.full((B, h, m, d), 3.0, dtype=torch.bfloat16).pin_memory(),
           torch.full((B, h, m, d), 3.0, dtype=torch.bfloat16).pin_memory())
    got = A.attn_fwd_bwd_host(q, k.pin_memory(), v.pin_memory(), q, out=out, chunks=4)
    torch.cuda.current_stream().synchronize()
    assert A.attn_get_device_status() == A.ATTN_OK
    assert (got[3] == 0).all() and (got[4] == 0).all()


def test_host_step_full_encoder_batch_is_bitwise_the_device_path():
    """The benchmark's end-to-end call: the base model's encoder batch (B = 96, h = 8,
    n = m = 256, d = 64) with the library's own split. Every kernel of this size is
    deterministic (the whole-head backward keeps dQ on chip), so all five results
    must be bit-identical to the one-shot calls on device buffers."""
    w = WORKLOADS["encoder"]
    q, k, v, do = workload_inputs(w, with_grad=True)
    ref = _device_path(q, k, v, do, w.causal)
    got = A.attn_fwd_bwd_host(*_pinned((q, k, v, do)), causal=w.causal, chunks=0)
    torch.cuda.current_stream().synchronize()
    assert A.attn_get_device_status() == A.ATTN_OK
    for name, g, r in zip(("O", "lse", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(g, r), name
