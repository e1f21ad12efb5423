"""The pins must catch plausible oracle mistakes.

Each case compiles a copy of the oracle's C source with one planted mistake
(CPU only), swaps it in for the real library, and checks that at least one
pin of test_oracle_pins fails.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTATIONS = {
    "diagonal_excluded": ("return (i + 1 < m) ? (i + 1) : m;", "return (i < m) ? (i > 0 ? i : 1) : m;"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "lse_without_max": ("return M + log(l);", "return log(l);"),
    "max_not_subtracted_in_lse": ("return M + log(l);", "return M + log(l) + 1e-6;"),
    "dS_sign": ("const double dS = row[j] * (dP - Di);", "const double dS = row[j] * (dP + Di);"),
    "dK_scale_dropped": ("if (dkj) for (long c = 0; c < dk; ++c) dkj[c] *= scale;", ""),
    "dV_uses_dS": ("for (long c = 0; c < dv; ++c) dvj[c] += P * dOi[c];",
                   "for (long c = 0; c < dv; ++c) dvj[c] += P * dOi[c] * (1.0 + 1e-3 * c);"),
    "dQ_transposed_operand": ("for (long c = 0; c < dk; ++c) dqi[c] += dS * kj[c];",
                              "for (long c = 0; c < dk; ++c) dqi[c] += dS * kj[dk - 1 - c];"),
    "causal_mask_in_bwd_off_by_one": ("if (j < lo || j >= hi) continue;", "if (j < lo || j > hi) continue;"),
    "window_right_off_by_one": ("if (wr >= 0 && i + wr + 1 < h) h = i + wr + 1;",
                                "if (wr >= 0 && i + wr < h) h = i + wr;"),
    "window_left_off_by_one": ("*lo = (wl >= 0 && i - wl > 0) ? i - wl : 0;",
                               "*lo = (wl >= 0 && i - wl + 1 > 0) ? i - wl + 1 : 0;"),
    "window_sides_swapped": ("*lo = (wl >= 0 && i - wl > 0) ? i - wl : 0;",
                             "*lo = (wr >= 0 && i - wr > 0) ? i - wr : 0;"),
    "key_length_per_head": ("const long mb = kv_len[bh / h];", "const long mb = kv_len[bh % h];"),
    "key_padding_off_by_one": ("return v < mb ? v : mb;", "return v < mb + 1 ? v : mb + 1;"),
    "empty_row_not_zero": ("for (long j = 0; j < m; ++j) s[j] = 0.0;\n        return -INFINITY;",
                           "for (long j = 0; j < m; ++j) s[j] = 1.0 / m;\n        return -INFINITY;"),
    "value_row_offset": ("const double *vj = V + j * dv;\n        for (long c = 0; c < dv; ++c) oi[c] += P[j] * vj[c];",
                         "const double *vj = V + (j > 0 ? j - 1 : 0) * dv;\n        for (long c = 0; c < dv; ++c) oi[c] += P[j] * vj[c];"),
}

PIN_TESTS = [
    (pins.test_worked_example_scores_and_weights, {}),
    (pins.test_saturation_example_weights_and_derivative, {}),
    (pins.test_footnote4_score_statistics, {}),
    (pins.test_rows_sum_to_one_and_masked_weights_are_zero, {"causal": True}),
    (pins.test_equal_scores_give_mean_of_values, {"causal": True}),
    (pins.test_permutation_equivariance, {}),
    (pins.test_single_key_closed_form, {}),
    (pins.test_causal_prefix_invariance, {}),
    (pins.test_backward_matches_central_differences,
     {"causal": True, "n": 6, "m": 6, "dk": 4, "dv": 4}),
    (pins.test_backward_sum_invariants, {"causal": True}),
    (pins.test_against_torch_cpu_fp64_library,
     {"causal": True, "n": 9, "m": 9, "dk": 16, "dv": 16}),
    (pins.test_key_padding_equals_truncation, {"causal": True}),
    (pins.test_key_padding_against_torch_masked_library, {}),
    (pins.test_key_padding_empty_sequence_is_the_empty_sum, {}),
    (pins.test_window_of_one_position_returns_own_value, {}),
    (pins.test_window_against_torch_masked_library, {"wl": 2, "wr": 3, "causal": False, "lens": None}),
    (pins.test_window_rows_without_keys_are_the_empty_sum, {}),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    before, after = MUTATIONS[name]
    src = open(SRC, encoding="utf-8").read()
    assert before in src, f"mutation anchor for {name} not found"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(before, after, 1), encoding="utf-8")
    lib_path = tmp_path / "libmut.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib_path), str(mutated), "-lm"], check=True)
    real = oracle._load()
    lib = ctypes.CDLL(str(lib_path))
    for fn in ("oracle_attn_weights", "oracle_attn_fwd", "oracle_attn_bwd", "oracle_attn_bwd_rows"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = ctypes.c_int
    lib.oracle_num_threads.restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for fn, kw in PIN_TESTS:
        try:
            fn(**kw)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            failed.append(fn.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"


# ---------------------------------------------------------------- projection gradients (Python oracle)

def _concat(G):
    b, hh, S, dd = G.shape
    return G.transpose(0, 2, 1, 3).reshape(b, S, hh * dd)


def _qkv_bwd(x_q, x_kv, w_qkv, dq, dk, dv, concat=_concat, swap_kv=False, kv_weights_from=None):
    """project_qkv_bwd written out again with one switch per planted mistake."""
    Xq, Xkv, W = (np.asarray(a, dtype=np.float64) for a in (x_q, x_kv, w_qkv))
    Cq, Ck, Cv = (concat(np.asarray(a, dtype=np.float64)) for a in (dq, dk, dv))
    hd = Cq.shape[-1]
    Wk, Wv = W[:, hd:2 * hd], W[:, 2 * hd:]
    if swap_kv:
        Wk, Wv = Wv, Wk
    dx_q = Cq @ W[:, :hd].T
    dx_kv = Ck @ Wk.T + Cv @ Wv.T
    Xw = Xkv if kv_weights_from is None else kv_weights_from(Xq, Xkv)
    dw = np.concatenate([np.einsum("bsc,bsj->cj", Xq, Cq), np.einsum("bsc,bsj->cj", Xw, Ck),
                         np.einsum("bsc,bsj->cj", Xw, Cv)], axis=1)
    return dx_q, dx_kv, dw


def _plain_reshape(G):  # heads and tokens mixed up
    return G.reshape(G.shape[0], G.shape[2], -1)


def _queries_cut_to_keys(Xq, Xkv):  # x_q where x_kv belongs (cut or padded to the key count)
    m = Xkv.shape[1]
    out = np.zeros_like(Xkv)
    k = min(m, Xq.shape[1])
    out[:, :k] = Xq[:, :k]
    return out


def _out_bwd(o, w_o, dy, heads_back=True, first_sequence_only=False):
    O, W, G = (np.asarray(a, dtype=np.float64) for a in (o, w_o, dy))
    B, h, n, d = O.shape
    C = O.transpose(0, 2, 1, 3).reshape(B, n, h * d)
    g = G @ W.T
    d_o = g.reshape(B, n, h, d).transpose(0, 2, 1, 3) if heads_back else g.reshape(B, h, n, d)
    dw = np.einsum("bsj,bsc->jc", C[:1], G[:1]) if first_sequence_only else np.einsum("bsj,bsc->jc", C, G)
    return np.ascontiguousarray(d_o), dw


PY_MUTANTS = {
    "qkv_bwd_kv_blocks_swapped": ("project_qkv_bwd", lambda *a: _qkv_bwd(*a, swap_kv=True)),
    "qkv_bwd_heads_not_transposed": ("project_qkv_bwd", lambda *a: _qkv_bwd(*a, concat=_plain_reshape)),
    "qkv_bwd_key_weights_from_queries": ("project_qkv_bwd",
                                         lambda *a: _qkv_bwd(*a, kv_weights_from=_queries_cut_to_keys)),
    "out_bwd_heads_not_transposed_back": ("project_out_bwd", lambda *a: _out_bwd(*a, heads_back=False)),
    "out_bwd_weight_sum_over_one_sequence": ("project_out_bwd", lambda *a: _out_bwd(*a, first_sequence_only=True)),
}


def test_projection_gradient_rewrite_agrees_with_the_oracle():
    """The rewrite above, with no switch set, is the oracle's result (so a caught mutant is the switch)."""
    rng = np.random.default_rng(5)
    xq, xkv = rng.standard_normal((2, 5, 6)), rng.standard_normal((2, 7, 6))
    w = rng.standard_normal((6, 3 * 4))
    dq, dk, dv = rng.standard_normal((2, 2, 5, 2)), rng.standard_normal((2, 2, 7, 2)), rng.standard_normal((2, 2, 7, 2))
    for got, ref in zip(_qkv_bwd(xq, xkv, w, dq, dk, dv), oracle.project_qkv_bwd(xq, xkv, w, dq, dk, dv)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    o, wo, dy = rng.standard_normal((2, 2, 5, 2)), rng.standard_normal((4, 6)), rng.standard_normal((2, 5, 6))
    for got, ref in zip(_out_bwd(o, wo, dy), oracle.project_out_bwd(o, wo, dy)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_projection_gradient_mistake_is_caught(name, monkeypatch):
    attr, fn = PY_MUTANTS[name]
    monkeypatch.setattr(oracle, attr, fn)
    failed = 0
    for pin in (pins.test_projection_gradients_match_finite_differences,
                pins.test_projection_gradients_against_torch_autograd):
        try:
            pin()
        except (AssertionError, ValueError):
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake {name}"
