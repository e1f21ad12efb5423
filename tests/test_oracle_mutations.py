"""The pins must catch plausible oracle mistakes.

Each case compiles a copy of the oracle's C source with one planted mistake
(CPU only), swaps it in for the real library, and checks that at least one
pin of test_oracle_pins fails.
"""
import ctypes
import os
import subprocess

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
