"""The pins catch plausible slips: each test plants one mistake in a copy of the
oracle's C source (on the CPU), builds it, and expects some pin to fail."""
import os

import pytest

import oracle
from oracle import build as obuild
import _pins

SRC = open(obuild.SRC).read()

# name -> (text in the oracle source, replacement, occurrence to replace: 0-based)
MUTANTS = {
    "tap_reversed": ("xm(P, t, t - 3 + k, c)", "xm(P, t, t - k, c)", 0),
    "no_zero_history": ("if (j < doc_start(P, t) || j > t) return 0.0;",
                        "if (j < 0 || j > t) return 0.0;", 0),
    "bias_dropped": ("if (P->b) { nsum_add(&acc, P->b[c]); m += fabs(P->b[c]); }", "", 0),
    "silu_grad_sign": ("return s * (1.0 + p * one_minus_s);",
                       "return s * (1.0 - p * one_minus_s);", 0),
    "sigmoid_sign": ("if (p >= 0.0) return 1.0 / (1.0 + exp(-p));",
                     "if (p >= 0.0) return 1.0 / (1.0 + exp(p));", 0),
    "dx_index": ("int64_t j = t + 3 - k;", "int64_t j = t + k;", 0),
    "dx_crosses_documents": ("if (j >= P->S || doc_start(P, j) != s) continue;",
                             "if (j >= P->S) continue;", 0),
    "ties_away": ("nearbyint(a / spacing)", "round(a / spacing)", 0),
    "policy_ignored": ("double p = vcd_oracle_round_bf16(pre);", "double p = pre;", 0),
    "dweight_unmasked": ("d * xm(P, t, t - 3 + k, c)",
                         "d * ((t - 3 + k) >= 0 ? x_at(P, t - 3 + k, c) : 0.0)", 0),
    "dbias_abs": ("nsum_add(&accb, d);", "nsum_add(&accb, fabs(d));", 0),
    "doc_start_strict": ("if ((int64_t)P->cu[mid] <= t) lo = mid; else hi = mid;",
                         "if ((int64_t)P->cu[mid] < t) lo = mid; else hi = mid;", 0),
    "weight_transposed": ("double term = P->w[c * 4 + k]", "double term = P->w[k * 4 + c % 4]", 0),
    "bias_doubled": ("if (P->b) { nsum_add(&acc, P->b[c]);", "if (P->b) { nsum_add(&acc, 2.0 * P->b[c]);", 0),
    "dpre_rounded_to_bf16": ("double d = g * silu_grad(p);",
                             "double d = vcd_oracle_round_bf16(g * silu_grad(p));", 0),
    "no_activation": ("double v = silu(pre);", "double v = pre;", 0),
    "dx_from_dy": ("double d = dpre_at(P, j, c, policy, &a);", "double d = dy_at(P, j, c); a = 0.0;", 0),
    "pre_tap_off_by_one": ("P->w[c * 4 + k] * xm(P, t, t - 3 + k, c)",
                           "P->w[c * 4 + k] * xm(P, t, t - 2 + k, c)", 0),
    "dweight_tap_off_by_one": ("double term = d * xm(P, t, t - 3 + k, c);",
                               "double term = d * xm(P, t, t - 4 + k, c);", 0),
    # allowances made 64 times too generous (each would hide GPU errors) ...
    "allow_pre_x64": ("return 10.0 * U32 * mag;", "return 640.0 * U32 * mag;", 0),
    "allow_fwd_pre_carry_x64": ("*allow = 1.1 * pre_allow(mag)", "*allow = 70.0 * pre_allow(mag)", 0),
    "allow_silu_x64": ("(16.0 + 2.0 * fabs(pre)) * U32 * fabs(v)",
                       "(1024.0 + 128.0 * fabs(pre)) * U32 * fabs(v)", 0),
    "allow_silu_grad_x64": ("double e_grad = (16.0 + 2.0 * fabs(p)) * U32",
                            "double e_grad = (1024.0 + 128.0 * fabs(p)) * U32", 0),
    "allow_dpre_product_x64": ("2.0 * U32 * fabs(d);", "128.0 * U32 * fabs(d);", 0),
    "allow_fp32_policy_dgrad_x64": ("*dgrad = 0.5 * e_pre;", "*dgrad = 32.0 * e_pre;", 0),
    "allow_midpoint_window_x64": ("double lo = vcd_oracle_round_bf16(pre - e_pre);",
                                  "double lo = vcd_oracle_round_bf16(pre - 64.0 * e_pre);", 0),
    "allow_dx_carry_x64": ("e += fabs(wk) * a;", "e += 64.0 * fabs(wk) * a;", 0),
    "allow_dx_sum_x64": ("*allow = e + 8.0 * U32 * mag;", "*allow = e + 512.0 * U32 * mag;", 0),
    # ... and too tight (GPU-correct values would be refused)
    "allow_pre_too_small": ("return 10.0 * U32 * mag;", "return 0.01 * U32 * mag;", 0),
    "allow_midpoint_neighbours_dropped": ("*dgrad = d;", "*dgrad = 0.0;", 0),
    "allow_silu_grad_dropped": ("double e_grad = (16.0 + 2.0 * fabs(p)) * U32",
                                "double e_grad = 0.0 * U32", 0),
}


def _mutate(text, old, new, occurrence):
    parts = text.split(old)
    assert len(parts) > occurrence + 1, f"mutation anchor not found: {old!r}"
    return old.join(parts[:occurrence + 1]) + new + old.join(parts[occurrence + 1:])


def _battery(lib):
    _pins.pin_rounding(lib)
    _pins.pin_silu(lib)
    _pins.pin_golden(lib)
    for seed in range(3):
        for pol in ("bf16", "fp32"):
            _pins.pin_banded(lib, seed, pol)
    for seed in range(2):
        _pins.pin_conv1d(lib, seed)
    _pins.pin_fd(lib, 0)
    _pins.pin_allowances(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new, occ = MUTANTS[name]
    src = tmp_path / f"mut_{name}.c"
    src.write_text(_mutate(SRC, old, new, occ))
    lib_path = obuild.compile_oracle(str(src), str(tmp_path / f"libmut_{name}.so"),
                                    werror=False)
    lib = oracle.load(lib_path)
    with pytest.raises((AssertionError, ValueError)):
        _battery(lib)


def test_unmutated_copy_passes(tmp_path):
    src = tmp_path / "copy.c"
    src.write_text(SRC)
    lib = oracle.load(obuild.compile_oracle(str(src), str(tmp_path / "libcopy.so")))
    _battery(lib)
