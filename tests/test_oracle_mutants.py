"""Planted mistakes in the oracle must be caught by its pins.

Each case copies gemm_oracle.c, applies one plausible mistake (a wrong
index, a transposed operand, a dropped term, a wrong sign or constant, a
wrong rounding), builds it with gcc into a temporary directory, routes the
oracle wrapper through that build and runs the pin tests: at least one pin
must fail.  All of this runs on the CPU.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")

MUTANTS = {
    "reversed_k_index": ("s += a[k] * b[k];", "s += a[k] * b[K - 1 - k];"),
    "transposed_b_operand": ("const double* b = Bd + j * K;", "const double* b = Bd + j;"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];",
                          "for (int64_t k = 0; k + 1 < K; ++k) s += a[k] * b[k];"),
    "gelu_cubic_sign": ("tanh(c * (x + 0.044715 * x * x * x))", "tanh(c * (x - 0.044715 * x * x * x))"),
    "gelu_bf16_constant": ("const double c = 0.7978845608;", "const double c = 0.796875;"),
    "gelu_cubic_coeff": ("0.044715 * x * x * x", "0.04715 * x * x * x"),
    "f16_exponent_bias": ("(int)expo - 25", "(int)expo - 24"),
    "bf16_subnormal_scale": ("ldexp((double)frac, -133)", "ldexp((double)frac, -134)"),
    "round_truncates": ("nearbyint(ldexp(a, -q))", "trunc(ldexp(a, -q))"),
    "round_ties_away": ("nearbyint(ldexp(a, -q))", "round(ldexp(a, -q))"),
    "entries_wrong_row": ("const uint16_t* a = A + rows[t] * K;",
                          "const uint16_t* a = A + cols[t] * K;"),
    "gelu_skipped_in_gemm": ("if (epilogue == 1) return oracle_gelu_tanh(s);",
                             "if (epilogue == 9) return oracle_gelu_tanh(s);"),
    "relu_reflects": ("return x > 0.0 ? x : 0.0;", "return x > 0.0 ? x : -x;"),
    "relu_leaky": ("return x > 0.0 ? x : 0.0;", "return x > 0.0 ? x : 0.01 * x;"),
    "bias_by_row": ("s + bias_of(bias, j, dtype)", "s + bias_of(bias, i, dtype)"),
    "bias_after_epilogue": ("apply_epilogue(s + bias_of(bias, j, dtype), epilogue)",
                            "apply_epilogue(s, epilogue) + bias_of(bias, j, dtype)"),
    "bias_ignored": ("return bias ? oracle_decode(bias[j], dtype) : 0.0;", "return 0.0;"),
    "bias_entries_by_row": ("s + bias_of(bias, cols[t], dtype)", "s + bias_of(bias, rows[t], dtype)"),
    "accumulate_in_float": ("      double s = 0.0;\n      for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];\n      C[i * N + j]",
                            "      float s = 0.0f;\n      for (int64_t k = 0; k < K; ++k) s += (float)(a[k] * b[k]);\n      C[i * N + j]"),
    "overflow_saturates": ("if (v > max_finite) return (uint16_t)(sign | inf_bits);",
                           "if (v > max_finite) return (uint16_t)(sign | (inf_bits - 1u));"),
    "f16_subnormal_scale": ("v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -25);"),
    "nan_rounds_to_inf": ("if (isnan(x)) return (uint16_t)(inf_bits | (1u << (mant_bits - 1)));",
                          "if (isnan(x)) return inf_bits;"),
}

PIN_TESTS = [
    lambda: pins.test_f16_decode_all_patterns_match_numpy(),
    lambda: pins.test_bf16_decode_all_patterns_match_binary32_top_half(),
    lambda: pins.test_f16_round_matches_numpy_rne(),
    lambda: pins.test_bf16_round_is_nearest_even_by_enumeration(),
    lambda: pins.test_rounding_of_nan_and_infinities(),
    lambda: pins.test_rounding_reproduces_printed_gelu_constants(),
    lambda: pins.test_gemm_matches_exact_rational_arithmetic("f16", (7, 5, 3)),
    lambda: pins.test_gemm_bit_exact_on_a_dyadic_grid("bf16"),
    lambda: pins.test_identity_gives_transpose("f16"),
    lambda: pins.test_permutation_gives_column_permutation(),
    lambda: pins.test_all_ones_gives_k(),
    lambda: pins.test_rank_one_closed_form(),
    lambda: pins.test_small_integers_exact_against_integer_matmul(),
    lambda: pins.test_library_cross_check_torch_fp64(),
    lambda: pins.test_entries_equal_full_product(),
    lambda: pins.test_gelu_zero_and_odd_even_identity(),
    lambda: pins.test_gelu_close_to_erf_gelu_with_known_max_error(),
    lambda: pins.test_gemm_gelu_epilogue_applies_after_sum(),
    lambda: pins.test_relu_epilogue_on_a_transposed_identity(),
    lambda: pins.test_relu_epilogue_is_the_triton_clamp(),
    lambda: pins.test_bias_alone_with_zero_a(),
    lambda: pins.test_bias_is_exact_on_integers(),
    lambda: pins.test_bias_is_added_before_the_epilogue(),
    lambda: pins.test_bias_entries_equal_the_full_product(),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor missing: %s" % name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-std=c11", "-shared",
                    "-fPIC", "-o", str(so), str(mutant), "-lm"], check=True)
    failures = 0
    with oracle.use_library(str(so)):
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                failures += 1
            except (RuntimeError, ValueError, FloatingPointError):
                failures += 1
    assert failures >= 1, "no pin caught mutant %s" % name


def test_unmutated_oracle_passes_every_pin():
    for t in PIN_TESTS:
        t()
