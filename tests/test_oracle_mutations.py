"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong or transposed index, an ignored leading
dimension, a lost absolute value), compiles that copy on the CPU, and runs
the pins of ``test_oracle_pins`` against it. At least one pin must fail for
every planted mistake; the unmodified source must pass them all. Every
mutation keeps all reads in bounds, so a mutant can only compute wrong
numbers, never crash the test process.
"""
import os

import pytest

import oracle
from oracle import build as oracle_build
from tests import test_oracle_pins as pins

SOURCE = oracle_build.SOURCE

MUTATIONS = {
    "dropped_last_term": ("    for (int k = 0; k < K; ++k) {\n        const double a = A[i * lda + k];",
                          "    for (int k = 0; k < K - 1; ++k) {\n        const double a = A[i * lda + k];"),
    "dropped_first_term": ("    for (int k = 0; k < K; ++k) {\n        const double a = A[i * lda + k];",
                           "    for (int k = 1; k < K; ++k) {\n        const double a = A[i * lda + k];"),
    "wrong_sign": ("c_row[j] += a * b_row[j];", "c_row[j] -= a * b_row[j];"),
    "reversed_k_in_A": ("const double a = A[i * lda + k];",
                        "const double a = A[i * lda + (K - 1 - k)];"),
    "mirrored_column_of_B": ("c_row[j] += a * b_row[j];", "c_row[j] += a * b_row[N - 1 - j];"),
    "ignores_ldb": ("const double* b_row = B + (long)k * ldb;",
                    "const double* b_row = B + (long)k * N;"),
    "lost_abs_in_scale": ("abs_row[j] += abs_a * fabs(b_row[j]);",
                          "abs_row[j] += a * b_row[j];"),
    "bad_init": ("        c_row[j] = 0.0;\n        abs_row[j] = 0.0;",
                 "        c_row[j] = (j == 0) ? 1.0 : 0.0;\n        abs_row[j] = 0.0;"),
    # the extended form
    "ex_trans_a_index": ("trans_a ? A[(long)k * lda + i]", "trans_a ? A[(long)k * lda + (M - 1 - i)]"),
    "ex_trans_b_index": ("trans_b ? B[(long)j * ldb + k]", "trans_b ? B[(long)(N - 1 - j) * ldb + k]"),
    "ex_alpha_dropped": ("double v = alpha * c_row[j];", "double v = c_row[j];"),
    "ex_beta_sign": ("v += beta * C0[i * ldc0 + j];", "v -= beta * C0[i * ldc0 + j];"),
    "ex_bias_dropped": ("                v += bias[j];\n", "                v += 0.0;\n"),
    "ex_dropped_last_term": ("        for (int k = 0; k < K; ++k) {\n            const double a = trans_a",
                             "        for (int k = 0; k < K - 1; ++k) {\n            const double a = trans_a"),
}


def battery(o):
    """The pins, as (name, call) pairs run against oracle handle ``o``."""
    from tests import test_oracle_ex_pins as ex
    return [
        ("ex_transposed", lambda: ex.test_transposed_storage_equals_plain_product(o, True, True)),
        ("ex_alpha", lambda: ex.test_alpha_power_of_two_scales_exactly(o)),
        ("ex_beta", lambda: ex.test_beta_only_returns_scaled_C0(o)),
        ("ex_bias", lambda: ex.test_bias_only_broadcasts_over_rows(o)),
        ("ex_int", lambda: ex.test_integer_full_expression_exact(o)),
        ("worked_block00", lambda: pins.test_worked_example_block00(o)),
        ("worked_phases", lambda: pins.test_worked_example_phases(o)),
        ("identity_right", lambda: pins.test_identity_right(o, 7, 3)),
        ("identity_left", lambda: pins.test_identity_left(o, 3, 8)),
        ("all_ones", lambda: pins.test_all_ones_gives_K(o, 3, 4, 5)),
        ("minus_ones", lambda: pins.test_all_minus_ones_sign(o)),
        ("fraction", lambda: pins.test_fraction_brute_force(o, 5, 3, 7, 2, "normal")),
        ("int64", lambda: pins.test_integer_values_exact_vs_int64_matmul(o, 37, 53, 129)),
        ("transpose", lambda: pins.test_transpose_identity_bitwise(o, 5, 7, 3)),
        ("ld_padding", lambda: pins.test_leading_dimension_padding_never_read(o)),
    ]


def failing_pins(o):
    failed = []
    for name, call in battery(o):
        try:
            call()
        except AssertionError:
            failed.append(name)
    return failed


def test_unmodified_oracle_passes_battery():
    assert failing_pins(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    with open(SOURCE) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    src = os.path.join(tmp_path, "mutant.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    lib = oracle_build.compile_oracle(src, os.path.join(tmp_path, "libmutant.so"))
    failed = failing_pins(oracle.Oracle(lib))
    assert failed, f"no pin caught the planted mistake {name}"
