"""Pins for the oracle's extended form (gemm_ex):

    C = alpha * op(A) op(B) + beta * C0 + bias[j]

tied to facts outside the oracle: the plain product (itself pinned in
test_oracle_pins), numpy's transpose (a library primitive) for the
transposed storage orders, exact closed forms for alpha, beta and bias, and
exact rational brute force for the whole expression on tiny inputs.
"""
from fractions import Fraction

import numpy as np
import pytest

from tiled_matrix_multiplication_sm_gb300 import inputs


def draw(rows, cols, dist, seed):
    return inputs.draw(rows, cols, dist, inputs.generator(seed)).numpy().astype(np.float64)


def test_defaults_equal_plain_product(oracle_lib):
    A, B = draw(9, 7, "normal", 1), draw(7, 11, "normal", 2)
    C, S = oracle_lib.gemm_ex(A, B)
    C0, S0 = oracle_lib.gemm(A, B)
    assert np.array_equal(C, C0) and np.array_equal(S, S0)


@pytest.mark.parametrize("ta,tb", [(True, False), (False, True), (True, True)])
def test_transposed_storage_equals_plain_product(oracle_lib, ta, tb):
    """A stored K x M (read transposed) gives the product of A, bit for bit:
    the same products in the same k order."""
    A, B = draw(13, 6, "normal", 3), draw(6, 10, "normal", 4)
    As = A.T.copy() if ta else A
    Bs = B.T.copy() if tb else B
    C, S = oracle_lib.gemm_ex(As, Bs, trans_a=ta, trans_b=tb)
    C0, S0 = oracle_lib.gemm(A, B)
    assert np.array_equal(C, C0) and np.array_equal(S, S0)


def test_transposed_with_padded_leading_dimension(oracle_lib):
    A = draw(5, 8, "uniform", 5)                  # stored K x M with ld 11 (NaN pad)
    store = np.full((5, 11), np.nan)
    store[:, :8] = A
    B = draw(5, 4, "uniform", 6)
    C, _ = oracle_lib.gemm_ex(store[:, :8], B, trans_a=True)
    assert np.isfinite(C).all()
    assert np.array_equal(C, oracle_lib.gemm(A.T.copy(), B)[0])


def test_alpha_power_of_two_scales_exactly(oracle_lib):
    A, B = draw(6, 9, "normal", 7), draw(9, 5, "normal", 8)
    C1, _ = oracle_lib.gemm_ex(A, B)
    C2, S2 = oracle_lib.gemm_ex(A, B, alpha=-4.0)
    assert np.array_equal(C2, -4.0 * C1)
    assert np.array_equal(S2, 4.0 * oracle_lib.gemm(A, B)[1])


def test_beta_only_returns_scaled_C0(oracle_lib):
    A, B = draw(4, 3, "normal", 9), draw(3, 6, "normal", 10)
    C0 = draw(4, 6, "normal", 11)
    C, S = oracle_lib.gemm_ex(A, B, alpha=0.0, beta=0.5, C0=C0)
    assert np.array_equal(C, 0.5 * C0) and np.array_equal(S, np.abs(0.5 * C0))


def test_beta_zero_never_reads_C0(oracle_lib):
    A, B = draw(4, 3, "normal", 12), draw(3, 6, "normal", 13)
    C, _ = oracle_lib.gemm_ex(A, B, beta=0.0, C0=np.full((4, 6), np.nan))
    assert np.isfinite(C).all()


def test_bias_only_broadcasts_over_rows(oracle_lib):
    A, B = draw(5, 3, "normal", 14), draw(3, 7, "normal", 15)
    bias = np.arange(7, dtype=np.float64) - 3.0
    C, S = oracle_lib.gemm_ex(A, B, alpha=0.0, bias=bias)
    assert np.array_equal(C, np.tile(bias, (5, 1)))
    assert np.array_equal(S, np.tile(np.abs(bias), (5, 1)))


def test_integer_full_expression_exact(oracle_lib):
    g = inputs.generator(16)
    A = inputs.draw(17, 23, "int4", g).numpy().astype(np.int64)
    B = inputs.draw(23, 19, "int4", g).numpy().astype(np.int64)
    C0 = inputs.draw(17, 19, "int4", g).numpy().astype(np.int64)
    bias = np.arange(19, dtype=np.int64) % 5 - 2
    C, _ = oracle_lib.gemm_ex(A.T.copy(), B, trans_a=True, alpha=3.0, beta=-2.0, C0=C0,
                              bias=bias)
    assert np.array_equal(C, (3 * (A @ B) - 2 * C0 + bias).astype(np.float64))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fraction_brute_force_full_expression(oracle_lib, seed):
    g = inputs.generator(500 + seed)
    M, N, K = 3, 4, 5
    A = inputs.draw(K, M, "uniform", g).numpy()             # stored transposed
    B = inputs.draw(N, K, "uniform", g).numpy()             # stored transposed
    C0 = inputs.draw(M, N, "uniform", g).numpy()
    bias = inputs.draw(1, N, "uniform", g).numpy()[0]
    alpha, beta = 0.75, -1.5
    C, S = oracle_lib.gemm_ex(A, B, trans_a=True, trans_b=True, alpha=alpha, beta=beta,
                              C0=C0, bias=bias)
    F = Fraction
    for i in range(M):
        for j in range(N):
            dot = sum((F(float(A[k, i])) * F(float(B[j, k])) for k in range(K)), F(0))
            exact = F(alpha) * dot + F(beta) * F(float(C0[i, j])) + F(float(bias[j]))
            assert abs(F(C[i, j]) - exact) <= (K + 3) * F(1, 2 ** 53) * F(S[i, j])


def test_rejects_bad_arguments(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm_ex(np.ones((2, 3)), np.ones((4, 2)))
    with pytest.raises(ValueError):
        oracle_lib.gemm_ex(np.ones((2, 3)), np.ones((3, 2)), beta=1.0)
