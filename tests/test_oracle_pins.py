"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

Nothing here compares the oracle with itself. Each check ties it to
something independent of it:

* the worked 4 x 4 example printed in "Tiled GEMM: Matrix Multiplication in
  CUDA", section 5 (operands from section 3), stored in
  ``tests/golden/worked_example_4x4.txt``;
* closed forms of the definition C[i][j] = sum_k A[i][k] B[k][j]
  ("Tiled Matrix Multiplication in CUDA", section 1): identity, all-ones and
  diagonal operands;
* exact rational brute force (``fractions.Fraction``) on tiny inputs;
* an exact integer product from numpy (a library routine on int64);
* the zero-padding property of "Tiled GEMM: Matrix Multiplication in CUDA",
  section 7.1 (zero rows/columns contribute exactly 0);
* the transpose identity (B^T A^T)^T = A B, which must hold bit for bit
  because the same exact products are added in the same k order.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from tiled_matrix_multiplication_sm_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_4x4.txt")


def load_golden(path=GOLDEN):
    blocks, name = {}, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line[0].isalpha():
                name = line
                blocks[name] = []
                continue
            row = [sum(float(t) for t in tok.split("+")) for tok in line.split()]
            blocks[name].append(row)
    return {k: np.array(v, dtype=np.float64) for k, v in blocks.items()}


# --------------------------------------------------------------------------
# worked example

def test_worked_example_block00(oracle_lib):
    g = load_golden()
    C, _ = oracle_lib.gemm(g["A"], g["B"])
    assert np.array_equal(C[:2, :2], g["block00"])


def test_worked_example_phases(oracle_lib):
    """Phase t=0 and the phase t=1 addends are 2x2 products of K-tiles."""
    g = load_golden()
    A, B = g["A"], g["B"]
    p0, _ = oracle_lib.gemm(A[:2, :2], B[:2, :2])
    p1, _ = oracle_lib.gemm(A[:2, 2:4], B[2:4, :2])
    assert np.array_equal(p0, g["phase0"])
    assert np.array_equal(p1, g["phase1_add"])
    assert np.array_equal(p0 + p1, g["block00"])


def test_worked_example_full_matches_integer_product(oracle_lib):
    g = load_golden()
    C, absAB = oracle_lib.gemm(g["A"], g["B"])
    exact = g["A"].astype(np.int64) @ g["B"].astype(np.int64)
    assert np.array_equal(C, exact.astype(np.float64))
    assert np.array_equal(absAB, exact.astype(np.float64))   # all entries positive


# --------------------------------------------------------------------------
# closed forms

@pytest.mark.parametrize("M,K", [(5, 5), (7, 3), (3, 9), (64, 33)])
def test_identity_right(oracle_lib, M, K):
    A = inputs.matrix(M, K, "normal", seed=11 + M).numpy()
    C, absAB = oracle_lib.gemm(A, np.eye(K))
    assert np.array_equal(C, A.astype(np.float64))
    assert np.array_equal(absAB, np.abs(A.astype(np.float64)))


@pytest.mark.parametrize("K,N", [(4, 4), (3, 8), (17, 5)])
def test_identity_left(oracle_lib, K, N):
    B = inputs.matrix(K, N, "uniform", seed=13 + N).numpy()
    C, _ = oracle_lib.gemm(np.eye(K), B)
    assert np.array_equal(C, B.astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 4, 5), (9, 2, 129), (16, 16, 1000)])
def test_all_ones_gives_K(oracle_lib, M, N, K):
    C, absAB = oracle_lib.gemm(np.ones((M, K)), np.ones((K, N)))
    assert np.array_equal(C, np.full((M, N), float(K)))
    assert np.array_equal(absAB, np.full((M, N), float(K)))


def test_all_minus_ones_sign(oracle_lib):
    C, absAB = oracle_lib.gemm(-np.ones((3, 6)), np.ones((6, 2)))
    assert np.array_equal(C, np.full((3, 2), -6.0))
    assert np.array_equal(absAB, np.full((3, 2), 6.0))


def test_diagonal_scales_rows(oracle_lib):
    d = np.array([2.0, -3.0, 0.5, 7.0])
    B = inputs.matrix(4, 6, "uniform", seed=5).numpy().astype(np.float64)
    C, _ = oracle_lib.gemm(np.diag(d), B)
    assert np.array_equal(C, d[:, None] * B)


def test_rank_one_outer_product(oracle_lib):
    """K = 1: C is the outer product of a column and a row."""
    a = inputs.matrix(6, 1, "normal", seed=1).numpy().astype(np.float64)
    b = inputs.matrix(1, 5, "normal", seed=2).numpy().astype(np.float64)
    C, _ = oracle_lib.gemm(a, b)
    assert np.array_equal(C, a * b)


# --------------------------------------------------------------------------
# brute force and library cross-checks

def fraction_product(A, B):
    M, K = A.shape
    N = B.shape[1]
    C = [[sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)),
              Fraction(0)) for j in range(N)] for i in range(M)]
    S = [[sum((abs(Fraction(float(A[i, k]))) * abs(Fraction(float(B[k, j])))
               for k in range(K)), Fraction(0)) for j in range(N)] for i in range(M)]
    return C, S


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (2, 3, 4, 1), (5, 3, 7, 2),
                                        (3, 6, 2, 3), (7, 7, 8, 4), (4, 1, 6, 5)])
@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_fraction_brute_force(oracle_lib, M, N, K, seed, dist):
    g = inputs.generator(1000 + seed)
    A = inputs.draw(M, K, dist, g).numpy()
    B = inputs.draw(K, N, dist, g).numpy()
    C, absAB = oracle_lib.gemm(A, B)
    Cx, Sx = fraction_product(A, B)
    u = Fraction(1, 2 ** 53)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(C[i, j]) - Cx[i][j])
            assert err <= K * u * Sx[i][j], (i, j)
            assert abs(Fraction(absAB[i, j]) - Sx[i][j]) <= K * u * Sx[i][j]


def test_bf16_inputs_exact_conversion(oracle_lib):
    """bf16 operands enter the oracle exactly (checked with exact fractions)."""
    g = inputs.generator(77)
    A = inputs.draw(3, 5, "normal002", g).to(torch.bfloat16)
    B = inputs.draw(5, 4, "normal002", g).to(torch.bfloat16)
    C, _ = oracle_lib.gemm(A, B)
    Cx, Sx = fraction_product(A.float().numpy(), B.float().numpy())
    for i in range(3):
        for j in range(4):
            assert abs(Fraction(C[i, j]) - Cx[i][j]) <= 5 * Fraction(1, 2 ** 53) * Sx[i][j]


@pytest.mark.parametrize("M,N,K", [(37, 53, 129), (128, 128, 128), (3, 300, 41)])
def test_integer_values_exact_vs_int64_matmul(oracle_lib, M, N, K):
    """Integer operands: every partial sum is exact, so C equals int64 matmul."""
    g = inputs.generator(M * 7 + N)
    A = inputs.draw(M, K, "int4", g).numpy()
    B = inputs.draw(K, N, "int4", g).numpy()
    C, absAB = oracle_lib.gemm(A, B)
    Ai, Bi = A.astype(np.int64), B.astype(np.int64)
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(absAB, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


# --------------------------------------------------------------------------
# invariants

@pytest.mark.parametrize("M,N,K", [(5, 7, 3), (31, 17, 64), (2, 40, 9)])
def test_transpose_identity_bitwise(oracle_lib, M, N, K):
    g = inputs.generator(M + 100 * N + K)
    A = inputs.draw(M, K, "normal", g).numpy()
    B = inputs.draw(K, N, "normal", g).numpy()
    C, S = oracle_lib.gemm(A, B)
    Ct, St = oracle_lib.gemm(B.T, A.T)
    assert np.array_equal(Ct.T, C)
    assert np.array_equal(St.T, S)


def test_zero_padding_leaves_block_unchanged(oracle_lib):
    """Zero rows/columns contribute exactly zero, so padding to tile multiples
    (section 7.1 of the second page) does not move the result by one bit."""
    g = inputs.generator(4242)
    M, N, K = 13, 11, 7
    A = inputs.draw(M, K, "uniform", g).numpy().astype(np.float64)
    B = inputs.draw(K, N, "uniform", g).numpy().astype(np.float64)
    C, _ = oracle_lib.gemm(A, B)
    Ap = np.zeros((16, 8))
    Bp = np.zeros((8, 16))
    Ap[:M, :K] = A
    Bp[:K, :N] = B
    Cp, _ = oracle_lib.gemm(Ap, Bp)
    assert np.array_equal(Cp[:M, :N], C)
    assert not Cp[M:, :].any() and not Cp[:, N:].any()


def test_k_split_sums_match_for_integers(oracle_lib):
    """Splitting K into tiles (the phase loop) reproduces the product exactly
    when all partial sums are exact (integer operands)."""
    g = inputs.generator(99)
    A = inputs.draw(20, 96, "int4", g).numpy()
    B = inputs.draw(96, 24, "int4", g).numpy()
    C, _ = oracle_lib.gemm(A, B)
    acc = np.zeros_like(C)
    for t in range(0, 96, 32):
        part, _ = oracle_lib.gemm(A[:, t:t + 32], B[t:t + 32, :])
        acc += part
    assert np.array_equal(acc, C)


def test_leading_dimension_padding_never_read(oracle_lib):
    A = inputs.matrix(9, 5, "uniform", seed=3, ld=8)       # NaN in columns 5..7
    B = inputs.matrix(5, 6, "uniform", seed=4, ld=11)      # NaN in columns 6..10
    C, S = oracle_lib.gemm(A, B)
    C2, S2 = oracle_lib.gemm(A.contiguous(), B.contiguous())
    assert np.isfinite(C).all()
    assert np.array_equal(C, C2) and np.array_equal(S, S2)


def test_rows_subset_matches_full(oracle_lib):
    g = inputs.generator(5)
    A = inputs.draw(40, 17, "normal", g).numpy()
    B = inputs.draw(17, 23, "normal", g).numpy()
    C, S = oracle_lib.gemm(A, B)
    rows = [39, 0, 7, 7, 22]
    Cr, Sr = oracle_lib.gemm_rows(A, B, rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])


# --------------------------------------------------------------------------
# degenerate shapes and argument checks

def test_empty_sum_is_zero(oracle_lib):
    C, S = oracle_lib.gemm(np.zeros((3, 0)), np.zeros((0, 4)))
    assert C.shape == (3, 4) and not C.any() and not S.any()


@pytest.mark.parametrize("M,N", [(0, 5), (4, 0), (0, 0)])
def test_empty_output(oracle_lib, M, N):
    C, _ = oracle_lib.gemm(np.ones((M, 3)), np.ones((3, N)))
    assert C.shape == (M, N)


def test_mismatched_inner_dimension_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm(np.ones((2, 3)), np.ones((4, 2)))


def test_row_index_out_of_range_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm_rows(np.ones((2, 3)), np.ones((3, 2)), [2])


def test_nan_propagates(oracle_lib):
    A = np.ones((2, 2))
    A[0, 1] = np.nan
    C, _ = oracle_lib.gemm(A, np.ones((2, 2)))
    assert np.isnan(C[0]).all() and np.isfinite(C[1]).all()
