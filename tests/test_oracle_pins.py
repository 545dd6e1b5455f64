"""Pins of the CPU oracle to facts fixed outside of it.

Each test is chosen so that a plausible slip in the oracle -- a dropped beta
term, a transposed operand, a wrong leading dimension, a k-range off by one,
C0 read when beta = 0 -- makes at least one of them fail.
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _read_golden_matrices(path):
    mats = {}
    with open(path, encoding="utf-8") as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    i = 0
    while i < len(lines):
        name, r, c = lines[i].split()
        r, c = int(r), int(c)
        rows = [[float(v) for v in lines[i + 1 + j].split()] for j in range(r)]
        mats[name] = np.array(rows, dtype=np.float64)
        assert mats[name].shape == (r, c)
        i += 1 + r
    return mats


def test_worked_example_2x2():
    m = _read_golden_matrices(os.path.join(GOLDEN, "worked_example_2x2.txt"))
    C = oracle.gemm(m["A"], m["B"])
    assert np.array_equal(C, m["C"])


def _brute_force_fraction(A, B, alpha, beta, C0):
    """Exact rational GEMM, column-outer j-k order (independent of oracle.c)."""
    M, K = len(A), len(A[0]) if A else 0
    N = len(B[0]) if B else len(C0[0])
    out = [[Fraction(0)] * N for _ in range(M)]
    for j in range(N):
        for i in range(M):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(A[i][k]) * Fraction(B[k][j])
            v = Fraction(alpha) * s
            if beta != 0:
                v += Fraction(beta) * Fraction(C0[i][j])
            out[i][j] = v
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (8, 2, 5), (5, 8, 1), (7, 7, 8), (2, 9, 3)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, 0.5), (-1.0, 1.0), (0.25, -2.0)])
def test_brute_force_integers(M, N, K, alpha, beta):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = rng.integers(-8, 9, size=(M, K)).astype(np.float64)
    B = rng.integers(-8, 9, size=(K, N)).astype(np.float64)
    C0 = rng.integers(-8, 9, size=(M, N)).astype(np.float64)
    got = oracle.gemm(A, B, alpha, beta, C0)
    want = _brute_force_fraction(A.tolist(), B.tolist(), alpha, beta, C0.tolist())
    for i, j in itertools.product(range(M), range(N)):
        # small integers, dyadic alpha/beta: fp64 is exact here
        assert Fraction(got[i, j]) == want[i][j], (i, j)


def test_identity_gives_alpha_b_plus_beta_c0():
    rng = np.random.default_rng(1)
    n = 33
    B = rng.uniform(-1, 1, size=(n, 17))
    C0 = rng.uniform(-1, 1, size=(n, 17))
    got = oracle.gemm(np.eye(n), B, 1.5, 0.5, C0)
    assert np.array_equal(got, 1.5 * B + 0.5 * C0)


def test_zero_matrix_and_zero_alpha():
    rng = np.random.default_rng(2)
    A = rng.uniform(-1, 1, size=(9, 13))
    B = rng.uniform(-1, 1, size=(13, 11))
    C0 = rng.uniform(-1, 1, size=(9, 11))
    assert np.array_equal(oracle.gemm(np.zeros_like(A), B, 2.0, -0.5, C0), -0.5 * C0)
    assert np.array_equal(oracle.gemm(A, B, 0.0, 0.75, C0), 0.75 * C0)


def test_beta_zero_never_reads_c0():
    rng = np.random.default_rng(3)
    A = rng.uniform(-1, 1, size=(6, 5))
    B = rng.uniform(-1, 1, size=(5, 4))
    C0 = np.full((6, 4), np.nan)
    got = oracle.gemm(A, B, 1.0, 0.0, C0)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, oracle.gemm(A, B))


def test_k_zero_gives_beta_c0():
    C0 = np.arange(12, dtype=np.float64).reshape(3, 4)
    got = oracle.gemm(np.zeros((3, 0)), np.zeros((0, 4)), 1.0, 2.0, C0)
    assert np.array_equal(got, 2.0 * C0)
    assert np.array_equal(oracle.gemm(np.zeros((3, 0)), np.zeros((0, 4))), np.zeros((3, 4)))


def test_rank_one_is_outer_product():
    rng = np.random.default_rng(4)
    a = rng.uniform(-1, 1, size=(19, 1))
    b = rng.uniform(-1, 1, size=(1, 23))
    assert np.array_equal(oracle.gemm(a, b), np.outer(a[:, 0], b[0]))


def test_all_ones():
    K = 37
    C0 = np.full((5, 6), 3.0)
    got = oracle.gemm(np.ones((5, K)), np.ones((K, 6)), 0.5, -1.0, C0)
    assert np.array_equal(got, np.full((5, 6), 0.5 * K - 3.0))


def test_transpose_identity_bitwise():
    # (AB)^T = B^T A^T: element (j,i) of the right side sums the same products
    # in the same k order, so the results agree bit for bit.
    rng = np.random.default_rng(5)
    A = rng.uniform(-1, 1, size=(21, 34))
    B = rng.uniform(-1, 1, size=(34, 15))
    assert np.array_equal(oracle.gemm(A, B).T, oracle.gemm(B.T, A.T))


def test_row_permutation_and_linearity():
    rng = np.random.default_rng(6)
    A = rng.uniform(-1, 1, size=(16, 40))
    B = rng.uniform(-1, 1, size=(40, 12))
    p = rng.permutation(16)
    assert np.array_equal(oracle.gemm(A[p], B), oracle.gemm(A, B)[p])
    # power-of-two alpha scales exactly
    assert np.array_equal(oracle.gemm(A, B, 4.0), 4.0 * oracle.gemm(A, B))


def test_matches_library_matmul_within_fp64_bound():
    rng = np.random.default_rng(7)
    A = rng.standard_normal((64, 300))
    B = rng.standard_normal((300, 48))
    got = oracle.gemm(A, B)
    ref = A @ B
    bound = 300 * np.finfo(np.float64).eps * (np.abs(A) @ np.abs(B))
    assert np.all(np.abs(got - ref) <= bound)


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(8)
    A = rng.uniform(-1, 1, size=(37, 64))
    B = rng.uniform(-1, 1, size=(64, 29))
    C0 = rng.uniform(-1, 1, size=(37, 29))
    r1 = oracle.gemm(A, B, 1.5, 0.5, C0, threads=1)
    r7 = oracle.gemm(A, B, 1.5, 0.5, C0, threads=7)
    assert np.array_equal(r1, r7)


def test_leading_dimension_padding_is_ignored():
    # the C entry point with lda > K and garbage in the pad must give the
    # same result as the packed matrices
    import ctypes
    rng = np.random.default_rng(9)
    M, N, K = 5, 7, 6
    A = rng.uniform(-1, 1, size=(M, K))
    B = rng.uniform(-1, 1, size=(K, N))
    Ap = np.full((M, K + 3), 1e30)
    Ap[:, :K] = A
    Bp = np.full((K, N + 2), -1e30)
    Bp[:, :N] = B
    R = np.full((M, N + 4), 7.0)
    lib = oracle._load()
    dp = ctypes.POINTER(ctypes.c_double)
    rc = lib.oracle_gemm(M, N, K, 1.0, Ap.ctypes.data_as(dp), K + 3, Bp.ctypes.data_as(dp), N + 2,
                         0.0, None, 0, R.ctypes.data_as(dp), N + 4, 2)
    assert rc == 0
    assert np.array_equal(R[:, :N], oracle.gemm(A, B))
    assert np.all(R[:, N:] == 7.0)


def test_bad_arguments_rejected():
    import ctypes
    lib = oracle._load()
    dp = ctypes.POINTER(ctypes.c_double)
    x = np.zeros(16)
    p = x.ctypes.data_as(dp)
    assert lib.oracle_gemm(2, 2, 2, 1.0, p, 1, p, 2, 0.0, None, 0, p, 2, 1) == 1   # lda < K
    assert lib.oracle_gemm(-1, 2, 2, 1.0, p, 2, p, 2, 0.0, None, 0, p, 2, 1) == 1
    assert lib.oracle_gemm(2, 2, 2, 1.0, p, 2, p, 2, 1.0, None, 0, p, 2, 1) == 1   # beta needs C0


def test_normwise_error_definition():
    A = np.array([[1.0, -2.0], [3.0, 4.0]])
    B = np.array([[5.0, 6.0], [-7.0, 8.0]])
    ref = oracle.gemm(A, B)
    denom = oracle.abs_product_max(A, B)
    # sum_k |A||B| = [[19, 22], [43, 50]] -> max 50
    assert denom == 50.0
    G = ref.copy()
    G[1, 0] += 0.5
    assert oracle.normwise_error(G, ref, denom) == 0.01
    G[0, 0] = np.nan
    assert oracle.normwise_error(G, ref, denom) == float("inf")


def test_normwise_denominator_of_the_full_expression():
    A = np.array([[1.0, -2.0], [3.0, 4.0]])
    B = np.array([[5.0, 6.0], [-7.0, 8.0]])
    C0 = np.array([[-10.0, 0.0], [1.0, 2.0]])
    # alpha = 1, beta = 0: the plain max sum_k |A||B| (= 50)
    assert oracle.normwise_denominator(A, B) == oracle.abs_product_max(A, B) == 50.0
    # |alpha| |A||B| + |beta| |C0| = 0.5*[[19,22],[43,50]] + 2*[[10,0],[1,2]] -> max(29.5, 11, 23.5, 29)
    assert oracle.normwise_denominator(A, B, -0.5, -2.0, C0) == 29.5
    # beta = 0 never reads C0
    assert oracle.normwise_denominator(A, B, 1.0, 0.0, np.full((2, 2), np.nan)) == 50.0
