"""Pins of the FP64 oracle against facts fixed by the mathematics and the pages.

None of these checks re-computes the oracle's own formula the same way: they
use exact rational brute force, closed forms, the blocked-matrix identity
("GEMM 性能优化", 台阶 1), the corner-turning addressing B[j*ld + k] ("PMPP
Chapter 06: Performance considerations", section 1) and an independent library
product.  ``test_oracle_mutants.py`` shows that plausible mistakes in the
oracle fail them.
"""
import itertools
import random
from fractions import Fraction

import numpy as np
import pytest

B_ROW, B_COL = 0, 1


def brute_force(A, B_logical):
    """Exact rational C and S by the textbook triple loop."""
    M, K = len(A), len(A[0]) if A else 0
    N = len(B_logical[0]) if B_logical else 0
    C = [[Fraction(0)] * N for _ in range(M)]
    S = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            for k in range(K):
                p = Fraction(A[i][k]) * Fraction(B_logical[k][j])
                C[i][j] += p
                S[i][j] += abs(p)
    return C, S


def stored(B_logical, layout):
    arr = np.array(B_logical, dtype=np.float64)
    return arr if layout == B_ROW else np.ascontiguousarray(arr.T)


def dyadic_matrix(rng, rows, cols):
    # multiples of 1/8 in [-2, 2]: every product and partial sum is exact in FP64
    return [[rng.randint(-16, 16) / 8.0 for _ in range(cols)] for _ in range(rows)]


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_bruteforce_exact_on_all_tiny_shapes(oracle_mod, layout):
    rng = random.Random(1234 + layout)
    for M, N, K in itertools.product(range(1, 5), repeat=3):
        A = dyadic_matrix(rng, M, K)
        B = dyadic_matrix(rng, K, N)
        C, S = oracle_mod.gemm(np.array(A), stored(B, layout), layout)
        Cx, Sx = brute_force(A, B)
        for i in range(M):
            for j in range(N):
                assert Fraction(C[i, j]) == Cx[i][j], (M, N, K, i, j)
                assert Fraction(S[i, j]) == Sx[i][j], (M, N, K, i, j)


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_bruteforce_within_fp64_bound_on_fp32_values(oracle_mod, layout):
    """FP32 inputs: products are exact in FP64, so the only error is the K-1
    FP64 additions: |C - exact| <= (K-1)·2^-53·S_exact (first order)."""
    rng = np.random.default_rng(7 + layout)
    u = 2.0 ** -53
    for M, N, K in [(1, 1, 1), (2, 3, 5), (5, 4, 3), (3, 7, 11), (6, 2, 17)]:
        A = rng.uniform(-1, 1, (M, K)).astype(np.float32).astype(np.float64)
        B = rng.standard_normal((K, N)).astype(np.float32).astype(np.float64)
        C, S = oracle_mod.gemm(A, stored(B.tolist(), layout), layout)
        Cx, Sx = brute_force(A.tolist(), B.tolist())
        for i in range(M):
            for j in range(N):
                bound = Fraction((K - 1) * u * 1.0000001) * Sx[i][j]
                assert abs(Fraction(C[i, j]) - Cx[i][j]) <= bound
                assert abs(Fraction(S[i, j]) - Sx[i][j]) <= bound


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
@pytest.mark.parametrize("M,K", [(1, 1), (7, 7), (33, 33), (5, 9), (40, 17)])
def test_identity_right(oracle_mod, layout, M, K):
    """A·I = A exactly."""
    rng = np.random.default_rng(M * 100 + K)
    A = rng.standard_normal((M, K)).astype(np.float32).astype(np.float64)
    eye = np.eye(K)
    C, S = oracle_mod.gemm(A, eye if layout == B_ROW else eye.T.copy(), layout)
    assert np.array_equal(C, A)
    assert np.array_equal(S, np.abs(A))


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_identity_left(oracle_mod, layout):
    """I·B = B exactly (checks B's indexing on its own)."""
    rng = np.random.default_rng(3)
    K, N = 13, 21
    B = rng.standard_normal((K, N)).astype(np.float32).astype(np.float64)
    C, _ = oracle_mod.gemm(np.eye(K), stored(B.tolist(), layout), layout)
    assert np.array_equal(C, B)


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (16, 9, 100), (2, 2, 1000)])
def test_all_ones(oracle_mod, layout, M, N, K):
    """ones(M,K)·ones(K,N) = K everywhere."""
    C, S = oracle_mod.gemm(np.ones((M, K)), np.ones((K, N) if layout == B_ROW else (N, K)), layout)
    assert np.all(C == K) and np.all(S == K)


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_ones_times_b_is_column_sums(oracle_mod, layout):
    rng = np.random.default_rng(11)
    K, N, M = 37, 19, 4
    B = rng.integers(-8, 9, (K, N)).astype(np.float64)
    C, _ = oracle_mod.gemm(np.ones((M, K)), stored(B.tolist(), layout), layout)
    colsum = np.array([sum(int(B[k, j]) for k in range(K)) for j in range(N)], dtype=np.float64)
    for i in range(M):
        assert np.array_equal(C[i], colsum)


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_blocked_matrix_identity(oracle_mod, layout):
    """Sum over K slices of A[:, Kt]·B[Kt, :] equals A·B ("GEMM 性能优化",
    台阶 1).  Integer inputs make every sum exact, so equality is exact."""
    rng = np.random.default_rng(5)
    M, N, K = 23, 29, 70
    A = rng.integers(-8, 9, (M, K)).astype(np.float64)
    B = rng.integers(-8, 9, (K, N)).astype(np.float64)
    C, S = oracle_mod.gemm(A, stored(B.tolist(), layout), layout)
    for cuts in ([0, 35, 70], [0, 1, 69, 70], [0, 8, 16, 24, 32, 40, 48, 56, 64, 70]):
        Cs = np.zeros((M, N))
        Ss = np.zeros((M, N))
        for k0, k1 in zip(cuts[:-1], cuts[1:]):
            Bp = B[k0:k1, :]
            Ct, St = oracle_mod.gemm(A[:, k0:k1].copy(), stored(Bp.tolist(), layout), layout)
            Cs += Ct
            Ss += St
        assert np.array_equal(Cs, C)
        assert np.array_equal(Ss, S)


def test_layout_invariance_bitwise(oracle_mod):
    """The same logical B stored row- or column-major gives identical bits."""
    rng = np.random.default_rng(9)
    M, N, K = 31, 45, 77
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32).astype(np.float64)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32).astype(np.float64)
    C1, S1 = oracle_mod.gemm(A, B, B_ROW)
    C2, S2 = oracle_mod.gemm(A, np.ascontiguousarray(B.T), B_COL)
    assert np.array_equal(C1, C2) and np.array_equal(S1, S2)


def test_not_symmetric_in_operands(oracle_mod):
    """A transposed or swapped operand would give a different matrix."""
    A = np.array([[1.0, 2.0], [3.0, 4.0]])
    B = np.array([[5.0, 6.0], [7.0, 8.0]])
    C, _ = oracle_mod.gemm(A, B, B_ROW)
    assert np.array_equal(C, np.array([[19.0, 22.0], [43.0, 50.0]]))
    C, _ = oracle_mod.gemm(A, B, B_COL)  # B stored column-major: logical [[5,7],[6,8]]
    assert np.array_equal(C, np.array([[17.0, 23.0], [39.0, 53.0]]))


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_matches_library_product(oracle_mod, layout):
    """Cross-check with numpy's float64 product (a library, not the oracle)."""
    rng = np.random.default_rng(21)
    M, N, K = 65, 130, 257
    A = rng.standard_normal((M, K)).astype(np.float32).astype(np.float64)
    B = rng.standard_normal((K, N)).astype(np.float32).astype(np.float64)
    C, S = oracle_mod.gemm(A, stored(B.tolist(), layout), layout)
    ref = A @ B
    assert np.all(np.abs(C - ref) <= 1e-13 * S)
    assert np.allclose(S, np.abs(A) @ np.abs(B), rtol=1e-13, atol=0)


def test_k_zero_is_empty_sum(oracle_mod):
    C, S = oracle_mod.gemm(np.zeros((3, 0)), np.zeros((0, 4)), B_ROW)
    assert C.shape == (3, 4) and np.all(C == 0) and np.all(S == 0)


def test_empty_outputs(oracle_mod):
    C, S = oracle_mod.gemm(np.zeros((0, 5)), np.zeros((5, 4)), B_ROW)
    assert C.shape == (0, 4)
    C, S = oracle_mod.gemm(np.zeros((3, 5)), np.zeros((5, 0)), B_ROW)
    assert C.shape == (3, 0)


def test_thread_count_does_not_change_bits(oracle_mod):
    rng = np.random.default_rng(2)
    A = rng.standard_normal((37, 50))
    B = rng.standard_normal((50, 41))
    C1, S1 = oracle_mod.gemm(A, B, B_ROW, nthreads=1)
    C2, S2 = oracle_mod.gemm(A, B, B_ROW, nthreads=7)
    C3, S3 = oracle_mod.gemm(A, B, B_ROW, nthreads=0)
    assert np.array_equal(C1, C2) and np.array_equal(C1, C3)
    assert np.array_equal(S1, S2) and np.array_equal(S1, S3)


@pytest.mark.parametrize("layout", [B_ROW, B_COL])
def test_sampled_equals_full(oracle_mod, layout):
    rng = np.random.default_rng(4)
    M, N, K = 40, 33, 29
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    Bs = stored(B.tolist(), layout)
    C, S = oracle_mod.gemm(A, Bs, layout)
    rows, cols = [0, 7, 39], [1, 2, 32]
    Cs, Ss = oracle_mod.gemm_sampled(A, Bs, rows, cols, layout)
    assert np.array_equal(Cs, C[np.ix_(rows, cols)])
    assert np.array_equal(Ss, S[np.ix_(rows, cols)])


def test_bad_arguments_raise(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.gemm(np.zeros((2, 3)), np.zeros((4, 2)), B_ROW)
    with pytest.raises(ValueError):
        oracle_mod.gemm(np.zeros((2, 3)), np.zeros((3, 2)), 5)
