"""Plant plausible mistakes in a copy of the oracle and check the pins catch them.

Each mutant is the oracle's C source with one textual change, compiled into a
temporary library on the CPU.  A pin is only worth trusting if it fails for
mistakes like these: a dropped term, a wrong sign, a transposed operand, a
wrong leading dimension.
"""
import ctypes
import os
import random
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_gemm.c")

MUTANTS = {
    "drop_last_k_term": ("for (int64_t k = 0; k < w->K; ++k)", "for (int64_t k = 0; k + 1 < w->K; ++k)"),
    "drop_first_k_term": ("for (int64_t k = 0; k < w->K; ++k)", "for (int64_t k = 1; k < w->K; ++k)"),
    "wrong_sign": ("c[j] += p;", "c[j] -= p;"),
    "transposed_row_major_b": ("? w->B[k * w->ldb + j]", "? w->B[j * w->ldb + k]"),
    "transposed_col_major_b": (": w->B[j * w->ldb + k];", ": w->B[k * w->ldb + j];"),
    "transposed_a": ("w->A[i * w->lda + k]", "w->A[k * w->lda + i]"),
    "abs_missing_in_scale": ("s[j] += fabs(p);", "s[j] += p;"),
    "c_not_cleared": ("c[j] = 0.0;", "(void)0;"),
}


def _compile(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", "-o", str(lib), str(path), "-lm"], check=True)
    cdll = ctypes.CDLL(str(lib))
    i64, dp = ctypes.c_int64, ctypes.c_void_p
    cdll.oracle_gemm_f64.argtypes = [ctypes.c_int, i64, i64, i64, dp, i64, dp, i64,
                                     dp, i64, dp, i64, ctypes.c_int]
    cdll.oracle_gemm_f64.restype = ctypes.c_int
    return cdll


def _run(cdll, A, Bs, layout, M, N, K):
    C = np.full((M, N), 7.0)   # stale values a mutant that skips clearing would keep
    S = np.full((M, N), 7.0)
    A = np.ascontiguousarray(A, dtype=np.float64)
    Bs = np.ascontiguousarray(Bs, dtype=np.float64)
    cdll.oracle_gemm_f64(layout, M, N, K, A.ctypes.data, K, Bs.ctypes.data, Bs.shape[1],
                         C.ctypes.data, N, S.ctypes.data, N, 1)
    return C, S


def _pins_pass(cdll):
    """The brute-force pin of test_oracle.py, on a few non-square shapes."""
    rng = random.Random(99)
    for layout in (0, 1):
        for M, N, K in [(2, 3, 4), (4, 3, 2), (3, 5, 3)]:
            A = [[rng.randint(-16, 16) / 8 for _ in range(K)] for _ in range(M)]
            B = [[rng.randint(-16, 16) / 8 for _ in range(N)] for _ in range(K)]
            Bs = np.array(B) if layout == 0 else np.array(B).T.copy()
            C, S = _run(cdll, np.array(A), Bs, layout, M, N, K)
            for i in range(M):
                for j in range(N):
                    terms = [Fraction(A[i][k]) * Fraction(B[k][j]) for k in range(K)]
                    if Fraction(C[i, j]) != sum(terms) or Fraction(S[i, j]) != sum(abs(t) for t in terms):
                        return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_unmutated_copy_passes(tmp_path):
    assert _pins_pass(_compile(tmp_path, "clean", "c[j] += p;", "c[j] += p;"))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert not _pins_pass(_compile(tmp_path, name, old, new))
