"""Oracle for the dense GEMM C = A·B.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never imports,
links or calls it, and the two share no code: the only module both sides use
is the seeded input generator ``dense_gemm_sm100_gb300.inputs``, which holds
none of the GEMM's arithmetic.

``gemm`` computes, in FP64 and in k order 0..K-1 (``oracle_gemm.c``)::

    C[i, j] = sum_k A(i, k) * B(k, j)
    S[i, j] = sum_k |A(i, k) * B(k, j)|

following the plain definition on "GEMM 性能优化" (section 指标与目标), the
K-sliced accumulation it describes in 台阶 1 (the blocked-matrix identity the
tests check), and the column-major B addressing B[j*ld + k] of the corner
turning example on "PMPP Chapter 06: Performance considerations" (section 1).
S is the per-element scale of the parity tolerance ``|C_gpu - C| <= tol * S``.

Every function here is pinned by ``tests/test_oracle.py`` against brute force
in exact rational arithmetic, closed forms (identity, all-ones), the
blocked-matrix identity and layout invariance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

B_ROW_MAJOR = 0
B_COL_MAJOR = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle_gemm.c`` into ``liboracle_gemm.so`` (plain gcc, -O2).

    ``-ffp-contract=off`` keeps every a*b and every + a separate rounding, so
    the oracle gives bit-identical results on x86-64 and aarch64 hosts.
    """
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64 = ctypes.c_int64
            dp = ctypes.c_void_p
            lib.oracle_gemm_f64.argtypes = [ctypes.c_int, i64, i64, i64,
                                            dp, i64, dp, i64, dp, i64, dp, i64,
                                            ctypes.c_int]
            lib.oracle_gemm_f64.restype = ctypes.c_int
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Host threads a call with ``nthreads=0`` uses (online cores)."""
    return int(_load().oracle_default_threads())


def _as_f64_rows(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.ndim != 2:
        raise ValueError("oracle operands are 2-D arrays")
    return np.ascontiguousarray(x, dtype=np.float64)


def gemm(A: np.ndarray, B: np.ndarray, layout_b: int = B_ROW_MAJOR,
         nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Return ``(C, S)`` for ``C = A·B`` as FP64 arrays of shape (M, N).

    ``A`` is the (M, K) matrix.  ``B`` is the array as stored: shape (K, N)
    for ``B_ROW_MAJOR``; shape (N, K) for ``B_COL_MAJOR``, where row j holds
    column j of the logical K x N matrix (address ``j*K + k``).  Values are
    widened to FP64 exactly (FP32 and BF16 values both fit).
    """
    A = _as_f64_rows(A)
    B = _as_f64_rows(B)
    M, K = A.shape
    if layout_b == B_ROW_MAJOR:
        Kb, N = B.shape
    elif layout_b == B_COL_MAJOR:
        N, Kb = B.shape
    else:
        raise ValueError(f"unknown layout_b {layout_b}")
    if Kb != K:
        raise ValueError(f"inner dimensions differ: A has K={K}, B has K={Kb}")
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    if M == 0 or N == 0:
        return C, S
    lda = max(K, 1)
    ldb = max(B.shape[1], 1)
    rc = _load().oracle_gemm_f64(int(layout_b), M, N, K,
                                 A.ctypes.data if K else None, lda,
                                 B.ctypes.data if K else None, ldb,
                                 C.ctypes.data, N, S.ctypes.data, N,
                                 int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f64 failed with code {rc}")
    return C, S


def gemm_sampled(A: np.ndarray, B: np.ndarray, rows, cols,
                 layout_b: int = B_ROW_MAJOR, nthreads: int = 0):
    """``(C, S)`` restricted to the given rows and columns of the product.

    Element (r, c) of the result is element (rows[r], cols[c]) of ``A·B``:
    the oracle runs on the gathered rows of A and the gathered columns of B,
    with the same k order, so each sampled value is bit-identical to the
    full product's.  This is how full-size workloads are checked.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    A_rows = np.asarray(A)[rows, :]
    if layout_b == B_ROW_MAJOR:
        B_cols = np.asarray(B)[:, cols]
    else:
        B_cols = np.asarray(B)[cols, :]
    return gemm(A_rows, B_cols, layout_b, nthreads)
