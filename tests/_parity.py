"""Shared helpers of the parity tests: tolerances and the element-wise check.

The bar, per element: |C_gpu - C_ref| <= tol * S with C_ref and
S = sum_k |a_ik * b_kj| from the FP64 oracle, tol = 1e-5 for the FP32 SIMT
mode and for the FP32-accurate tensor-core mode (three TF32 products), 2e-3
for TF32 and 1e-2 for BF16 (the oracle then reads the same BF16-rounded
inputs).  Any NaN in C_gpu fails.
"""
import numpy as np
import torch

TOL = {"f32": 1e-5, "f32x3": 1e-5, "tf32": 2e-3, "bf16": 1e-2}


def to_f64(t) -> np.ndarray:
    """Exact FP64 copy of a CPU or GPU tensor (FP32 and BF16 widen exactly)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


def parity_report(C_gpu, C_ref: np.ndarray, S: np.ndarray, tol: float):
    C = to_f64(C_gpu)
    assert C.shape == C_ref.shape, (C.shape, C_ref.shape)
    nan = ~np.isfinite(C)
    err = np.abs(C - C_ref)
    bound = tol * S
    bad = (err > bound) | nan
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(S > 0, err / np.where(S > 0, S, 1), np.where(err > 0, np.inf, 0.0))
    return {
        "violations": int(bad.sum()),
        "nan": int(nan.sum()),
        "max_err_over_S": float(np.nanmax(ratio)) if ratio.size else 0.0,
        "first_bad": tuple(int(x) for x in np.argwhere(bad)[0]) if bad.any() else None,
    }


def assert_parity(C_gpu, C_ref, S, tol, label=""):
    rep = parity_report(C_gpu, C_ref, S, tol)
    assert rep["violations"] == 0, f"{label}: {rep}"
    return rep
