"""The labelled ladder suite (include/gemm_ladder.h): every kernel against
the FP64 oracle, per element, through the C ABI.  These kernels are not the
library's GEMM path; they reproduce the pages' optimisation steps
("GEMM 性能优化", 八个台阶) and worked kernels ("PMPP Chapter 06", sections 1
and 3) so they can be measured on GB300."""
import numpy as np
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, assert_parity, to_f64

pytestmark = pytest.mark.gpu

STEP_SHAPES = {
    1: [(37, 53, 29), (256, 384, 96)],
    2: [(37, 53, 29), (256, 384, 96)],
    3: [(256, 384, 96)], 4: [(256, 384, 96)], 5: [(256, 384, 96)],
    6: [(256, 384, 96)], 7: [(256, 384, 96), (128, 128, 8)], 8: [(256, 384, 96), (128, 128, 8)],
    102: [(96, 256, 64)],
}


def _run(step, A, B, M, N, K):
    from dense_gemm_sm100_gb300 import gemm
    dev = torch.device("cuda", 0)
    A_d, B_d = A.to(dev), B.to(dev)
    C = torch.full((M, N), float("nan"), device=dev)
    rc = gemm.gemm_ladder_run(step, M, N, K, A_d.data_ptr(), B_d.data_ptr(), C.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == gemm.GEMM_OK, gemm.gemm_status_string(rc)
    torch.cuda.synchronize()
    return C


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build
    build.build()


@pytest.mark.parametrize("step,shape", [(s, sh) for s, shs in STEP_SHAPES.items() for sh in shs])
def test_ladder_step_matches_oracle(oracle_mod, step, shape):
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, dist="normal", seed=step * 10 + M % 7)
    C = _run(step, A, B, M, N, K)
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), inp.B_ROW_MAJOR)
    assert_parity(C, Cr, S, TOL["f32"], f"ladder step {step} {shape}")


@pytest.mark.parametrize("shape", [(37, 53, 29), (64, 80, 48), (200, 136, 130)])
def test_pmpp_corner_turn_matches_oracle(oracle_mod, shape):
    """Column-major B (element (k, j) at B[j*K + k]), bounds-checked tiles."""
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=inp.B_COL_MAJOR, dist="normal", seed=K)
    C = _run(101, A, B, M, N, K)
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), inp.B_COL_MAJOR)
    assert_parity(C, Cr, S, TOL["f32"], f"corner turn {shape}")


def test_ladder_steps_agree_on_integer_inputs(oracle_mod):
    """Integer inputs: every step is exact, so all agree bit for bit."""
    M, N, K = 256, 256, 64
    A, B = inp.make_integer_operands(M, N, K, seed=3)
    Cr, _ = oracle_mod.gemm(to_f64(A), to_f64(B), inp.B_ROW_MAJOR)
    for step in [1, 2, 3, 4, 5, 6, 7, 8]:
        assert np.array_equal(to_f64(_run(step, A, B, M, N, K)), Cr), step


def test_pmpp_kernels_exact_on_integer_inputs(oracle_mod):
    """Integer inputs make every sum exact: the corner-turning kernel (on the
    column-major copy of B, ragged sizes) and the coarsening kernel equal the
    oracle bit for bit."""
    M, N, K = 200, 136, 130
    A, Bc = inp.make_integer_operands(M, N, K, layout_b=inp.B_COL_MAJOR, seed=5)
    Cr, _ = oracle_mod.gemm(to_f64(A), to_f64(Bc), inp.B_COL_MAJOR)
    assert np.array_equal(to_f64(_run(101, A, Bc, M, N, K)), Cr)
    M, N, K = 96, 384, 96
    A, B = inp.make_integer_operands(M, N, K, seed=6)
    Cr, _ = oracle_mod.gemm(to_f64(A), to_f64(B), inp.B_ROW_MAJOR)
    assert np.array_equal(to_f64(_run(102, A, B, M, N, K)), Cr)
