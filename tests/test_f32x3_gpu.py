"""GPU parity of the FP32-accurate tensor-core mode (GEMM_F32_3XTF32).

Each FP32 operand is split into a TF32 part and the FP32 rest (x = hi + lo)
and one TF32 product over 3K computes hi(A)hi(B) + hi(A)lo(B) + lo(A)hi(B).
The result must meet the FP32 mode's bound, |C - C_ref| <= 1e-5 * S per
element, against the FP64 oracle on the same FP32 inputs; integer inputs
(lo = 0, every partial sum exact) must match bit for bit.
"""
import numpy as np
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, assert_parity, to_f64

pytestmark = pytest.mark.gpu

ROW, COL = inp.B_ROW_MAJOR, inp.B_COL_MAJOR
SHAPES = [(1, 1, 1), (3, 5, 7), (128, 128, 128), (129, 257, 33), (300, 520, 260), (64, 1000, 65),
          (1000, 40, 300), (640, 1024, 512), (385, 300, 1001)]


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    h = gemm.Gemm(0)
    yield h
    h.close()


def run(g, A, B, layout, C=None):
    dev = torch.device("cuda", 0)
    M = A.shape[0]
    N = B.shape[1] if layout == ROW else B.shape[0]
    if C is None:
        C = torch.full((M, N), float("nan"), device=dev)
    g.run(A.to(dev), B.to(dev), C, layout, "f32x3")
    g.sync_status()
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", SHAPES)
def test_matches_oracle_at_fp32_tolerance(g, oracle_mod, layout, shape):
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + 3 * N + K)
    C = run(g, A, B, layout)
    assert "f32x3" in g.last_path and "+split3" in g.last_path, g.last_path
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
    rep = assert_parity(C, Cr, S, TOL["f32x3"], f"f32x3 {shape}")
    # well inside the FP32 bound: the dropped lo*lo term is ~2^-22 of |a*b|
    assert rep["max_err_over_S"] < 2e-6, rep


@pytest.mark.parametrize("layout", [ROW, COL])
def test_integer_inputs_bit_exact(g, oracle_mod, layout):
    A, B = inp.make_integer_operands(300, 257, 700, layout_b=layout, seed=17)
    C = run(g, A, B, layout)
    Cr, _ = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
    assert np.array_equal(to_f64(C), Cr)


def test_more_accurate_than_tf32(g, oracle_mod):
    """The same operands in TF32 mode miss the FP32 bound by orders of
    magnitude; the split recovers it."""
    A, B = inp.make_operands(256, 384, 1024, layout_b=ROW, dist="uniform", seed=3)
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), ROW)
    dev = torch.device("cuda", 0)
    C3 = run(g, A, B, ROW)
    Ct = torch.empty((256, 384), device=dev)
    g.run(A.to(dev), B.to(dev), Ct, ROW, "tf32")
    g.sync_status()
    err3 = np.max(np.abs(to_f64(C3) - Cr) / S)
    errt = np.max(np.abs(to_f64(Ct) - Cr) / S)
    assert err3 < 2e-6 < errt, (err3, errt)


@pytest.mark.parametrize("layout", [ROW, COL])
def test_unaligned_operands_and_ldc_padding(g, oracle_mod, layout):
    """Operands at pitches and offsets TMA cannot use (the split reads them
    element-wise) and a C with padding that must stay untouched."""
    M, N, K = 301, 517, 303
    dev = torch.device("cuda", 0)
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=29)
    Ab = torch.zeros((M, K + 3), device=dev)
    Ab[:, 1:K + 1] = A.to(dev)
    rows, cols = B.shape
    Bb = torch.zeros((rows, cols + 5), device=dev)
    Bb[:, 2:cols + 2] = B.to(dev)
    Cb = torch.full((M, N + 7), float("nan"), device=dev)
    C = Cb[:, :N]
    g.run(Ab[:, 1:K + 1], Bb[:, 2:cols + 2], C, layout, "f32x3")
    g.sync_status()
    assert torch.isnan(Cb[:, N:]).all()
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
    assert_parity(C, Cr, S, TOL["f32x3"], "f32x3 unaligned")


@pytest.mark.parametrize("layout", [ROW, COL])
def test_deterministic_and_host_buffers_match(g, layout):
    A, B = inp.make_operands(211, 390, 300, layout_b=layout, seed=51)
    C1 = run(g, A, B, layout).cpu()
    C2 = run(g, A, B, layout).cpu()
    assert torch.equal(C1, C2)
    Ch = torch.empty((211, 390), dtype=torch.float32).pin_memory()
    g.run_host(A.pin_memory(), B.pin_memory(), Ch, layout, "f32x3")
    g.sync_status()
    assert g.last_path.startswith("host+")
    assert torch.equal(C1, Ch)


def test_k_split_for_small_problems(g, oracle_mod):
    """A few tiles over a long K: the tensor-core K split runs over 3K."""
    A, B = inp.make_operands(256, 256, 4096, layout_b=ROW, dist="normal", seed=5)
    C = run(g, A, B, ROW)
    assert "+splitk" in g.last_path, g.last_path
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), ROW)
    assert_parity(C, Cr, S, TOL["f32x3"], "f32x3 split-K")


def test_workload_8192_sampled(g, oracle_mod):
    """The 8192^3 FP32 workload's operands on sampled outputs (first and last
    rows and columns included)."""
    w = inp.ALL_WORKLOADS["fp32x3_8192_row"]
    A, B = inp.make_workload(w)
    dev = torch.device("cuda", 0)
    C = torch.empty((w.M, w.N), device=dev)
    g.run(A.to(dev), B.to(dev), C, w.layout_b, w.dtype)
    g.sync_status()
    rows = inp.sample_indices(w.M, 40, seed=103)
    cols = inp.sample_indices(w.N, 40, seed=203)
    Cs = C[torch.tensor(rows, device=dev)][:, torch.tensor(cols, device=dev)]
    Cr, S = oracle_mod.gemm_sampled(to_f64(A), to_f64(B), rows, cols, w.layout_b)
    assert_parity(Cs, Cr, S, TOL["f32x3"], w.name)


def test_allocation_free_entry_point_refuses_it(g):
    """The split operands need the workspace, which gemm_run_noalloc does not
    have: it refuses the mode before launching anything."""
    from dense_gemm_sm100_gb300 import gemm
    dev = torch.device("cuda", 0)
    A = torch.ones((16, 16), device=dev)
    C = torch.full((16, 16), float("nan"), device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    rc = gemm.gemm_run_noalloc(0, 16, 16, 16, A.data_ptr(), 16, A.data_ptr(), 16, C.data_ptr(), 16,
                               gemm.GEMM_F32_3XTF32, stream)
    assert rc == gemm.GEMM_ERR_INVALID
    torch.cuda.synchronize()
    assert torch.isnan(C).all()
