"""gemm_run_noalloc: the entry point for callers that cannot allocate device
memory (their memory is owned by a framework's memory manager, or they must
not take cudaMalloc's implicit device synchronisation).

Every case is called through the C ABI twice in a row on the same device,
with different operands, so the second call runs on scratch that still holds
the first call's re-packed operands.  Each output is checked element by
element against the FP64 oracle at the mode's tolerance, and against
gemm_run's output for the same operands.  Cases: the three modes, both B
layouts, operands TMA can read directly (no scratch used) and operands whose
pitch and address are not 16-byte multiples (re-packed into the scratch),
K = 0, the size limit of the scratch, and an in-kernel wait that expires
(reported through the allocation-free status word).  This file is collected
last.
"""
import numpy as np
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, assert_parity, to_f64

pytestmark = pytest.mark.gpu


def _unaligned(t, dev, shift):
    """A copy of t on dev whose rows start `shift` elements into a wider,
    oddly pitched buffer (never a 16-byte multiple)."""
    rows, cols = t.shape
    buf = torch.zeros((rows, cols + 3), dtype=t.dtype, device=dev)
    buf[:, shift:shift + cols] = t.to(dev)
    return buf[:, shift:shift + cols]


def _call_noalloc(gemm, A, B, C, layout, mode):
    M, K = A.shape
    N = C.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return gemm.gemm_run_noalloc(layout, M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(),
                                 B.stride(0), C.data_ptr(), C.stride(0), gemm.DTYPES[mode], stream)


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    with gemm.Gemm(0) as g:
        yield gemm, g, dev


# Aligned shapes keep every pitch a 16-byte multiple (K and N multiples of
# 8), so no operand goes through the scratch; M stays ragged.  Unaligned
# shapes are re-packed.  Both span several tiles with a ragged last one.
SHAPES = {True: [(333, 520, 264), (200, 392, 136)], False: [(333, 517, 271), (290, 400, 350)]}


@pytest.mark.parametrize("mode", ["f32", "tf32", "bf16"])
@pytest.mark.parametrize("layout", [inp.B_ROW_MAJOR, inp.B_COL_MAJOR])
@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "repacked"])
def test_noalloc_matches_oracle_on_two_calls(env, oracle_mod, mode, layout, aligned):
    gemm, g, dev = env
    assert gemm.gemm_noalloc_sync_status(torch.cuda.current_stream().cuda_stream) == gemm.GEMM_OK
    for call, (M, N, K) in enumerate(SHAPES[aligned]):
        A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=7 + 11 * call + layout,
                                 dtype=mode)
        if aligned:
            A_d, B_d = A.to(dev), B.to(dev)
        else:
            A_d, B_d = _unaligned(A, dev, 1), _unaligned(B, dev, 1)
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        rc = _call_noalloc(gemm, A_d, B_d, C, layout, mode)
        assert rc == gemm.GEMM_OK, gemm.gemm_status_string(rc)
        assert gemm.gemm_noalloc_sync_status(torch.cuda.current_stream().cuda_stream) == gemm.GEMM_OK
        Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
        assert_parity(C, Cr, S, TOL[mode], f"noalloc call {call} {mode} layout={layout} aligned={aligned}")
        # the handle-based entry point on the same operands agrees within the same bound
        C_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
        g.run(A_d, B_d, C_ref, layout, mode)
        g.sync_status()
        diff = np.abs(to_f64(C) - to_f64(C_ref))
        assert np.all(diff <= TOL[mode] * S), f"{mode}: max |diff|/S = {np.max(diff / np.maximum(S, 1e-300))}"


@pytest.mark.parametrize("mode", ["f32", "bf16"])
def test_noalloc_integer_inputs_exact(env, oracle_mod, mode):
    """Integer inputs make every partial sum exact: the result equals the
    oracle bit for bit, on re-packed operands."""
    gemm, _, dev = env
    M, N, K = 257, 300, 199
    A, B = inp.make_integer_operands(M, N, K, layout_b=inp.B_ROW_MAJOR, seed=3, dtype=mode)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    rc = _call_noalloc(gemm, _unaligned(A, dev, 1), _unaligned(B, dev, 2), C, inp.B_ROW_MAJOR, mode)
    assert rc == gemm.GEMM_OK
    torch.cuda.synchronize()
    Cr, _ = oracle_mod.gemm(to_f64(A), to_f64(B), inp.B_ROW_MAJOR)
    assert np.array_equal(to_f64(C), Cr)


def test_noalloc_k_zero_writes_zeros(env):
    gemm, _, dev = env
    M, N = 130, 70
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    rc = gemm.gemm_run_noalloc(inp.B_ROW_MAJOR, M, N, 0, 0, 0, 0, N, C.data_ptr(), N, gemm.GEMM_F32, stream)
    assert rc == gemm.GEMM_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


def test_noalloc_expired_wait_is_reported(env, oracle_mod):
    """The test hook makes CTA 0 skip the copies of its first stage while
    still expecting their bytes; its waits expire after a 20 ms limit, the
    kernel ends and the status word reports it.  The next call is clean."""
    gemm, _, dev = env
    M, N, K = 640, 1024, 512
    A, B = inp.make_operands(M, N, K, layout_b=inp.B_ROW_MAJOR, dist="normal", seed=81, dtype="f32")
    A_d, B_d = A.to(dev), B.to(dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert gemm.gemm_noalloc_sync_status(stream) == gemm.GEMM_OK
    assert gemm.gemm_noalloc_set_option(gemm.GEMM_OPT_WAIT_TIMEOUT_NS, 20_000_000) == gemm.GEMM_OK
    try:
        assert gemm.gemm_noalloc_set_option(gemm.GEMM_OPT_DEBUG_DROP_LOAD, 1) == gemm.GEMM_OK
        assert _call_noalloc(gemm, A_d, B_d, C, inp.B_ROW_MAJOR, "f32") == gemm.GEMM_OK
        assert gemm.gemm_noalloc_sync_status(stream) == gemm.GEMM_ERR_TIMEOUT
        assert gemm.gemm_noalloc_sync_status(stream) == gemm.GEMM_OK  # cleared by the report
    finally:
        gemm.gemm_noalloc_set_option(gemm.GEMM_OPT_DEBUG_DROP_LOAD, 0)
        gemm.gemm_noalloc_set_option(gemm.GEMM_OPT_WAIT_TIMEOUT_NS, 4_000_000_000)
    assert _call_noalloc(gemm, A_d, B_d, C, inp.B_ROW_MAJOR, "f32") == gemm.GEMM_OK
    assert gemm.gemm_noalloc_sync_status(stream) == gemm.GEMM_OK
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), inp.B_ROW_MAJOR)
    assert_parity(C, Cr, S, TOL["f32"], "noalloc after the expired wait")


def test_noalloc_rejects_operands_beyond_the_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import gemm
    # A pitch that forces a re-pack of A, sized past the static scratch: the
    # call must refuse before launching anything.  No memory is touched, so
    # fake 4-byte-aligned addresses are enough.
    M, K, N = 1 << 14, (gemm.GEMM_NOALLOC_SCRATCH_BYTES // (4 * (1 << 14))) + 1, 8
    fake = 0x1000004
    rc = gemm.gemm_run_noalloc(0, M, N, K, fake, K, fake, N, fake, N, gemm.GEMM_F32, 0)
    assert rc == gemm.GEMM_ERR_INVALID
