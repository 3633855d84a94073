"""gemm_run_noalloc: the entry point for callers that cannot allocate device
memory (their memory is owned by a framework's memory manager, or they must
not take cudaMalloc's implicit device synchronisation).

It is called through the C ABI, twice in a row on the same device, with
operands whose pitch and address are not 16-byte multiples, so both calls
re-pack A and B into the library's static scratch array and the second call
runs on scratch that still holds the first call's operands.  Each output is
compared with gemm_run's output for the same operands, within the parity
tolerance of the other GPU tests.  This file is collected last.
"""
import numpy as np
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, to_f64

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


def test_noalloc_matches_gemm_run_on_two_calls(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cases = [("f32", inp.B_ROW_MAJOR, (333, 517, 271), 7),
             ("bf16", inp.B_COL_MAJOR, (290, 400, 350), 8)]
    with gemm.Gemm(0) as g:
        for mode, layout, (M, N, K), seed in cases:
            A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=seed, dtype=mode)
            A_d = _unaligned(A, dev, 1)
            B_d = _unaligned(B, dev, 1)
            C_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
            g.run(A_d, B_d, C_ref, layout, mode)
            g.sync_status()
            C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
            rc = _call_noalloc(gemm, A_d, B_d, C, layout, mode)
            assert rc == gemm.GEMM_OK, gemm.gemm_status_string(rc)
            torch.cuda.synchronize()
            _, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
            diff = np.abs(to_f64(C) - to_f64(C_ref))
            assert np.all(np.isfinite(to_f64(C)))
            assert np.all(diff <= TOL[mode] * S), f"{mode}: max |diff|/S = {np.max(diff / S)}"


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
