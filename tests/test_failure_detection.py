"""Failure detection without a GPU fault.

Every wait inside the GEMM kernels is bounded: when a wait expires, the
kernel records the expiry in the handle's status word, every role leaves its
loop, copies and MMAs already in flight are waited for (again bounded), tensor
memory is freed, and the kernel ends.  gemm_sync_status turns the status word
into GEMM_ERR_TIMEOUT.

The test hook GEMM_OPT_DEBUG_DROP_LOAD makes CTA 0 skip the copies of its
first stage while still expecting their bytes, a barrier phase that nothing
completes, so the dependent waits expire after the (shortened) wait limit.
The same context then runs a normal GEMM that must match the oracle.
"""
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, assert_parity, to_f64

pytestmark = pytest.mark.gpu

CASES = [  # mode, layout, tensor-core mode, FP32 configuration (0 = chosen)
    ("f32", inp.B_ROW_MAJOR, None, 0),
    ("f32", inp.B_COL_MAJOR, None, 0),
    ("f32", inp.B_ROW_MAJOR, None, 6),  # producer warpgroup with register reallocation
    ("f32", inp.B_COL_MAJOR, None, 6),  # the same, four producer warps turning B
    ("bf16", inp.B_ROW_MAJOR, 1, 0),
    ("bf16", inp.B_ROW_MAJOR, 3, 0),
    ("bf16", inp.B_COL_MAJOR, 3, 0),
    ("tf32", inp.B_ROW_MAJOR, 3, 0),
]


@pytest.mark.parametrize("mode,layout,tc_mode,simt_config", CASES)
def test_expired_wait_is_reported_and_context_survives(oracle_mod, mode, layout, tc_mode, simt_config):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    dev = torch.device("cuda", 0)
    M, N, K = 640, 1024, 512
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=81, dtype=mode)
    A_d, B_d = A.to(dev), B.to(dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    with gemm.Gemm(0) as g:
        g.set_option(gemm.GEMM_OPT_WAIT_TIMEOUT_NS, 20_000_000)  # 20 ms
        if tc_mode is not None:
            g.set_option(gemm.GEMM_OPT_TC_CLUSTER, tc_mode)
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, simt_config)
        g.sync_status()  # clean start

        g.set_option(gemm.GEMM_OPT_DEBUG_DROP_LOAD, 1)
        g.run(A_d, B_d, C, layout, mode)
        with pytest.raises(gemm.GemmError) as err:
            g.sync_status()
        assert err.value.code == gemm.GEMM_ERR_TIMEOUT
        assert "wait expired" in gemm.gemm_last_error_string(g.handle)
        g.sync_status()  # the status word was cleared by the report

        g.set_option(gemm.GEMM_OPT_DEBUG_DROP_LOAD, 0)
        g.run(A_d, B_d, C, layout, mode)
        g.sync_status()
        torch.cuda.synchronize()
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
    assert_parity(C, Cr, S, TOL[mode], f"after recovery {mode}")
