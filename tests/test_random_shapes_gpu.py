"""Seeded random shapes across every path the dispatcher can take: all three
modes, both B layouts, the FP32 tile configurations (128x128 with 8 or 16
consumer warps, 192x128), the tensor-core CTA modes, and CTA caps that make
the tail split (as slices or stream-K) and the tensor-core K split run on
small problems, on device or host buffers.  Each result is checked
against the oracle within the mode's tolerance; integer inputs must match
exactly."""
import random

import numpy as np
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, assert_parity, to_f64

pytestmark = pytest.mark.gpu

N_CASES = 120


def cases():
    rng = random.Random(20261202)
    out = []
    for i in range(N_CASES):
        mode = rng.choice(["f32", "f32", "tf32", "bf16"])
        layout = rng.choice([inp.B_ROW_MAJOR, inp.B_COL_MAJOR])
        M = rng.choice([1, 7, 64, 127, 128, 129, 200, 255, 256, 257, 383, 512, 700])
        N = rng.choice([1, 3, 32, 64, 100, 128, 129, 256, 257, 448, 520, 640])
        K = rng.choice([1, 5, 16, 31, 32, 33, 64, 100, 256, 333, 512, 1000])
        simt_config = rng.choice([0, 0, 1, 6, 7]) if mode == "f32" else 0
        tc_mode = rng.choice([1, 3, 3, 3]) if mode != "f32" else 3
        max_ctas = rng.choice([0, 0, 4, 8, 16])
        integer = rng.random() < 0.3
        elementwise = 1 if (mode == "f32" and layout == inp.B_ROW_MAJOR and rng.random() < 0.3) else 0
        host = rng.random() < 0.2  # through gemm_run_host (pinned host buffers)
        # FP32 tail split: chosen, slices or stream-K (own generator, so the
        # cases above stay as they were)
        stream_k = random.Random(1000 + i).choice([0, 0, 1, 2])
        out.append((i, mode, layout, (M, N, K), simt_config, tc_mode, max_ctas, integer, host, elementwise,
                    stream_k))
    return out


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    h = gemm.Gemm(0)
    yield h
    h.close()


@pytest.mark.parametrize("case", cases(), ids=lambda c: f"case{c[0]}")
def test_random_shape(g, oracle_mod, case):
    from dense_gemm_sm100_gb300 import gemm
    _, mode, layout, (M, N, K), simt_config, tc_mode, max_ctas, integer, host, elementwise, stream_k = case
    if integer:
        A, B = inp.make_integer_operands(M, N, K, layout_b=layout, seed=M * 7 + N, dtype=mode)
    else:
        A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M * 7 + N, dtype=mode)
    g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, simt_config)
    g.set_option(gemm.GEMM_OPT_TC_CLUSTER, tc_mode)
    g.set_option(gemm.GEMM_OPT_MAX_CTAS, max_ctas)
    g.set_option(gemm.GEMM_OPT_ELEMENTWISE, elementwise)
    g.set_option(gemm.GEMM_OPT_STREAM_K, stream_k)
    try:
        if host:
            C = torch.full((M, N), float("nan")).pin_memory()
            g.run_host(A.pin_memory(), B.pin_memory(), C, layout, mode)
        else:
            dev = torch.device("cuda", 0)
            C = torch.full((M, N), float("nan"), device=dev)
            g.run(A.to(dev), B.to(dev), C, layout, mode)
        g.sync_status()
        torch.cuda.synchronize()
        path = g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, 0)
        g.set_option(gemm.GEMM_OPT_TC_CLUSTER, 3)
        g.set_option(gemm.GEMM_OPT_MAX_CTAS, 0)
        g.set_option(gemm.GEMM_OPT_ELEMENTWISE, 0)
        g.set_option(gemm.GEMM_OPT_STREAM_K, 0)
    Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
    if integer:
        assert np.array_equal(to_f64(C), Cr), path
    else:
        assert_parity(C, Cr, S, TOL[mode], path)
