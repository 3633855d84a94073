"""GPU parity of the C-ABI GEMM against the FP64 oracle, element by element.

Every case draws seeded inputs (dense_gemm_sm100_gb300.inputs), runs the
library through its C ABI on cuda:0, and checks |C_gpu - C_ref| <= tol * S
per element (tests/_parity.py).  Integer-valued inputs make every mode exact,
so those cases must match bit for bit.
"""
import numpy as np
import pytest
import torch

from dense_gemm_sm100_gb300 import inputs as inp
from tests._parity import TOL, assert_parity, to_f64

pytestmark = pytest.mark.gpu

MODES = ["f32", "tf32", "bf16"]
ROW, COL = inp.B_ROW_MAJOR, inp.B_COL_MAJOR


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    h = gemm.Gemm(0)
    yield h
    h.close()


def run_gpu(g, A, B, layout, mode, C=None):
    dev = torch.device("cuda", 0)
    A_d, B_d = A.to(dev), B.to(dev)
    M = A.shape[0]
    N = B.shape[1] if layout == ROW else B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
    g.run(A_d, B_d, C, layout, mode)
    g.sync_status()
    torch.cuda.synchronize()
    return C


def oracle_of(oracle_mod, A, B, layout):
    return oracle_mod.gemm(to_f64(A), to_f64(B), layout)


SMALL_SHAPES = [
    (1, 1, 1), (3, 5, 7), (16, 16, 16), (128, 128, 128), (129, 257, 33),
    (200, 300, 100), (255, 129, 127), (300, 520, 260), (64, 1000, 65), (1000, 40, 300),
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_small_shapes_random(g, oracle_mod, mode, layout, shape):
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal",
                             seed=M * 7 + N * 3 + K, dtype=mode)
    C = run_gpu(g, A, B, layout, mode)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C, Cr, S, TOL[mode], f"{mode} layout={layout} {shape}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", [ROW, COL])
def test_integer_inputs_bit_exact(g, oracle_mod, mode, layout):
    M, N, K = 257, 515, 300
    A, B = inp.make_integer_operands(M, N, K, layout_b=layout, seed=5, dtype=mode)
    C = run_gpu(g, A, B, layout, mode)
    Cr, _ = oracle_of(oracle_mod, A, B, layout)
    assert np.array_equal(to_f64(C), Cr)


@pytest.mark.parametrize("mode", MODES)
def test_padding_and_neighbours_untouched(g, oracle_mod, mode):
    """Only C[i, j] with i < M and j < N is written ("PMPP Chapter 06",
    corner-turning example: guarded stores)."""
    M, N, K = 131, 261, 77
    A, B = inp.make_operands(M, N, K, seed=9, dtype=mode)
    dev = torch.device("cuda", 0)
    big = torch.full((M + 3, N + 13), float("nan"), dtype=torch.float32, device=dev)
    C = big[1:M + 1, 4:N + 4]  # ldc = N + 13, guard rows and columns on each side
    run_gpu(g, A, B, ROW, mode, C=C)
    Cr, S = oracle_of(oracle_mod, A, B, ROW)
    assert_parity(C, Cr, S, TOL[mode])
    host = big.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[1:M + 1, 4:N + 4] = False
    assert torch.isnan(host[mask]).all()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", [ROW, COL])
def test_deterministic(g, mode, layout):
    A, B = inp.make_operands(300, 600, 500, layout_b=layout, seed=3, dtype=mode)
    C1 = run_gpu(g, A, B, layout, mode).cpu()
    C2 = run_gpu(g, A, B, layout, mode).cpu()
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", [ROW, COL])
def test_blocked_matrix_identity(g, oracle_mod, mode, layout):
    """Sum of the products over two K slices equals the full product ("GEMM
    性能优化", 台阶 1).  The slices start at pointer offsets, so the second one
    is generally not 16-byte aligned and goes through the re-pack path.
    Integer inputs: exact."""
    M, N, K, k0 = 190, 330, 300, 137
    A, B = inp.make_integer_operands(M, N, K, layout_b=layout, seed=17, dtype=mode)
    dev = torch.device("cuda", 0)
    A_d, B_d = A.to(dev), B.to(dev)
    full = torch.empty((M, N), dtype=torch.float32, device=dev)
    p1 = torch.empty_like(full)
    p2 = torch.empty_like(full)
    g.run(A_d, B_d, full, layout, mode)
    if layout == ROW:
        g.run(A_d[:, :k0], B_d[:k0, :], p1, layout, mode)
        g.run(A_d[:, k0:], B_d[k0:, :], p2, layout, mode)
    else:
        g.run(A_d[:, :k0], B_d[:, :k0], p1, layout, mode)
        g.run(A_d[:, k0:], B_d[:, k0:], p2, layout, mode)
    g.sync_status()
    assert torch.equal((p1 + p2).cpu(), full.cpu())
    Cr, _ = oracle_of(oracle_mod, A, B, layout)
    assert np.array_equal(to_f64(full), Cr)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", [ROW, COL])
def test_unaligned_leading_dimensions(g, oracle_mod, mode, layout):
    """Odd leading dimensions and an offset base pointer, which TMA cannot
    address: re-packed first; FP32 with row-major B can instead copy them
    element by element into the shared-memory ring (cp.async,
    GEMM_OPT_ELEMENTWISE = 1).  Same bits either way, given the same K split
    (the element-wise form has no stream-K, so both runs take slices).  The
    small-problem kernel, which reads any pitch where it is, is kept out."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = 97, 203, 151
    A, B = inp.make_operands(M, N, K, layout_b=layout, seed=23, dist="normal", dtype=mode)
    dev = torch.device("cuda", 0)
    Ap = torch.zeros((M, K + 3), dtype=A.dtype, device=dev)
    Ap[:, 1:K + 1] = A.to(dev)
    rows_b, cols_b = B.shape
    Bp = torch.zeros((rows_b, cols_b + 5), dtype=B.dtype, device=dev)
    Bp[:, 1:cols_b + 1] = B.to(dev)
    Cbig = torch.zeros((M, N + 1), dtype=torch.float32, device=dev)
    C = Cbig[:, :N]
    g.set_option(gemm.GEMM_OPT_STREAM_K, 1)
    g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 1)
    try:
        g.run(Ap[:, 1:K + 1], Bp[:, 1:cols_b + 1], C, layout, mode)
        g.sync_status()
        assert "repackA" in g.last_path and "repackB" in g.last_path
        if mode == "f32" and layout == ROW:
            C_first = C.clone()
            g.set_option(gemm.GEMM_OPT_ELEMENTWISE, 1)
            try:
                g.run(Ap[:, 1:K + 1], Bp[:, 1:cols_b + 1], C, layout, mode)
                g.sync_status()
                assert "+cpasync" in g.last_path and "repack" not in g.last_path, g.last_path
            finally:
                g.set_option(gemm.GEMM_OPT_ELEMENTWISE, 0)
            assert torch.equal(C_first, C)
    finally:
        g.set_option(gemm.GEMM_OPT_STREAM_K, 0)
        g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 0)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C, Cr, S, TOL[mode])


@pytest.mark.parametrize("mode", MODES)
def test_forced_repack_gives_same_bits(g, mode):
    """The same persistent kernel on the operands in place and re-packed (the
    small-problem kernel, which would take this shape, is kept out)."""
    from dense_gemm_sm100_gb300 import gemm
    A, B = inp.make_operands(160, 288, 192, seed=31, dtype=mode)
    g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 1)
    try:
        C1 = run_gpu(g, A, B, ROW, mode).cpu()
        g.set_option(gemm.GEMM_OPT_FORCE_REPACK, 1)
        C2 = run_gpu(g, A, B, ROW, mode).cpu()
        assert "repack" in g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_FORCE_REPACK, 0)
        g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 0)
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("mode", MODES)
def test_layout_invariance(g, mode):
    """The same logical B stored either way gives the same C."""
    A, Br = inp.make_operands(200, 333, 271, layout_b=ROW, seed=41, dtype=mode)
    _, Bc = inp.make_operands(200, 333, 271, layout_b=COL, seed=41, dtype=mode)
    C1 = run_gpu(g, A, Br, ROW, mode).cpu()
    C2 = run_gpu(g, A, Bc, COL, mode).cpu()
    if mode == "f32":
        assert torch.equal(C1, C2)  # same k order per element in both layouts
    else:
        assert torch.allclose(C1, C2, rtol=0, atol=1e-5 * float(C1.abs().max()) + 1e-30)


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", [(300, 520, 260), (257, 600, 64)])
def test_tma_store_epilogue_matches_thread_stores(g, mode, shape):
    """C written through TMA stores (the default when C is 16-byte aligned)
    equals C written by per-thread stores, bit for bit, and leaves the ldc
    padding alone."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, dist="normal", seed=K + 5, dtype=mode)
    dev = torch.device("cuda", 0)
    big = torch.full((M, N + 12), float("nan"), device=dev)  # ldc = N + 12 keeps 16-byte rows
    C_tma = big[:, :N]
    g.set_option(gemm.GEMM_OPT_SPLIT_K, 1)  # a K split would write C from its reduction kernel
    try:
        run_gpu(g, A, B, ROW, mode, C=C_tma)
        g.set_option(gemm.GEMM_OPT_TC_TMA_STORE, 0)
        C_thr = run_gpu(g, A, B, ROW, mode).cpu()
    finally:
        g.set_option(gemm.GEMM_OPT_TC_TMA_STORE, 1)
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    assert torch.equal(C_tma.cpu(), C_thr)
    assert torch.isnan(big[:, N:].cpu()).all()


@pytest.mark.parametrize("mode", MODES)
def test_k_zero_writes_zeros(g, mode):
    dev = torch.device("cuda", 0)
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    A = torch.empty((5, 0), dtype=dt, device=dev)
    B = torch.empty((0, 9), dtype=dt, device=dev)
    C = torch.full((5, 9), 3.0, device=dev)
    g.run(A, B, C, ROW, mode)
    g.sync_status()
    assert torch.equal(C.cpu(), torch.zeros(5, 9))


def test_empty_output_is_noop(g):
    dev = torch.device("cuda", 0)
    A = torch.ones((0, 4), device=dev)
    B = torch.ones((4, 6), device=dev)
    C = torch.empty((0, 6), device=dev)
    g.run(A, B, C)
    g.sync_status()
    assert g.last_path == "noop"


def test_errors_are_reported(g):
    from dense_gemm_sm100_gb300 import gemm
    dev = torch.device("cuda", 0)
    A = torch.ones((4, 4), device=dev)
    rc = gemm.gemm_run(g.handle, 0, 4, 4, 4, A.data_ptr(), 3, A.data_ptr(), 4, A.data_ptr(), 4, 0, 0)
    assert rc == gemm.GEMM_ERR_INVALID
    assert "lda" in gemm.gemm_last_error_string(g.handle)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", [ROW, COL])
def test_run_host_matches_device(g, mode, layout):
    A, B = inp.make_operands(211, 390, 300, layout_b=layout, seed=51, dtype=mode)
    Cd = run_gpu(g, A, B, layout, mode).cpu()
    Ch = torch.empty((211, 390), dtype=torch.float32).pin_memory()
    g.run_host(A.pin_memory(), B.pin_memory(), Ch, layout, mode)
    g.sync_status()
    assert g.last_path.startswith("host+")
    assert torch.equal(Cd, Ch)


HOST_BLOCK_CASES = [  # mode, layout, CTA cap, shape, blocks (None: one launch)
    ("f32", ROW, 2, (2048, 2048, 256), None),
    ("f32", COL, 4, (3000, 3000, 256), "16x1"),
    ("f32", ROW, 2, (3000, 1000, 256), None),
    ("f32", ROW, 2, (10000, 256, 1024), "14x1"),
    ("f32", COL, 4, (2000, 1000, 512), None),
    ("bf16", ROW, 16, (1000, 3000, 256), "1x2"),
    ("bf16", COL, 8, (1000, 3000, 256), "2x2"),
    ("bf16", ROW, 8, (3000, 3000, 1024), "6x2"),
    ("tf32", COL, 8, (2300, 2000, 512), "5x2"),
    ("tf32", ROW, 4, (1000, 1000, 512), "2x2"),
]


@pytest.mark.parametrize("mode,layout,max_ctas,shape,blocks", HOST_BLOCK_CASES)
def test_run_host_blocks_match_oracle(g, oracle_mod, mode, layout, max_ctas, shape, blocks):
    """gemm_run_host cuts C into blocks (row panels of A x column panels of B)
    whose copies in and out overlap the GEMMs of the neighbouring blocks.  The
    tile-slot cap shrinks the waves so that small problems exercise the
    plans; host leading dimensions are wider than the matrices.  Same
    tolerance as one call, exact on integer inputs, nothing written past N."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    g.set_option(gemm.GEMM_OPT_MAX_CTAS, max_ctas)
    try:
        for integer in (False, True):
            if integer:
                A, B = inp.make_integer_operands(M, N, K, layout_b=layout, seed=M, dtype=mode)
            else:
                A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + N, dtype=mode)
            Ap = torch.zeros((M, K + 5), dtype=A.dtype).pin_memory()[:, :K]
            Ap.copy_(A)
            Bp = torch.zeros((B.shape[0], B.shape[1] + 7), dtype=B.dtype).pin_memory()[:, :B.shape[1]]
            Bp.copy_(B)
            Ch = torch.full((M, N + 3), -1.0).pin_memory()
            g.run_host(Ap, Bp, Ch[:, :N], layout, mode)
            g.sync_status()
            torch.cuda.synchronize()
            assert g.last_path.startswith("host+")
            if blocks is None:
                assert "+blocks" not in g.last_path
            else:
                assert g.last_path.endswith(f"+blocks{blocks}"), g.last_path
            assert torch.all(Ch[:, N:] == -1.0)  # nothing written past N
            Cr, S = oracle_of(oracle_mod, A, B, layout)
            if integer:
                assert np.array_equal(to_f64(Ch[:, :N]), Cr), g.last_path
            else:
                assert_parity(Ch[:, :N], Cr, S, TOL[mode], g.last_path)
    finally:
        g.set_option(gemm.GEMM_OPT_MAX_CTAS, 0)


@pytest.mark.parametrize("mode", MODES)
def test_run_host_pageable_memory(g, oracle_mod, mode):
    """Host buffers that are not page-locked work too (the copies then block
    the calling thread); large enough to be cut into blocks."""
    from dense_gemm_sm100_gb300 import gemm
    g.set_option(gemm.GEMM_OPT_MAX_CTAS, 8)
    try:
        M, N, K = 3000, 3000, 1024
        A, B = inp.make_integer_operands(M, N, K, seed=11, dtype=mode)
        C = torch.full((M, N), -1.0)
        g.run_host(A, B, C, ROW, mode)
        g.sync_status()
        torch.cuda.synchronize()
        assert "+blocks" in g.last_path, g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_MAX_CTAS, 0)
    Cr, _ = oracle_of(oracle_mod, A, B, ROW)
    assert np.array_equal(to_f64(C), Cr)


def test_run_host_orders_with_the_callers_stream(g, oracle_mod):
    """The copies of A and B start after work queued earlier on the caller's
    stream (here: the copy that fills the host buffer of A), and C is
    complete once that stream is synchronised."""
    from dense_gemm_sm100_gb300 import gemm
    g.set_option(gemm.GEMM_OPT_MAX_CTAS, 4)
    try:
        s = torch.cuda.Stream()
        M, N, K = 3000, 3000, 256
        A, B = inp.make_integer_operands(M, N, K, layout_b=COL, seed=7)
        A_d = A.cuda()
        Cr, _ = oracle_of(oracle_mod, A, B, COL)
        for _ in range(3):
            Ap = torch.zeros((M, K)).pin_memory()
            Ch = torch.zeros((M, N)).pin_memory()
            with torch.cuda.stream(s):
                torch.cuda._sleep(2_000_000)  # keep the stream busy before the fill
                Ap.copy_(A_d, non_blocking=True)
            g.run_host(Ap, B.pin_memory(), Ch, COL, "f32", stream=s)
            s.synchronize()
            assert g.last_path.endswith("+blocks16x1")
            assert np.array_equal(to_f64(Ch), Cr)
    finally:
        g.set_option(gemm.GEMM_OPT_MAX_CTAS, 0)


def test_workspace_limit_reports_nomem_without_launching(g, oracle_mod):
    """An allocation failure injected on the host: with the workspace capped,
    a run that needs to re-pack its operands returns GEMM_ERR_NOMEM before
    any launch, C stays untouched, and the handle works again once the cap
    is lifted."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = 300, 257, 131  # K and N odd: both operands need a re-pack
    A, B = inp.make_integer_operands(M, N, K, seed=3)
    dev = torch.device("cuda", 0)
    A_d, B_d = A.to(dev), B.to(dev)
    C = torch.full((M, N), -7.0, device=dev)
    g.sync_status()
    before = g.launch_count
    g.set_option(gemm.GEMM_OPT_WORKSPACE_LIMIT, 4096)
    try:
        h = gemm.Gemm(0)  # a fresh handle has no workspace yet
        h.set_option(gemm.GEMM_OPT_WORKSPACE_LIMIT, 4096)
        h.set_option(gemm.GEMM_OPT_SIMT_SMALL, 1)  # the small-problem kernel would read in place
        with pytest.raises(gemm.GemmError) as err:
            h.run(A_d, B_d, C, ROW, "f32")
        assert err.value.code == gemm.GEMM_ERR_NOMEM
        assert "GEMM_OPT_WORKSPACE_LIMIT" in gemm.gemm_last_error_string(h.handle)
        assert h.launch_count == 0
        torch.cuda.synchronize()
        assert torch.all(C == -7.0)
        h.set_option(gemm.GEMM_OPT_WORKSPACE_LIMIT, 0)
        h.run(A_d, B_d, C, ROW, "f32")
        h.sync_status()
        h.close()
    finally:
        g.set_option(gemm.GEMM_OPT_WORKSPACE_LIMIT, 0)
    assert g.launch_count == before
    Cr, _ = oracle_of(oracle_mod, A, B, ROW)
    assert np.array_equal(to_f64(C), Cr)


def test_launch_count_increments(g):
    before = g.launch_count
    A, B = inp.make_operands(64, 64, 64, seed=1)
    run_gpu(g, A, B, ROW, "f32")
    assert g.launch_count == before + 1


# ------------------------------------------------------- clustered tensor-core kernel

CLUSTER_SHAPES = [(129, 257, 33), (257, 600, 64), (300, 520, 260), (385, 300, 100),
                  (1000, 40, 300), (640, 1024, 512),
                  (300, 448, 96)]  # whole 128-byte chunks of B, the last box half past N


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", CLUSTER_SHAPES)
def test_cluster_pairs_match_oracle_and_single_cta(g, oracle_mod, mode, layout, shape):
    """CTA pairs (mode 3) run the pair MMA (tcgen05 cta_group::2, 256x256
    per pair).  Odd tile-row counts leave one CTA of the last pair entirely
    out of range.  Same parity, and the same bits as the one-CTA kernel
    (mode 1)."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + 3 * N + K, dtype=mode)
    g.set_option(gemm.GEMM_OPT_SPLIT_K, 1)  # these small shapes would otherwise be cut along K
    g.set_option(gemm.GEMM_OPT_TC_CLUSTER, 1)
    C1 = run_gpu(g, A, B, layout, mode).cpu()
    assert "pair" not in g.last_path
    g.set_option(gemm.GEMM_OPT_TC_CLUSTER, 3)
    try:
        C2 = run_gpu(g, A, B, layout, mode).cpu()
        assert "pair256x256" in g.last_path
        # pair MMA with row-major B: one 3-D TMA box per stage when N is whole chunks
        chunk = 64 if mode == "bf16" else 32
        b3d = layout == ROW and M > 128 and N % chunk == 0
        assert ("+b3d" in g.last_path) == b3d, g.last_path
        # the one-CTA run above used the 3-D box under the same condition
        g.set_option(gemm.GEMM_OPT_TC_CLUSTER, 1)
        run_gpu(g, A, B, layout, mode)
        assert ("+b3d" in g.last_path) == (layout == ROW and N % chunk == 0), g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_TC_CLUSTER, 3)
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C2, Cr, S, TOL[mode], f"pair MMA {mode} {shape}")
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("value", [0, 2, 4, -1])
def test_tc_cluster_option_accepts_only_one_cta_and_pair_modes(g, value):
    """Only the one-CTA (1) and pair-MMA (3) tensor-core modes exist; any
    other value is refused and leaves the handle's mode unchanged."""
    from dense_gemm_sm100_gb300 import gemm
    with pytest.raises(gemm.GemmError) as err:
        g.set_option(gemm.GEMM_OPT_TC_CLUSTER, value)
    assert err.value.code == gemm.GEMM_ERR_INVALID
    A, B = inp.make_operands(300, 256, 64, layout_b=ROW, dist="normal", seed=5, dtype="bf16")
    run_gpu(g, A, B, ROW, "bf16")
    assert "pair256x256" in g.last_path


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", CLUSTER_SHAPES + [(520, 300, 33), (600, 512, 200), (300, 256, 1000)])
def test_pair_wide_stages_same_bits(g, oracle_mod, mode, layout, shape):
    """Pair MMA with two 128-byte K slices per ring stage (three stages)
    against one slice per stage (six stages): the MMA instructions run in the
    same K order, so the bits are the same; K lengths that end inside a
    stage, or inside its first slice, take zero-filled slices."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=2 * M + N + 5 * K, dtype=mode)
    g.set_option(gemm.GEMM_OPT_SPLIT_K, 1)
    try:
        g.set_option(gemm.GEMM_OPT_TC_STAGE_SLICES, 1)
        C1 = run_gpu(g, A, B, layout, mode).cpu()
        assert "pair256x256_" in g.last_path, g.last_path
        g.set_option(gemm.GEMM_OPT_TC_STAGE_SLICES, 2)
        C2 = run_gpu(g, A, B, layout, mode).cpu()
        assert "pair256x256w_" in g.last_path, g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_TC_STAGE_SLICES, 0)
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C2, Cr, S, TOL[mode], f"wide stages {mode} {shape}")
    assert torch.equal(C1, C2)


# ------------------------------------------------------- split-K (FP32 path)

SIMT_CONFIG_SHAPES = [(1, 1, 1), (129, 257, 33), (300, 520, 260), (640, 1030, 512)]


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", SIMT_CONFIG_SHAPES)
def test_simt_configs_match_oracle(g, oracle_mod, config, layout, shape):
    """Every FP32 tile configuration (GEMM_OPT_SIMT_CONFIG 1..5: 128x128
    packed and scalar, 64x128, 64x64, and 128x256 with register reallocation
    for row-major B) on ragged shapes spanning several tiles."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, config)
    try:
        A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + N + K + config)
        C = run_gpu(g, A, B, layout, "f32")
        Cr, S = oracle_mod.gemm(to_f64(A), to_f64(B), layout)
        assert_parity(C, Cr, S, TOL["f32"], f"config {config} {shape}")
        Ai, Bi = inp.make_integer_operands(M, N, K, layout_b=layout, seed=config)
        Ci = run_gpu(g, Ai, Bi, layout, "f32")
        Cri, _ = oracle_mod.gemm(to_f64(Ai), to_f64(Bi), layout)
        assert np.array_equal(to_f64(Ci), Cri), f"config {config} integer inputs"
    finally:
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, 0)


@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", [(129, 257, 300), (640, 1030, 512), (385, 200, 1001)])
def test_simt_configs_same_bits(g, layout, shape):
    """Without a K split every FP32 configuration adds each element's
    products in k order with one FMA per product (8x8 or 8x4 thread tiles,
    8, 12 or 16 consumer warps alike), so the dispatcher's choices give the
    same bits: 128x128 with 8 warps (1), 192x128 (6), 128x128 with 16 warps
    (7, the row-major 128x128 choice)."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + N + K)
    outs = []
    g.set_option(gemm.GEMM_OPT_SPLIT_K, 1)
    try:
        for config in (1, 6, 7):
            g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, config)
            outs.append(run_gpu(g, A, B, layout, "f32").cpu())
    finally:
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, 0)
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("splits", [2, 3, 7])
def test_split_k_forced(g, oracle_mod, layout, splits):
    """K cut into slices whose partial products are summed in a second
    kernel ("GEMM 性能优化", 台阶 1): same tolerance, deterministic."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = 200, 333, 1000
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=61 + splits)
    g.set_option(gemm.GEMM_OPT_SPLIT_K, splits)
    try:
        C1 = run_gpu(g, A, B, layout, "f32").cpu()
        assert f"splitk{splits}" in g.last_path
        C2 = run_gpu(g, A, B, layout, "f32").cpu()
    finally:
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    assert torch.equal(C1, C2)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C1, Cr, S, TOL["f32"], f"split {splits}")


def test_split_k_integer_exact(g, oracle_mod):
    from dense_gemm_sm100_gb300 import gemm
    A, B = inp.make_integer_operands(150, 260, 900, seed=71)
    g.set_option(gemm.GEMM_OPT_SPLIT_K, 4)
    try:
        C = run_gpu(g, A, B, ROW, "f32")
        assert "splitk4" in g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    Cr, _ = oracle_of(oracle_mod, A, B, ROW)
    assert np.array_equal(to_f64(C), Cr)


def test_split_k_chosen_for_underfilled_shape(g):
    """1024^3 fills 64 of the SMs with 128x128 tiles: the K dimension is
    split, as stream-K (32 k-tiles of 64 tiles on 152 CTAs, 14 each) since
    that is shorter than two slices of 16."""
    A, B = inp.make_operands(1024, 1024, 1024, layout_b=COL, seed=1)
    run_gpu(g, A, B, COL, "f32")
    assert "+splitk" in g.last_path or "+streamk" in g.last_path, g.last_path


@pytest.mark.parametrize("stream_k", [1, 2])
@pytest.mark.parametrize("config,layout,M", [(1, ROW, 700), (1, COL, 700), (6, ROW, 500)])
def test_tail_tiles_split_along_k(g, oracle_mod, config, layout, M, stream_k):
    """Tiles of a partial last wave are cut along K and spread over all CTA
    slots, and a second kernel adds each tile's pieces in k order ("GEMM
    性能优化", Wave 模型): as equal slices per tile (stream_k 1) or as one
    equal, contiguous range of the tail's k-tiles per CTA that may cross
    tile boundaries (stream-K, 2).  An 8-CTA cap makes the wave small: 700
    rows x 650 columns in 128x128 tiles is 36 tiles = 4 waves + 4 tiles,
    500 rows in 192x128 tiles is 18 tiles = 2 waves + 2 tiles.  Same
    tolerance, deterministic, and exact on integer inputs."""
    from dense_gemm_sm100_gb300 import gemm
    N, K = 650, 640
    g.set_option(gemm.GEMM_OPT_MAX_CTAS, 8)
    g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, config)
    g.set_option(gemm.GEMM_OPT_STREAM_K, stream_k)
    try:
        A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + config)
        C1 = run_gpu(g, A, B, layout, "f32").cpu()
        assert ("+tail" if stream_k == 1 else "+streamk") in g.last_path, g.last_path
        C2 = run_gpu(g, A, B, layout, "f32").cpu()
        Ai, Bi = inp.make_integer_operands(M, N, K, layout_b=layout, seed=config)
        Ci = run_gpu(g, Ai, Bi, layout, "f32")
    finally:
        g.set_option(gemm.GEMM_OPT_MAX_CTAS, 0)
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, 0)
        g.set_option(gemm.GEMM_OPT_STREAM_K, 0)
    assert torch.equal(C1, C2)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C1, Cr, S, TOL["f32"], f"tail split config {config} stream_k {stream_k}")
    Cri, _ = oracle_of(oracle_mod, Ai, Bi, layout)
    assert np.array_equal(to_f64(Ci), Cri)


@pytest.mark.parametrize("config,layout,shape,max_ctas,elementwise", [
    (1, COL, (1024, 1024, 1024), 0, 0),  # 64 tiles, 2048 k-tiles on 152 CTAs: ranges cross tiles
    (6, COL, (1000, 900, 1000), 0, 0),   # 192x128, corner turn, ragged M, N and K
    (1, ROW, (700, 651, 640), 8, 0),     # N not a multiple of 4: element-wise C writes
    (1, ROW, (300, 520, 40), 8, 0),      # 2 k-tiles per tile: ranges of two tiles' pieces
    (1, ROW, (130, 130, 64), 0, 0),      # 8 k-tiles in all, fewer than the CTAs: most CTAs idle
    (4, ROW, (200, 300, 700), 16, 0),    # 64x64 tiles
    (6, ROW, (1000, 1000, 3000), 0, 0),  # 192x128, 48 tiles x 94 k-tiles: several pieces per tile
    (1, ROW, (333, 444, 555), 8, 1),     # element-wise producer: no stream-K form, slices instead
])
def test_stream_k_forced(g, oracle_mod, config, layout, shape, max_ctas, elementwise):
    """Stream-K forced on shapes whose tiles all fit in one wave: every CTA
    takes an equal range of the k-tiles, tile after tile, writes one partial
    tile per tile its range touches, and a second kernel adds each tile's
    partial tiles in k order.  Same tolerance, deterministic, exact on
    integer inputs.  The element-wise producer has no stream-K form and cuts
    the tiles into slices."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, config)
    g.set_option(gemm.GEMM_OPT_STREAM_K, 2)
    g.set_option(gemm.GEMM_OPT_MAX_CTAS, max_ctas)
    g.set_option(gemm.GEMM_OPT_ELEMENTWISE, elementwise)
    try:
        # K = 555: A's pitch of 2220 bytes is no multiple of 16, so TMA cannot
        # address A and the element-wise case copies it with cp.async
        A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + N + K)
        C1 = run_gpu(g, A, B, layout, "f32").cpu()
        if elementwise:
            assert "+cpasync" in g.last_path and "+tail" in g.last_path, g.last_path
        else:
            assert "+streamk" in g.last_path, g.last_path
        C2 = run_gpu(g, A, B, layout, "f32").cpu()
        Ai, Bi = inp.make_integer_operands(M, N, K, layout_b=layout, seed=K)
        Ci = run_gpu(g, Ai, Bi, layout, "f32")
    finally:
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, 0)
        g.set_option(gemm.GEMM_OPT_STREAM_K, 0)
        g.set_option(gemm.GEMM_OPT_MAX_CTAS, 0)
        g.set_option(gemm.GEMM_OPT_ELEMENTWISE, 0)
    assert torch.equal(C1, C2)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C1, Cr, S, TOL["f32"], f"stream-K {shape} config {config}")
    Cri, _ = oracle_of(oracle_mod, Ai, Bi, layout)
    assert np.array_equal(to_f64(Ci), Cri)


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("cluster_mode,shape,splits", [
    (1, (128, 600, 700), 3),     # one CTA per tile, ragged N and K
    (3, (300, 520, 640), 2),     # pair MMA, 3 tile rows: the odd CTA of the last pair is past M
    (3, (640, 512, 1000), 5),
])
def test_tc_split_k_forced(g, oracle_mod, mode, layout, cluster_mode, shape, splits):
    """Tensor-core K split: each tile unit in `splits` K slices whose partial
    tiles a second kernel adds in slice order.  Same tolerance,
    deterministic, exact on integer inputs."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    g.set_option(gemm.GEMM_OPT_TC_CLUSTER, cluster_mode)
    g.set_option(gemm.GEMM_OPT_SPLIT_K, splits)
    try:
        A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + N + splits, dtype=mode)
        C1 = run_gpu(g, A, B, layout, mode).cpu()
        stages = -(-K // (64 if mode == "bf16" else 32))  # 128-byte K stages
        per = -(-stages // splits)
        assert f"+splitk{-(-stages // per)}" in g.last_path, g.last_path  # no empty slice
        C2 = run_gpu(g, A, B, layout, mode).cpu()
        Ai, Bi = inp.make_integer_operands(M, N, K, layout_b=layout, seed=splits, dtype=mode)
        Ci = run_gpu(g, Ai, Bi, layout, mode)
    finally:
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
        g.set_option(gemm.GEMM_OPT_TC_CLUSTER, 3)
    assert torch.equal(C1, C2)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(C1, Cr, S, TOL[mode], f"tc split {splits} {mode} {shape}")
    Cri, _ = oracle_of(oracle_mod, Ai, Bi, layout)
    assert np.array_equal(to_f64(Ci), Cri)


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_tc_split_k_chosen_for_underfilled_shape(g, oracle_mod, mode):
    """128 x 2048 is 8 tiles of 128x256 on 152 SMs: the K split is chosen
    (a third of a wave or less)."""
    M, N, K = 128, 2048, 1024
    A, B = inp.make_operands(M, N, K, dist="normal", seed=9, dtype=mode)
    C = run_gpu(g, A, B, ROW, mode)
    assert "+splitk" in g.last_path, g.last_path
    Cr, S = oracle_of(oracle_mod, A, B, ROW)
    assert_parity(C, Cr, S, TOL[mode], f"tc chosen split {mode}")


# ------------------------------------------------------- the five workloads

def _sampled_check(g, oracle_mod, w, n_rows=40, n_cols=40):
    A, B = inp.make_workload(w)
    dev = torch.device("cuda", 0)
    A_d, B_d = A.to(dev), B.to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
    g.run(A_d, B_d, C, w.layout_b, w.dtype)
    g.sync_status()
    rows = inp.sample_indices(w.M, n_rows, seed=w.seed + 100)
    cols = inp.sample_indices(w.N, n_cols, seed=w.seed + 200)
    Cs = C[torch.tensor(rows, device=dev)][:, torch.tensor(cols, device=dev)]
    Cr, S = oracle_mod.gemm_sampled(to_f64(A), to_f64(B), rows, cols, w.layout_b)
    return assert_parity(Cs, Cr, S, TOL[w.dtype], w.name)


@pytest.mark.parametrize("name", ["fp32_128_row", "fp32_1024_colB"])
def test_workload_full(g, oracle_mod, name):
    w = inp.WORKLOADS[name]
    A, B = inp.make_workload(w)
    C = run_gpu(g, A, B, w.layout_b, w.dtype)
    Cr, S = oracle_of(oracle_mod, A, B, w.layout_b)
    assert_parity(C, Cr, S, TOL[w.dtype], name)


@pytest.mark.parametrize("elementwise", [1, 0])
def test_workload_ragged_4095x3073x2047(g, oracle_mod, elementwise):
    """Non-tile-multiple edges with tight (not 16-byte multiple) leading
    dimensions, through the element-wise producer and through re-packing:
    checked on every row in a band at each edge and a sample of the
    interior."""
    from dense_gemm_sm100_gb300 import gemm
    w = inp.WORKLOADS["fp32_4095x3073x2047_row"]
    A, B = inp.make_workload(w)
    g.set_option(gemm.GEMM_OPT_ELEMENTWISE, elementwise)
    try:
        C = run_gpu(g, A, B, w.layout_b, w.dtype)
    finally:
        g.set_option(gemm.GEMM_OPT_ELEMENTWISE, 0)
    if elementwise:
        assert "+cpasync" in g.last_path, g.last_path
    else:
        assert "repackA" in g.last_path and "repackB" in g.last_path
    rows = sorted(set(range(0, 130)) | set(range(w.M - 130, w.M)) |
                  set(inp.sample_indices(w.M, 64, seed=7)))
    cols = sorted(set(range(0, 260)) | set(range(w.N - 260, w.N)) |
                  set(inp.sample_indices(w.N, 64, seed=8)))
    Cr, S = oracle_mod.gemm_sampled(to_f64(A), to_f64(B), rows, cols, w.layout_b)
    assert_parity(C[rows][:, cols], Cr, S, TOL[w.dtype], w.name)


@pytest.mark.parametrize("name", ["fp32_8192_row", "ffn_bf16_8192x14336x4096",
                                  "ffn_tf32_8192x14336x4096"])
def test_workload_sampled(g, oracle_mod, name):
    _sampled_check(g, oracle_mod, inp.WORKLOADS[name])


def _odd_pitch(t, dev):
    """t on dev with a row pitch of cols + 1 elements (not a multiple of 16
    bytes), so the library re-packs it into the handle's workspace."""
    rows, cols = t.shape
    buf = torch.zeros((rows, cols + 1), dtype=t.dtype, device=dev)
    buf[:, :cols] = t.to(dev)
    return buf[:, :cols]


def test_workspace_grows_in_stream_order(oracle_mod):
    """A fresh handle's workspace grows while earlier calls that use it are
    still queued: small re-packed call, a larger one that must grow the
    workspace, and the small one again, back to back on one stream with no
    host synchronisation; then a larger call on a second stream ordered
    after the first by an event.  Every result matches the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import gemm
    dev = torch.device("cuda", 0)
    shapes = [(300, 260, 130), (1100, 900, 700), (300, 260, 130)]
    with gemm.Gemm(0) as h:
        h.set_option(gemm.GEMM_OPT_SIMT_SMALL, 1)  # the persistent kernels, whose operands get re-packed
        s1 = torch.cuda.Stream()
        ops, outs = [], []
        for i, (M, N, K) in enumerate(shapes):
            A, B = inp.make_integer_operands(M, N, K, seed=40 + i)
            ops.append((A, B))
            with torch.cuda.stream(s1):
                A_d, B_d = _odd_pitch(A, dev), _odd_pitch(B, dev)
                C = torch.full((M, N), float("nan"), device=dev)
                h.run(A_d, B_d, C, ROW, "f32", s1)
                outs.append((A_d, B_d, C))
        assert "+repackA" in h.last_path
        ev = torch.cuda.Event()
        ev.record(s1)
        s2 = torch.cuda.Stream()
        s2.wait_event(ev)
        M, N, K = 1500, 1300, 900
        A, B = inp.make_integer_operands(M, N, K, seed=49)
        ops.append((A, B))
        with torch.cuda.stream(s2):
            A_d, B_d = _odd_pitch(A, dev), _odd_pitch(B, dev)
            C = torch.full((M, N), float("nan"), device=dev)
            h.run(A_d, B_d, C, ROW, "f32", s2)
            outs.append((A_d, B_d, C))
        h.sync_status(s2)
        torch.cuda.synchronize()
    for (A, B), (_, _, C) in zip(ops, outs):
        Cr, _ = oracle_of(oracle_mod, A, B, ROW)
        assert np.array_equal(to_f64(C), Cr)


@pytest.mark.parametrize("mode,layout,shape", [
    ("f32", ROW, (128, 128, 128)),     # one kernel
    ("f32", COL, (1024, 1024, 1024)),  # re-pack-free stream-K: GEMM + dependent reduction kernel
    ("f32", ROW, (1301, 1257, 131)),   # unaligned pitches: re-pack kernels first
    ("bf16", ROW, (256, 512, 192)),    # tensor cores, pair MMA
])
def test_run_captures_in_a_cuda_graph(mode, layout, shape):
    """gemm_run only queues work on the caller's stream (no host waits), so
    a sequence of calls can be captured in a CUDA graph and replayed: the
    replay gives the same bits as the calls run directly.  A first direct
    call sizes the workspace, so nothing is allocated during the capture.
    A handle of its own: the graph refers to its workspace."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + 3 * N, dtype=mode)
    dev = torch.device("cuda", 0)
    A_d, B_d = A.to(dev), B.to(dev)
    h = gemm.Gemm(0)
    try:
        C_direct = torch.empty((M, N), dtype=torch.float32, device=dev)
        h.run(A_d, B_d, C_direct, layout, mode)
        h.sync_status()
        torch.cuda.synchronize()
        C_graph = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(3):
                    h.run(A_d, B_d, C_graph, layout, mode, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert torch.isnan(C_graph).all()  # captured, not run
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        h.sync_status()
        assert torch.equal(C_graph, C_direct)
        del graph
        torch.cuda.synchronize()
    finally:
        h.close()


SMALL_KERNEL_SHAPES = [(1, 1, 1), (3, 5, 7), (32, 32, 32), (33, 31, 65), (128, 128, 128), (100, 300, 1000),
                       (257, 129, 2049), (640, 96, 33)]


@pytest.mark.parametrize("layout", [ROW, COL])
@pytest.mark.parametrize("shape", SMALL_KERNEL_SHAPES)
@pytest.mark.parametrize("pitch_pad", [0, 1])
def test_small_kernel_matches_oracle(g, oracle_mod, layout, shape, pitch_pad):
    """The FP32 small-problem kernel (32 x 32 tiles, four K groups of 2 x 2
    outputs per thread, operands read in place at any pitch), forced on:
    ragged edges in every dimension, K past one chunk and past 1024, 16-byte
    and odd pitches.  Same tolerance as the other FP32 kernels, exact on
    integer inputs, and within the same tolerance of the persistent kernel
    without a K split (the two add an element's products in different
    orders)."""
    from dense_gemm_sm100_gb300 import gemm
    M, N, K = shape
    dev = torch.device("cuda", 0)

    def placed(t):
        if not pitch_pad:
            return t.to(dev)
        buf = torch.zeros((t.shape[0], t.shape[1] + pitch_pad), dtype=t.dtype, device=dev)
        buf[:, :t.shape[1]] = t.to(dev)
        return buf[:, :t.shape[1]]

    A, B = inp.make_operands(M, N, K, layout_b=layout, dist="normal", seed=M + N + K + pitch_pad)
    Ai, Bi = inp.make_integer_operands(M, N, K, layout_b=layout, seed=K + pitch_pad)
    outs = []
    g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 2)
    try:
        for (a, b) in ((A, B), (Ai, Bi)):
            C = torch.full((M, N), float("nan"), device=dev)
            g.run(placed(a), placed(b), C, layout, "f32")
            g.sync_status()
            assert "small32x32" in g.last_path, g.last_path
            outs.append(C.cpu())
        g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 1)
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 1)
        C_tile = torch.empty((M, N), device=dev)
        g.run(A.to(dev), B.to(dev), C_tile, layout, "f32")
        g.sync_status()
        assert "small" not in g.last_path, g.last_path
    finally:
        g.set_option(gemm.GEMM_OPT_SIMT_SMALL, 0)
        g.set_option(gemm.GEMM_OPT_SPLIT_K, 0)
    Cr, S = oracle_of(oracle_mod, A, B, layout)
    assert_parity(outs[0], Cr, S, TOL["f32"], f"small kernel {shape}")
    Cri, _ = oracle_of(oracle_mod, Ai, Bi, layout)
    assert np.array_equal(to_f64(outs[1]), Cri)
    assert_parity(C_tile.cpu(), Cr, S, TOL["f32"], f"persistent kernel {shape}")


def test_small_kernel_is_the_choice_for_a_few_tiles(g):
    """128^3 (C1) is 16 tiles of 32 x 32 with K = 128: the small-problem kernel;
    1024^3 (C2) is 1024 such tiles: the persistent kernels."""
    A, B = inp.make_operands(128, 128, 128, seed=0)
    run_gpu(g, A, B, ROW, "f32")
    assert "small32x32" in g.last_path, g.last_path
    A, B = inp.make_operands(1024, 1024, 1024, layout_b=COL, seed=1)
    run_gpu(g, A, B, COL, "f32")
    assert "small" not in g.last_path, g.last_path


def test_small_kernel_selection_bounds(g, oracle_mod):
    """The small-problem kernel is chosen for K <= 384 and at most one 32 x 32
    tile per SM, and not past either bound; GEMM_OPT_SIMT_CONFIG, MAX_CTAS
    and SPLIT_K keep it out, SIMT_SMALL 1 never and 2 always uses it.  Every
    run is checked against the oracle (exact on integer inputs)."""
    from dense_gemm_sm100_gb300 import gemm
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def path_of(M, N, K, opts=()):
        A, B = inp.make_integer_operands(M, N, K, layout_b=ROW, seed=M + N + K)
        for k, v in opts:
            g.set_option(k, v)
        try:
            C = run_gpu(g, A, B, ROW, "f32")
        finally:
            for k, _ in opts:
                g.set_option(k, 0)
        Cr, _ = oracle_of(oracle_mod, A, B, ROW)
        assert np.array_equal(to_f64(C.cpu()), Cr), (M, N, K, opts)
        return g.last_path

    assert "small32x32" in path_of(96, 64, 384)
    assert "small" not in path_of(96, 64, 385)
    assert "small32x32" in path_of(32, 32 * sms, 64)        # one tile per SM
    assert "small" not in path_of(32, 32 * sms + 1, 64)     # one tile more
    for opt, val in ((gemm.GEMM_OPT_SIMT_CONFIG, 4), (gemm.GEMM_OPT_MAX_CTAS, 8), (gemm.GEMM_OPT_SPLIT_K, 1),
                     (gemm.GEMM_OPT_SIMT_SMALL, 1)):
        assert "small" not in path_of(128, 128, 128, ((opt, val),)), opt
    assert "small32x32" in path_of(512, 512, 512, ((gemm.GEMM_OPT_SIMT_SMALL, 2),))
