"""The seeded input generator: reproducible, layout-independent values."""
import torch

from dense_gemm_sm100_gb300 import inputs as inp


def test_seeded_and_reproducible():
    a1, b1 = inp.make_operands(5, 7, 3, seed=11)
    a2, b2 = inp.make_operands(5, 7, 3, seed=11)
    a3, _ = inp.make_operands(5, 7, 3, seed=12)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    assert not torch.equal(a1, a3)


def test_col_major_stores_same_logical_matrix():
    a_r, b_r = inp.make_operands(4, 6, 5, layout_b=inp.B_ROW_MAJOR, seed=3)
    a_c, b_c = inp.make_operands(4, 6, 5, layout_b=inp.B_COL_MAJOR, seed=3)
    assert torch.equal(a_r, a_c)
    assert b_r.shape == (5, 6) and b_c.shape == (6, 5)
    assert torch.equal(b_r, b_c.t())


def test_distributions():
    a, b = inp.make_operands(256, 256, 256, dist="uniform", seed=0)
    assert a.min() >= -1 and a.max() < 1 and b.min() >= -1 and b.max() < 1
    a, _ = inp.make_operands(512, 8, 512, dist="normal", sigma=0.02, seed=4)
    assert abs(a.std().item() - 0.02) < 1e-3 and abs(a.mean().item()) < 1e-3


def test_bf16_is_rounded_fp32_draw():
    a32, b32 = inp.make_operands(8, 9, 10, dist="normal", sigma=0.02, seed=4)
    a16, b16 = inp.make_operands(8, 9, 10, dist="normal", sigma=0.02, seed=4, dtype=inp.BF16)
    assert a16.dtype == torch.bfloat16
    assert torch.equal(a16, a32.to(torch.bfloat16)) and torch.equal(b16, b32.to(torch.bfloat16))


def test_integer_operands_exact_in_all_types():
    a, b = inp.make_integer_operands(16, 16, 16, dtype=inp.BF16)
    assert torch.equal(a.float(), a.float().round()) and a.float().abs().max() <= 8


def test_workloads_match_their_specification():
    w = inp.WORKLOADS
    assert (w["fp32_8192_row"].M, w["fp32_8192_row"].seed) == (8192, 3)
    assert w["fp32_1024_colB"].layout_b == inp.B_COL_MAJOR
    f = w["ffn_bf16_8192x14336x4096"]
    assert (f.M, f.N, f.K, f.sigma, f.dtype) == (8192, 14336, 4096, 0.02, inp.BF16)
    assert w["fp32_4095x3073x2047_row"].dist == "normal"


def test_sample_indices_include_edges():
    idx = inp.sample_indices(1000, 10, seed=1)
    assert idx[0] == 0 and idx[-1] == 999 and len(idx) == 10 and idx == sorted(set(idx))
