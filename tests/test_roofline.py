"""The performance model against the values the pages print
(tests/golden/pages_traffic_model.txt, each line citing its page and section)."""
import os

import pytest

from dense_gemm_sm100_gb300 import roofline as rl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "pages_traffic_model.txt")


def load_golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, cite = line.split("|", 1)
        name, value = head.split()
        assert cite.strip(), f"{name} has no citation"
        vals[name] = float(value)
    return vals


G = load_golden()


def test_balance_point():
    bp = rl.balance_point(G["v100_fp32_peak_tflops"] * 1e12, G["v100_hbm_gbs"] * 1e9)
    assert round(bp, 1) == G["v100_balance_point_flop_per_byte"]


def test_wave_size():
    assert rl.wave_size(int(G["v100_sms"]), int(G["v100_blocks_per_sm"])) == G["v100_wave_blocks"]


def test_thread_tile_access_fraction():
    # shared-memory accesses per multiply-add scale with 1/TM + 1/TN; the
    # page's "down to 1/4" is that expression's value at TM = TN = 8
    frac = 1 / 8 + 1 / 8
    assert frac == pytest.approx(G["thread_tile_tm_tn_8_smem_access_fraction"])
    assert (128 // 8) * (128 // 8) == G["block_threads_for_128x128_tile_8x8_per_thread"]


def test_tiled_and_coarsened_intensity():
    assert rl.tiled_intensity(32) == pytest.approx(G["tiled_intensity_T32"])
    assert rl.coarsened_intensity(32, 4) == pytest.approx(G["coarsened_intensity_T32_CF4"])
    gain = rl.coarsened_intensity(32, 4) / rl.tiled_intensity(32) - 1
    assert gain == pytest.approx(G["coarsened_intensity_gain_T32_CF4"])


def test_intensity_from_load_counts():
    # the intensities must follow from the load counts: 2mnk flops / (4 B * loads)
    m, n, k, T, CF = 4096, 2048, 1024, 32, 4
    flops = rl.gemm_flops(m, n, k)
    assert flops / (4 * rl.tiled_loads_elements(m, n, k, T)) == pytest.approx(rl.tiled_intensity(T))
    assert flops / (4 * rl.coarsened_loads_elements(m, n, k, T, CF)) == pytest.approx(
        rl.coarsened_intensity(T, CF))


@pytest.mark.parametrize("cf", [1, 2, 4, 8])
def test_coarsening_saving(cf):
    assert rl.coarsening_saving(cf) == pytest.approx(G[f"coarsening_saving_CF{cf}"])
    m = n = k = 1024
    t = rl.tiled_loads_elements(m, n, k, 32)
    c = rl.coarsened_loads_elements(m, n, k, 32, cf)
    assert (t - c) / t == pytest.approx(rl.coarsening_saving(cf))


def test_saving_limit():
    assert rl.coarsening_saving(10 ** 9) == pytest.approx(G["coarsening_saving_limit"], abs=1e-8)


def test_tiled_traffic_reduces_to_pages_formula():
    # square T tiles, FP32, without the C write: 8·m·k·n / T bytes
    m, n, k, T = 512, 256, 128, 32
    got = rl.tiled_traffic_bytes(m, n, k, T, T, 4, 0)
    assert got == pytest.approx(8 * m * k * n / T)


def test_compulsory_and_flops():
    assert rl.gemm_flops(8192, 8192, 8192) == 1099511627776
    assert rl.compulsory_bytes(8192, 8192, 8192, 4) == 3 * 8192 * 8192 * 4
    assert rl.compulsory_bytes(8192, 14336, 4096, 2) == 2 * (8192 * 4096 + 4096 * 14336) + 4 * 8192 * 14336
    assert rl.tflops(1000, 1000, 500, 1e-3) == pytest.approx(1.0)


def test_fp32_peak_and_roofline():
    assert rl.fp32_simt_peak_tflops(152, 2070) == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    # tiny K makes the GEMM bandwidth-bound under the same peak
    low = rl.roofline_tflops(8192, 8192, 4, 80.0, 6760.6, 4)
    assert low < 80.0
    assert rl.roofline_tflops(8192, 8192, 8192, 80.0, 6760.6, 4) == 80.0


def test_wave_efficiency():
    assert rl.wave_efficiency(152, 152) == 1.0
    assert rl.wave_efficiency(153, 152) == pytest.approx(153 / 304)
    assert rl.waves(4096, 152) == pytest.approx(4096 / 152)
