"""The peak-rate microbenchmarks (include/gemm_peaks.h) on the GPU: they run
to completion without an expired wait and measure rates that are plausible
for the unit they load (FP32 CUDA cores: SMs x 128 lanes x 2 FLOP per cycle;
tcgen05: BF16 about twice TF32)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sms():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_sm100_gb300 import build
    build.build()
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_fma_peaks(sms):
    from dense_gemm_sm100_gb300 import gemm
    roof_2ghz = sms * 128 * 2 * 2.2e9 / 1e12  # above any SM clock of this GPU
    scalar = gemm.measure_peak("ffma", 16 * 2000)
    packed = gemm.measure_peak("ffma2", 16 * 2000)
    assert 0.2 * roof_2ghz < scalar["tflops"] < roof_2ghz
    assert 0.2 * roof_2ghz < packed["tflops"] < roof_2ghz
    # 32 warps per SM of independent chains: close to one FMA per lane per cycle either way
    assert packed["tflops"] > 0.8 * scalar["tflops"]


def test_mma_peaks(sms):
    from dense_gemm_sm100_gb300 import gemm
    bf16 = gemm.measure_peak("mma_bf16", 4000)
    tf32 = gemm.measure_peak("mma_tf32", 4000)
    assert 300.0 < bf16["tflops"] < 3000.0
    assert 0.3 < tf32["tflops"] / bf16["tflops"] < 0.7
