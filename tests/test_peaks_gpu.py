"""The peak-rate microbenchmarks (include/gemm_peaks.h) on the GPU: they run
to completion without an expired wait and measure rates that are possible
for the unit they load.  The FP32 rate cannot exceed SMs x 128 lanes x 2
FLOP x the maximum SM clock (the FLOP count is what the kernel executes: no
chain may be folded away at compile time); tcgen05 BF16 is about twice
TF32."""
import subprocess

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


def max_sm_mhz():
    """The GPU's maximum SM clock as nvidia-smi reports it (None if unavailable)."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits",
                              "-i", "0"], capture_output=True, text=True, timeout=30).stdout.strip()
        return float(out.splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        return None


def test_fma_peaks(sms):
    from dense_gemm_sm100_gb300 import gemm
    mhz = max_sm_mhz() or 2070.0
    roof = sms * 128 * 2 * mhz * 1e6 / 1e12  # FP32 FMA peak at the maximum SM clock
    scalar = gemm.measure_peak("ffma", 16 * 8000)
    packed = gemm.measure_peak("ffma2", 16 * 8000)
    assert 0.5 * roof < scalar["tflops"] <= 1.01 * roof, (scalar, roof)
    assert 0.5 * roof < packed["tflops"] <= 1.01 * roof, (packed, roof)
    # 32 warps per SM of independent chains: close to one FMA per lane per cycle either way
    assert packed["tflops"] > 0.8 * scalar["tflops"]


def test_mma_peaks(sms):
    from dense_gemm_sm100_gb300 import gemm
    bf16 = gemm.measure_peak("mma_bf16", 4000)
    tf32 = gemm.measure_peak("mma_tf32", 4000)
    assert 300.0 < bf16["tflops"] < 3000.0
    assert 0.3 < tf32["tflops"] / bf16["tflops"] < 0.7
