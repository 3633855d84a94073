"""Work, traffic and roofline model of the GEMM (host-side arithmetic only).

The formulas restate the pages' analysis for this library's tiles:

* "GEMM 性能优化", 指标与目标: TFLOPS = 2·M·N·K / (t · 1e12).
* "GEMM 性能优化", Roofline 与平衡点: balance point = compute peak / memory
  bandwidth; below it a kernel is bandwidth-bound, above it compute-bound.
* "GEMM 性能优化", Wave 模型: a wave is the set of blocks resident at once,
  SMs × blocks per SM.
* "PMPP Chapter 06: Performance considerations", section 3 (Thread
  coarsening, global memory access analysis): a tiled kernel with square
  tiles of width T loads each element of the m×k input n/T times and each
  element of the k×n input m/T times, 8·m·k·n/T bytes in FP32, so its
  arithmetic intensity is T/4; coarsening the column direction by CF gives
  (m·k·n/T)·(1 + 1/CF) loads and intensity T/(2·(1 + 1/CF)).

``tiled_traffic_bytes`` generalises the last item to rectangular BM×BN tiles
and adds the one write of C.  ``tests/golden/pages_traffic_model.txt`` holds
the values the pages print for these formulas.
"""
from __future__ import annotations

# FP32 lanes per SM on the Blackwell SM (4 sub-partitions × 32 lanes); each
# lane retires one fused multiply-add (2 flops) per clock.
FP32_LANES_PER_SM = 128


def gemm_flops(M: int, N: int, K: int) -> int:
    """Algorithmic flops of C = A·B: one multiply and one add per (i, j, k)."""
    return 2 * M * N * K


def tflops(M: int, N: int, K: int, seconds: float) -> float:
    """The pages' metric: 2·M·N·K / (t · 1e12)."""
    return gemm_flops(M, N, K) / (seconds * 1e12)


def compulsory_bytes(M: int, N: int, K: int, ab_bytes: int, c_bytes: int = 4) -> int:
    """Bytes a GEMM must move at least: read A and B once, write C once."""
    return ab_bytes * (M * K + K * N) + c_bytes * M * N


def tiled_traffic_bytes(M: int, N: int, K: int, BM: int, BN: int,
                        ab_bytes: int = 4, c_bytes: int = 4) -> float:
    """Global->SM bytes of a kernel with BM×BN output tiles and no reuse
    across tiles: A is re-read N/BN times, B M/BM times, C written once."""
    return ab_bytes * M * N * K * (1.0 / BN + 1.0 / BM) + c_bytes * M * N


def tiled_loads_elements(m: int, n: int, k: int, T: int) -> float:
    """Elements loaded by the square-tiled kernel: 2·m·k·n / T."""
    return 2.0 * m * k * n / T


def coarsened_loads_elements(m: int, n: int, k: int, T: int, CF: int) -> float:
    """Elements loaded with column-direction coarsening: (m·k·n/T)(1 + 1/CF)."""
    return (m * k * n / T) * (1.0 + 1.0 / CF)


def tiled_intensity(T: int, elem_bytes: int = 4) -> float:
    """FLOP per byte of the square-tiled kernel: 2mnk / (es · 2mnk/T)."""
    return T / elem_bytes


def coarsened_intensity(T: int, CF: int, elem_bytes: int = 4) -> float:
    """FLOP per byte with coarsening: 2 / (es · (1 + 1/CF) / T)."""
    return 2.0 * T / (elem_bytes * (1.0 + 1.0 / CF))


def coarsening_saving(CF: int) -> float:
    """Fraction of the tiled kernel's loads that coarsening removes."""
    return 0.5 * (1.0 - 1.0 / CF)


def balance_point(peak_flops: float, bandwidth_bytes: float) -> float:
    """FLOP/byte at which compute and memory time are equal."""
    return peak_flops / bandwidth_bytes


def wave_size(sms: int, blocks_per_sm: int) -> int:
    """Blocks that run at once."""
    return sms * blocks_per_sm


def waves(tiles: int, sms: int, blocks_per_sm: int = 1) -> float:
    """Tiles divided by the wave size (fractional)."""
    return tiles / wave_size(sms, blocks_per_sm)


def wave_efficiency(tiles: int, sms: int, blocks_per_sm: int = 1) -> float:
    """Useful fraction of the last-wave-rounded schedule."""
    w = wave_size(sms, blocks_per_sm)
    full = -(-tiles // w)
    return tiles / (full * w) if tiles else 1.0


def fp32_simt_peak_tflops(sms: int, sm_mhz: float) -> float:
    """FP32 FMA peak: SMs × 128 lanes × 2 flops × clock."""
    return sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def roofline_tflops(M: int, N: int, K: int, peak_tflops: float, hbm_gbs: float,
                    ab_bytes: int, c_bytes: int = 4) -> float:
    """min(compute peak, arithmetic intensity × bandwidth) in TFLOP/s, with
    intensity taken over the compulsory bytes."""
    ai = gemm_flops(M, N, K) / compulsory_bytes(M, N, K, ab_bytes, c_bytes)
    return min(peak_tflops, ai * hbm_gbs * 1e9 / 1e12)
