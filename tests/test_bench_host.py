"""Host-side logic of bench.py, without a GPU: throughput aggregation over
ranks (two gloo processes on the CPU), peak selection and the clock parser."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ctx = {"rank": rank, "world": world, "local": rank}
    my_ms = [12.0, 20.0][rank]  # rank 1 is the slow one
    ms_all = bench.all_gather_max(ctx, my_ms)
    ms, value = bench.aggregate(ms_all, 1e12)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms_all": ms_all, "ms": ms, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_slowest_rank(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = json.load(open(tmp_path / "r0.json"))
    r1 = json.load(open(tmp_path / "r1.json"))
    assert r0 == r1
    assert r0["ms_all"] == [12.0, 20.0]
    assert r0["ms"] == 20.0
    # two replicas x 1e12 flops in 20 ms = 100 TFLOP/s
    assert r0["value"] == pytest.approx(100.0)


def test_single_rank_aggregation():
    ms, value = bench.aggregate([10.0], 2e12)
    assert ms == 10.0 and value == pytest.approx(200.0)


def test_tensor_peak_scaling():
    peaks = {"hbm_gbs": 1.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1600.0,
             "sm_max_mhz": 2000.0}
    assert bench.tensor_peak("bf16", peaks) == 1800.0
    assert bench.tensor_peak("tf32", peaks) == pytest.approx(1800.0 * 1.1 / 2.25)
    assert bench.tensor_peak("bf16", peaks, sustained=True) == 1600.0


def test_roofline_entry_fraction():
    r = bench.roofline_entry("alu", 40.0, 80.0, "TFLOP/s", None, "x")
    assert r["frac"] == 0.5 and r["bound"] == "alu" and r["traffic"] is None


def test_clock_summary_filters_window(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "c.csv")
    with open(s.path, "w") as f:
        f.write("2026/12/02 10:00:00.100, 0, 1500, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("2026/12/02 10:00:01.100, 0, 1900, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("2026/12/02 10:00:01.300, 0, 1950, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active\n")
    import time
    t0 = time.mktime(time.strptime("2026/12/02 10:00:01", "%Y/%m/%d %H:%M:%S"))
    out = s.summary(t0, t0 + 1.0)
    assert out["samples"] == 2 and out["sm_mhz"] == 1925 and out["reasons"] == ["sw_power_cap"]


def test_ncu_summary_table_from_raw_csv():
    """The ncu summary turns `ncu -i ... --page raw --csv` text into a
    Markdown table: labelled metrics with units, missing metrics skipped,
    stall reasons sorted by their per-instruction weight."""
    import bench
    csv_text = (
        '"ID","Kernel Name","gpu__time_duration.sum","sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active",'
        '"launch__registers_per_thread","smsp__average_warps_issue_stalled_wait_per_issue_active.ratio",'
        '"smsp__average_warps_issue_stalled_math_pipe_throttle_per_issue_active.ratio"\n'
        '"","","ms","%","register/thread","inst","inst"\n'
        '"0","sgemm_simt_kernel","1.83","83.6","128","1.13","2.10"\n')
    md = bench.ncu_summary_markdown(csv_text)
    lines = md.splitlines()
    assert lines[0] == "| metric | `sgemm_simt_kernel` |"
    assert "| duration | 1.83 ms |" in lines
    assert "| FMA pipe busy (% of active) | 83.6 % |" in lines
    assert "| registers / thread | 128 register/thread |" in lines
    assert not any(l.startswith("| tensor pipe") for l in lines)  # not in the report
    assert lines[-1].startswith("| top stalls per issued instruction (sgemm_simt_kernel) | math_pipe_throttle 2.10, wait 1.13")


def test_tensor_modes_are_described_and_peaked():
    """Every tensor-core mode the benchmark runs is a known workload with a
    description, and its peak is the measured BF16 burst scaled by the nominal
    rate of its input type: TF32 = 1.1/2.25 of BF16, and the FP32-accurate
    mode (three TF32 products per FP32 product) a third of TF32."""
    from dense_gemm_sm100_gb300 import inputs
    peaks = dict(bench.FALLBACK)
    for name in bench.TC_WORKLOADS:
        assert name in inputs.ALL_WORKLOADS and name in bench.DESCRIPTIONS
        assert inputs.ALL_WORKLOADS[name].dtype in bench.NOMINAL_PF
    bf16 = bench.tensor_peak("bf16", peaks)
    assert bf16 == peaks["bf16_tflops"]
    assert abs(bench.tensor_peak("tf32", peaks) - bf16 * 1.1 / 2.25) < 1e-9
    assert abs(bench.tensor_peak("f32x3", peaks) - bench.tensor_peak("tf32", peaks) / 3) < 1e-9
    w = inputs.ALL_WORKLOADS["fp32x3_8192_row"]
    ref = inputs.WORKLOADS["fp32_8192_row"]
    assert (w.M, w.N, w.K, w.layout_b, w.dist, w.seed) == (ref.M, ref.N, ref.K, ref.layout_b, ref.dist, ref.seed)


def test_every_specified_workload_is_a_bench_mode():
    """The default bench line covers every specified workload: the headline
    FP32 8192^3 case as `value`, and the other four (128^3, 1024^3 with
    column-major B, 4095x3073x2047, and the FFN shape in BF16 and TF32) under
    `modes`, each described; a mode's minimum step count is what it records."""
    from dense_gemm_sm100_gb300 import inputs
    covered = {bench.DEFAULT_WORKLOAD, *bench.TC_WORKLOADS, *bench.SIMT_WORKLOADS}
    assert set(inputs.WORKLOADS) <= covered
    for name in bench.SIMT_WORKLOADS:
        assert name in bench.DESCRIPTIONS and inputs.ALL_WORKLOADS[name].dtype == "f32"
    assert all(v >= 1 for v in bench.MIN_MODE_STEPS.values())
