"""Benchmark of the GB300 GEMM library: TFLOPS = 2MNK/t and roofline fraction.

Default workload: FP32 SIMT GEMM, M = N = K = 8192, A, B, C row-major, values
U[-1, 1) from seed 3 (the SIMT headline case).  The same run also measures,
under "modes", every other specified workload: the tensor-core headline case
(FFN-shaped M=8192, N=14336, K=4096, N(0, 0.02) from seed 4, BF16 and TF32
inputs, FP32 C), the FP32 cases 128^3, 1024^3 with column-major B and
4095x3073x2047, and the extra FP32-accurate tensor-core mode; each mode
records the steps and warm-up steps it ran.

One step = one gemm_run of the whole workload through the C ABI with inputs
resident in HBM.  Inputs are larger than L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the FP64 CPU oracle (the only reference this project
has) on a bounded sample of the same workload on the host cores.  Under
torchrun (N > 1) each rank runs an independent replica on its own GPU
("scaling": "weak"); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2MNK/t) and % of GB300 FP32-SIMT / tensor-core roofline"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "fp32_8192_row"
TC_WORKLOADS = ["ffn_bf16_8192x14336x4096", "ffn_tf32_8192x14336x4096", "fp32x3_8192_row"]
# Bursts in which a workload's timed steps alternate with the cuBLAS side
# reference's (same count), when the side reference is measured.
SIDE_ROUNDS = 5
# The other specified FP32 workloads, measured under "modes" too.
SIMT_WORKLOADS = ["fp32_128_row", "fp32_1024_colB", "fp32_4095x3073x2047_row"]
# Launch-bound workloads: also timed as calls captured in a CUDA graph and
# replayed (this library and the cuBLAS side reference alike), which takes
# the per-call host and launch cost out of the time.
GRAPH_WORKLOADS = ["fp32_128_row", "fp32_1024_colB"]
GRAPH_CALLS, GRAPH_REPLAYS = 20, 10
# Modes whose step is short run at least this many timed steps (recorded in
# the mode's "steps"): the tensor-core modes reach their steady power state,
# and the microsecond-scale FP32 cases get a stable mean.
MIN_MODE_STEPS = {"ffn_bf16_8192x14336x4096": 200, "ffn_tf32_8192x14336x4096": 200,
                  "fp32x3_8192_row": 100, "fp32_128_row": 200, "fp32_1024_colB": 200}

# Fallback peaks (one earlier GB300 measurement) if MEASURED_PEAKS.json is absent.
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}
# Nominal dense tensor rates (PFLOP/s) used only to scale the measured BF16 peak
# to TF32: a contraction is compared with the peak of its own input type.
NOMINAL_PF = {"bf16": 2.25, "tf32": 1.1, "f32x3": 1.1 / 3}  # f32x3: three TF32 products per FP32 one

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the kernel as it is now; absent (reported as null) until
# captured for this version of the kernel.
# Key: workload name -> (bytes per launch, summary file under profiles/).
NCU_TRAFFIC: dict[str, tuple[float, str]] = {
    "fp32_8192_row": (2836.4e6 + 267.4e6, "profiles/dram_traffic_per_kernel.md"),
    "fp32_4095x3073x2047_row": (61.0e6 + 22.1e6, "profiles/dram_traffic_per_kernel.md"),
    "ffn_bf16_8192x14336x4096": (467.1e6 + 435.8e6, "profiles/dram_traffic_per_kernel.md"),
    "ffn_tf32_8192x14336x4096": (1806.8e6 + 448.1e6, "profiles/dram_traffic_per_kernel.md"),
    # the dominant kernel of the mode: the TF32 product over 3K
    "fp32x3_8192_row": (10363.2e6 + 262.5e6, "profiles/dram_traffic_per_kernel.md"),
}

DESCRIPTIONS = {
    "fp32_8192_row": "FP32 SIMT GEMM M=N=K=8192, A/B/C row-major, U[-1,1) seed 3",
    "ffn_bf16_8192x14336x4096": "tensor-core GEMM, BF16 A/B, FP32 C, M=8192 N=14336 K=4096, N(0,0.02) seed 4",
    "ffn_tf32_8192x14336x4096": "tensor-core GEMM, TF32 (FP32 storage), FP32 C, M=8192 N=14336 K=4096, N(0,0.02) seed 4",
    "fp32x3_8192_row": "FP32-accurate tensor-core GEMM (three TF32 products of split operands), M=N=K=8192, "
                       "A/B/C row-major, U[-1,1) seed 3 (the FP32 workload's operands)",
    "fp32_1024_colB": "FP32 SIMT GEMM M=N=K=1024, B column-major, U[-1,1) seed 1",
    "fp32_4095x3073x2047_row": "FP32 SIMT GEMM M=4095 N=3073 K=2047, row-major, N(0,1) seed 2",
    "fp32_128_row": "FP32 SIMT GEMM M=N=K=128, row-major, U[-1,1) seed 0",
    "fp32_4096_row": "FP32 SIMT GEMM M=N=K=4096, row-major, U[-1,1) seed 3 (profiling size)",
    "fp32_3648x4096x4096_row": "FP32 SIMT GEMM M=3648 N=K=4096, row-major, U[-1,1) seed 3 "
                               "(profiling size: whole waves of 192x128 tiles)",
    "ffn_bf16_4096x7168x4096": "tensor-core GEMM, BF16, M=4096 N=7168 K=4096 (profiling size)",
    "ffn_tf32_4096x7168x4096": "tensor-core GEMM, TF32, M=4096 N=7168 K=4096 (profiling size)",
}


# ---------------------------------------------------------------- host logic

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, ValueError, KeyError):
        return dict(FALLBACK), "fallback"


def tensor_peak(dtype: str, peaks: dict, sustained: bool = False) -> float:
    bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return bf16 * NOMINAL_PF[dtype] / NOMINAL_PF["bf16"]


def roofline_entry(bound, achieved, peak, unit, traffic, note):
    return {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 3),
            "unit": unit, "frac": round(achieved / peak, 4) if peak else None,
            "traffic": traffic, "peak_source": note}


def measure_peaks(dev_index=0, max_mhz=None):
    """The compute roofs measured on this GPU by the library's own
    microbenchmarks (include/gemm_peaks.h), each launch ~20-50 ms, best of 3,
    with the SM clock sampled while they ran: the FP32 readings are also
    given scaled to the maximum clock (rate x max MHz / median MHz), which
    can never exceed SMs x 128 x 2 x the maximum clock."""
    from dense_gemm_sm100_gb300 import gemm
    out = {}
    sampler = ClockSampler(dev_index)
    sampler.start()
    t0 = time.time()
    for kind, iters in (("ffma", 320000), ("ffma2", 320000), ("mma_bf16", 64000), ("mma_tf32", 64000)):
        r = gemm.measure_peak(kind, iters)
        out[f"{kind}_tflops"] = round(r["tflops"], 2)
        if kind == "ffma2":
            t_fma = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t_fma)
    if clocks and clocks.get("sm_mhz") and max_mhz:
        out["fma_clocks"] = clocks
        for kind in ("ffma", "ffma2"):
            out[f"{kind}_tflops_at_max_clock"] = round(out[f"{kind}_tflops"] * max_mhz / clocks["sm_mhz"], 2)
    out["what"] = ("FP32 multiply-adds on the CUDA cores, scalar and packed pairs (32 warps/SM of "
                   "independent chains); tcgen05 MMA 128x256 from shared memory into tensor memory, "
                   "one CTA per SM, no copies")
    return out


def add_microbench(roof, peak):
    """Beside the contract's peak: the same kernel against the microbenchmark roof."""
    if roof is None or not peak:
        return
    roof["peak_microbench"] = peak
    roof["frac_of_microbench"] = round(roof["achieved"] / peak, 4)


def aggregate(ms_per_rank, flops_per_rank_step):
    """Whole-job throughput over ranks: total work / slowest rank's time."""
    ms = max(ms_per_rank)
    total = flops_per_rank_step * len(ms_per_rank)
    return ms, total / (ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, kept only
    for the wall-clock window [t0, t1] of the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        deadline = time.time() + 10
        while time.time() < deadline and os.path.getsize(self.path) == 0:
            time.sleep(0.05)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[4], parts[5:]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows[-3:]
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4][1:5]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "samples": len(inside), "reasons": reasons}


# ---------------------------------------------------------------- GPU timing

def graph_us_per_call(fn, calls=GRAPH_CALLS, replays=GRAPH_REPLAYS):
    """Capture `calls` calls of fn (which queues its work on the current
    stream) in a CUDA graph, replay it, and return the device time per call
    in microseconds (CUDA events around the replays)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(calls):
                fn()
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (replays * calls)
    del graph
    torch.cuda.synchronize()
    return us


def time_device(run, stream, steps, warmup, counter=None):
    """Run `warmup` untimed steps, then `steps` timed steps with a CUDA event
    pair around each launch on `stream`.  Returns (total ms, per-step ms,
    kernels launched in the timed region according to `counter`)."""
    import torch
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    c0 = counter() if counter else 0
    for i in range(steps):
        starts[i].record(stream)
        run()
        ends[i].record(stream)
    c1 = counter() if counter else 0
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return starts[0].elapsed_time(ends[-1]), per, c1 - c0


L2_BYTES = 129e6


def l2_note(res) -> str:
    """How the timed steps relate to the L2 cache (no flush between steps)."""
    es = 2 if res["dtype"] == "bf16" else 4
    total = es * (res["M"] * res["K"] + res["K"] * res["N"]) + 4 * res["M"] * res["N"]
    mib = total / 2**20
    if total > L2_BYTES:
        return f"inputs larger than L2 (A, B, C {mib:.0f} MiB vs 129 MB L2); no flush"
    return f"A, B, C ({mib:.1f} MiB) fit in the 129 MB L2: warm-L2 steps, no flush"


def bench_workload(g, name, steps, warmup, dist_ctx, peaks, peak_note, with_e2e, side_cublas=False):
    import torch
    from dense_gemm_sm100_gb300 import inputs as inp
    from dense_gemm_sm100_gb300 import roofline as rl

    w = inp.ALL_WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    A, B = inp.make_workload(w)
    A_d, B_d = A.to(dev), B.to(dev)
    C_d = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def run():
        g.run(A_d, B_d, C_d, w.layout_b, w.dtype, stream)

    cub = None
    if side_cublas:
        # Labelled side reference: cuBLAS through torch on the same operands.
        # Never part of this library's path.  Its steps are interleaved with
        # this library's in SIDE_ROUNDS bursts, so both see the same power
        # and thermal state (timed one after the other, the second one ran
        # in a hotter GPU and the comparison depended on the order).
        torch.backends.cuda.matmul.allow_tf32 = w.dtype == "tf32"
        Bl = B_d if w.layout_b == 0 else B_d.t()
        cub_fn, cub_what = cublas_side_call(A_d, Bl, w.dtype)
    barrier(dist_ctx)
    t0 = time.time()
    if side_cublas:
        per_round = max(1, steps // SIDE_ROUNDS)
        steps = per_round * SIDE_ROUNDS
        for _ in range(warmup):
            cub_fn()
        total_ms, per, launches, cub_ms = 0.0, [], 0, 0.0
        for r in range(SIDE_ROUNDS):
            tm, pr, ln = time_device(run, stream, per_round, warmup if r == 0 else 0, lambda: g.launch_count)
            total_ms, per, launches = total_ms + tm, per + pr, launches + ln
            ctm, _, _ = time_device(cub_fn, stream, per_round, 0)
            cub_ms += ctm
        torch.backends.cuda.matmul.allow_tf32 = False
        cub = {"tflops": w.flops / (cub_ms / steps * 1e-3) / 1e12,
               "what": "cuBLAS through torch on the same operands; " + cub_what,
               "steps": steps, "interleaved_rounds": SIDE_ROUNDS}
    else:
        total_ms, per, launches = time_device(run, stream, steps, warmup, lambda: g.launch_count)
    t1 = time.time()
    g.sync_status(stream)
    barrier(dist_ctx)
    ms_step = total_ms / steps
    ms_all = all_gather_max(dist_ctx, ms_step)
    ms_max, value = aggregate(ms_all, w.flops)
    kernel_ms = statistics.mean(per)
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    es = 2 if w.dtype == "bf16" else 4
    if w.dtype == "f32":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = rl.fp32_simt_peak_tflops(sms, peaks["sm_max_mhz"])
        roof = roofline_entry("alu", achieved, peak, UNIT, NCU_TRAFFIC.get(name, (None,))[0],
                              f"derived: {sms} SMs x 128 FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz")
    else:
        peak = tensor_peak(w.dtype, peaks)
        note = f"{peak_note} cuBLAS BF16 burst" + {
            "bf16": "", "tf32": " x 1.1/2.25 (nominal TF32/BF16)",
            "f32x3": " x 1.1/2.25 / 3 (nominal TF32/BF16, three TF32 products per FP32 product)"}[w.dtype]
        roof = roofline_entry("tensor", achieved, peak, UNIT, NCU_TRAFFIC.get(name, (None,))[0], note)
    res = {
        "workload": name, "description": DESCRIPTIONS.get(name, name),
        "M": w.M, "N": w.N, "K": w.K, "layout_b": "row" if w.layout_b == 0 else "col",
        "dtype": w.dtype, "value": value, "ms_per_step": ms_max, "kernel_ms": kernel_ms,
        "kernel_ms_min": min(per), "kernel_ms_median": statistics.median(per),
        "path": g.last_path, "roofline": roof, "steps": steps,
        "launches_timed": launches, "wall_window": (t0, t1),
        "compulsory_bytes": rl.compulsory_bytes(w.M, w.N, w.K, es),
    }
    if cub is not None:
        res["cublas_side"] = cub
    if name in GRAPH_WORKLOADS:
        def run_current():
            g.run(A_d, B_d, C_d, w.layout_b, w.dtype, torch.cuda.current_stream())
        us = graph_us_per_call(run_current)
        res["graph"] = {"us_per_call": us, "tflops": w.flops / (us * 1e-6) / 1e12,
                        "calls_per_graph": GRAPH_CALLS, "replays": GRAPH_REPLAYS}
        if side_cublas:
            Bl = B_d if w.layout_b == 0 else B_d.t()
            cub_fn, _ = cublas_side_call(A_d, Bl, w.dtype)
            torch.backends.cuda.matmul.allow_tf32 = w.dtype == "tf32"
            cus = graph_us_per_call(cub_fn)
            torch.backends.cuda.matmul.allow_tf32 = False
            res["graph"]["cublas_us_per_call"] = cus
            res["graph"]["cublas_tflops"] = w.flops / (cus * 1e-6) / 1e12
    if with_e2e:
        Ah = A.pin_memory()
        Bh = B.pin_memory()
        Ch = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()

        def run_host():
            g.run_host(Ah, Bh, Ch, w.layout_b, w.dtype, stream)

        e2e_ms, _, _ = time_device(run_host, stream, steps, warmup)
        g.sync_status(stream)
        e2e_ms_all = all_gather_max(dist_ctx, e2e_ms / steps)
        _, e2e_value = aggregate(e2e_ms_all, w.flops)
        res["e2e"] = {"value": e2e_value, "unit": UNIT,
                      "h2d_bytes_per_step": A.numel() * A.element_size() + B.numel() * B.element_size(),
                      "d2h_bytes_per_step": w.M * w.N * 4,
                      "ms_per_step": max(e2e_ms_all), "steps": steps, "warmup": warmup,
                      "path": g.last_path}
    del A_d, B_d, C_d
    torch.cuda.empty_cache()
    return res


def cublas_side_call(A_d, B_view, dtype):
    """The labelled cuBLAS side reference for one workload: a callable and
    what it computes.  BF16 inputs ask for FP32 output (torch.mm out_dtype),
    as this library writes; without that overload, BF16 output, said so."""
    import torch
    if dtype == "bf16":
        try:
            torch.mm(A_d[:8, :8], B_view[:8, :8], out_dtype=torch.float32)
            return (lambda: torch.mm(A_d, B_view, out_dtype=torch.float32)), "BF16 inputs, FP32 output"
        except (TypeError, RuntimeError):
            return (lambda: torch.matmul(A_d, B_view)), "BF16 inputs, BF16 output (no FP32-output overload)"
    what = "TF32 math allowed, FP32 output" if dtype == "tf32" else "FP32, TF32 disallowed"
    return (lambda: torch.matmul(A_d, B_view)), what


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(name, target_s):
    """Time the FP64 oracle on a row sample of the workload sized to take
    about target_s seconds; returns (TFLOP/s, seconds, rows, threads)."""
    import oracle
    from dense_gemm_sm100_gb300 import inputs as inp
    w = inp.ALL_WORKLOADS[name]
    A, B = inp.make_workload(w)
    A64 = A.double().numpy()
    B64 = B.double().numpy()
    threads = oracle.default_threads()
    rows = max(1, min(w.M, threads))
    t = time.perf_counter()
    oracle.gemm(A64[:rows], B64, w.layout_b)
    dt = time.perf_counter() - t
    rows = int(max(1, min(w.M, rows * target_s / max(dt, 1e-3))))
    return A64, B64, w, rows, threads


def time_oracle(A64, B64, w, rows):
    import oracle
    t = time.perf_counter()
    oracle.gemm(A64[:rows], B64, w.layout_b)
    dt = time.perf_counter() - t
    return 2.0 * rows * w.N * w.K / dt / 1e12, dt


# ---------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return None
    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return {"rank": dist.get_rank(), "world": dist.get_world_size(), "local": local}


def barrier(ctx):
    if ctx is not None:
        import torch.distributed as dist
        dist.barrier()


def all_gather_max(ctx, value: float):
    """Every rank's value (list), for max-over-ranks timing."""
    if ctx is None:
        return [value]
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(ctx["world"])]
    dist.all_gather(out, t)
    return [float(x.item()) for x in out]


# ---------------------------------------------------------------- ladder

# "GEMM 性能优化", 八个台阶: each step's share of cuBLAS on the page's (V100)
# hardware, as ranges in percent.  Context for the GB300 measurements.
PAGES_LADDER_PCT = {1: (6, 11), 2: (25, 40), 3: (50, 65), 4: (60, 75), 5: (70, 80),
                    6: (80, 87), 7: (90, 97)}


NCU_SUMMARY_METRICS = [
    ("duration", "gpu__time_duration.sum"),
    ("SM clock", "sm__cycles_elapsed.avg.per_second"),
    ("FMA pipe busy (% of active)", "sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active"),
    ("tensor pipe busy (% of active)", "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"),
    ("issue active (%)", "smsp__issue_active.avg.pct_of_peak_sustained_active"),
    ("DRAM read", "dram__bytes_read.sum"),
    ("DRAM write", "dram__bytes_write.sum"),
    ("L2 hit rate", "lts__t_sector_hit_rate.pct"),
    ("L2 -> SM bytes", "l1tex__m_xbar2l1tex_read_bytes.sum"),
    ("shared-load bank conflicts", "l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_ld.sum"),
    ("registers / thread", "launch__registers_per_thread"),
    ("warps active (% of peak)", "sm__warps_active.avg.pct_of_peak_sustained_active"),
    ("grid", "launch__grid_size"),
    ("block", "launch__block_size"),
    ("dynamic shared memory", "launch__shared_mem_per_block_dynamic"),
]
STALL_PREFIX = "smsp__average_warps_issue_stalled_"
STALL_SUFFIX = "_per_issue_active.ratio"


def ncu_summary_markdown(csv_text: str, top_stalls: int = 5) -> str:
    """Markdown table of the usual metrics, one column per captured launch,
    from `ncu -i REPORT --page raw --csv` output (rows: header, units, one
    row per launch).  Metrics the report lacks are skipped."""
    import csv
    import io
    rows = [r for r in csv.reader(io.StringIO(csv_text)) if r]
    head, units, launches = rows[0], rows[1], rows[2:]
    col = {name: i for i, name in enumerate(head)}
    names = [r[col["Kernel Name"]][:60] if "Kernel Name" in col else f"launch {j}"
             for j, r in enumerate(launches)]
    out = ["| metric | " + " | ".join(f"`{n}`" for n in names) + " |",
           "|---|" + "---|" * len(launches)]
    for label, metric in NCU_SUMMARY_METRICS:
        if metric in col:
            i = col[metric]
            out.append(f"| {label} | " + " | ".join(f"{r[i]} {units[i]}".strip() for r in launches) + " |")
    stalls = [(name[len(STALL_PREFIX):-len(STALL_SUFFIX)], i) for name, i in col.items()
              if name.startswith(STALL_PREFIX) and name.endswith(STALL_SUFFIX)]
    for j, r in enumerate(launches):
        vals = []
        for stall, i in stalls:
            try:
                vals.append((float(r[i].replace(",", "")), stall))
            except ValueError:
                pass
        vals.sort(reverse=True)
        top = ", ".join(f"{s} {v:.2f}" for v, s in vals[:top_stalls])
        out.append(f"| top stalls per issued instruction ({names[j]}) | {top} |" + " |" * (len(launches) - 1))
    return "\n".join(out) + "\n"


def run_ncu_summary(path):
    import subprocess
    r = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True, text=True)
    if r.returncode != 0:
        print(r.stderr, file=sys.stderr)
        return r.returncode
    print(ncu_summary_markdown(r.stdout), end="")
    return 0


def apply_options(g, args):
    from dense_gemm_sm100_gb300 import gemm
    if args.simt_config:
        g.set_option(gemm.GEMM_OPT_SIMT_CONFIG, args.simt_config)
    if args.tc_mode:
        g.set_option(gemm.GEMM_OPT_TC_CLUSTER, args.tc_mode)
    if args.split_k:
        g.set_option(gemm.GEMM_OPT_SPLIT_K, args.split_k)
    if args.tc_group_m:
        g.set_option(gemm.GEMM_OPT_TC_GROUP_M, args.tc_group_m)
    if args.simt_group_m:
        g.set_option(gemm.GEMM_OPT_SIMT_GROUP_M, args.simt_group_m)


def run_configs(args):
    """Every workload of the specification, timed two ways: warm (back-to-back
    steps) and with the L2 scrubbed before each step (a 2 x L2 buffer written
    between the event pairs, outside the timed region), median and min of the
    per-step CUDA-event times; then the oracle on the two small cases with one
    host thread and with all of them.  One JSON document."""
    import torch
    import oracle
    from dense_gemm_sm100_gb300 import gemm
    from dense_gemm_sm100_gb300 import inputs as inp
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    steps = max(5, min(args.steps, 30))
    scrub = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
    g = gemm.Gemm(0)
    apply_options(g, args)
    done = {}
    if args.results and os.path.exists(args.results):
        for line in open(args.results):
            if line.strip():
                r = json.loads(line)
                done[r["workload"]] = r
    out = []
    small_c = {}
    for name, w in inp.WORKLOADS.items():
        if name in done:  # resume: measured by an earlier run
            out.append(done[name])
            continue
        A, B = inp.make_workload(w)
        A_d, B_d = A.to(dev), B.to(dev)
        C_d = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)

        def run():
            g.run(A_d, B_d, C_d, w.layout_b, w.dtype, stream)

        _, warm, _ = time_device(run, stream, steps, args.warmup)
        path = g.last_path
        for _ in range(args.warmup):
            run()
        cold = []
        for _ in range(steps):
            scrub.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            e1.synchronize()
            cold.append(e0.elapsed_time(e1))
        g.sync_status(stream)
        if name in ("fp32_128_row", "fp32_1024_colB"):
            small_c[name] = C_d.double().cpu().numpy()
        # labelled side reference: cuBLAS through torch on the same operands
        torch.backends.cuda.matmul.allow_tf32 = w.dtype == "tf32"
        Bl = B_d if w.layout_b == 0 else B_d.t()
        cub_fn, cub_what = cublas_side_call(A_d, Bl, w.dtype)
        _, cub, _ = time_device(cub_fn, stream, steps, args.warmup)
        torch.backends.cuda.matmul.allow_tf32 = False
        tf = lambda ms: round(w.flops / (ms * 1e-3) / 1e12, 3)
        out.append({"workload": name, "description": DESCRIPTIONS.get(name, name), "dtype": w.dtype,
                    "path": path, "steps": steps,
                    "warm": {"ms_median": statistics.median(warm), "ms_min": min(warm),
                             "tflops_median": tf(statistics.median(warm)), "tflops_max": tf(min(warm))},
                    "l2_scrubbed": {"ms_median": statistics.median(cold), "ms_min": min(cold),
                                    "tflops_median": tf(statistics.median(cold)),
                                    "tflops_max": tf(min(cold))},
                    "cublas_side": {"tflops_median": tf(statistics.median(cub)),
                                    "what": "cuBLAS through torch, warm, " + cub_what}})
        if args.results:
            with open(args.results, "a") as f:
                f.write(json.dumps(out[-1]) + "\n")
        del A_d, B_d, C_d
        torch.cuda.empty_cache()
    g.close()
    cpu = []
    for name in ("fp32_128_row", "fp32_1024_colB"):
        w = inp.WORKLOADS[name]
        A, B = inp.make_workload(w)
        A64, B64 = A.double().numpy(), B.double().numpy()
        for threads in (1, oracle.default_threads()):
            t = time.perf_counter()
            Cr, S = oracle.gemm(A64, B64, w.layout_b, nthreads=threads)
            dt = time.perf_counter() - t
            entry = {"workload": name, "threads": threads, "seconds": round(dt, 4),
                     "gflops": round(w.flops / dt / 1e9, 3)}
            if name in small_c:  # this run's GPU result against the oracle
                import numpy as np
                err = np.abs(small_c[name] - Cr) / np.maximum(S, 1e-300)
                entry["gpu_max_err_over_sum_abs"] = float(err.max())
            cpu.append(entry)
    print(json.dumps({"configs": out, "oracle": cpu}))
    return 0


def run_ladder(args):
    """Time every kernel of the labelled ladder suite (include/gemm_ladder.h),
    this library's FP32 path and cuBLAS SGEMM (TF32 off) on one square
    problem; report TFLOP/s and the share of cuBLAS."""
    import torch
    from dense_gemm_sm100_gb300 import gemm
    from dense_gemm_sm100_gb300 import inputs as inp
    n = args.ladder_size
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flops = 2.0 * n * n * n
    steps = max(1, min(args.steps, 10))
    A, B = inp.make_operands(n, n, n, seed=3)
    _, Bc = inp.make_operands(n, n, n, layout_b=inp.B_COL_MAJOR, seed=3)
    A, B, Bc = A.to(dev), B.to(dev), Bc.to(dev)
    C = torch.empty((n, n), device=dev)

    def tf(run):
        _, per, _ = time_device(run, stream, steps, args.warmup)
        return flops / (statistics.median(per) * 1e-3) / 1e12

    torch.backends.cuda.matmul.allow_tf32 = False
    cublas = tf(lambda: torch.matmul(A, B))
    g = gemm.Gemm(0)
    lib = tf(lambda: g.run(A, B, C, "row", "f32", stream))
    rows = []
    for step in [int(x) for x in args.ladder_steps.split(",")]:
        Bs = Bc if step == gemm.GEMM_LADDER_PMPP_CORNER_TURN else B
        rc = gemm.gemm_ladder_run(step, n, n, n, A.data_ptr(), Bs.data_ptr(), C.data_ptr(),
                                  stream.cuda_stream)
        if rc != gemm.GEMM_OK:
            rows.append({"step": step, "error": gemm.gemm_status_string(rc)})
            continue
        t = tf(lambda: gemm.gemm_ladder_run(step, n, n, n, A.data_ptr(), Bs.data_ptr(),
                                            C.data_ptr(), stream.cuda_stream))
        row = {"step": step, "name": gemm.gemm_ladder_name(step), "tflops": round(t, 2),
               "pct_of_cublas": round(100 * t / cublas, 1)}
        if step in PAGES_LADDER_PCT:
            row["pages_pct_of_cublas_v100"] = PAGES_LADDER_PCT[step]
        rows.append(row)
    g.close()
    print(json.dumps({
        "ladder": rows, "size": n, "unit": UNIT,
        "library_fp32": {"tflops": round(lib, 2), "pct_of_cublas": round(100 * lib / cublas, 1),
                         "path": "gemm_run FP32 (TMA + mbarrier + packed FMA)"},
        "cublas_fp32": {"tflops": round(cublas, 2), "what": "torch.matmul, TF32 disallowed (side reference)"},
    }))
    return 0


# ---------------------------------------------------------------- entry

def run_reference(args, ctx):
    """The reference arm: the FP64 CPU oracle, each step one row sample."""
    if ctx is not None and ctx["rank"] != 0:
        return 0
    name = args.workload
    A64, B64, w, rows, threads = oracle_sample(name, target_s=args.ref_step_s)
    for _ in range(args.warmup):
        time_oracle(A64, B64, w, max(1, rows // 8))
    times = []
    for _ in range(args.steps):
        _, dt = time_oracle(A64, B64, w, rows)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = 2.0 * rows * w.N * w.K / (ms * 1e-3) / 1e12
    sample = f"rows 0..{rows - 1} of A times all of B ({rows}x{w.N}x{w.K} of the {w.M}x{w.N}x{w.K} product)"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS.get(name, name), "M": w.M, "N": w.N, "K": w.K},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-modes", action="store_true", help="skip the tensor-core workloads")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-peaks", action="store_true",
                    help="skip the FMA and tensor-core peak microbenchmarks")
    ap.add_argument("--no-side-reference", action="store_true",
                    help="skip the labelled cuBLAS side reference")
    ap.add_argument("--peaks-only", action="store_true",
                    help="run only the FMA and tensor-core peak microbenchmarks (one JSON line)")
    ap.add_argument("--ladder", action="store_true",
                    help="time the labelled ladder suite (pages' optimisation steps) instead")
    ap.add_argument("--simt-config", type=int, default=0,
                    help="force the FP32 tile configuration (GEMM_OPT_SIMT_CONFIG; 0 = chosen per shape)")
    ap.add_argument("--tc-mode", type=int, default=0,
                    help="force the tensor-core mode (GEMM_OPT_TC_CLUSTER: 1 one CTA per tile, 3 pair MMA; 0 = default)")
    ap.add_argument("--tc-group-m", type=int, default=0,
                    help="GEMM_OPT_TC_GROUP_M: tensor-core tile-order group height in units (0 = chosen)")
    ap.add_argument("--simt-group-m", type=int, default=0,
                    help="GEMM_OPT_SIMT_GROUP_M: FP32 SIMT tile-order group height in tile rows (0 = chosen)")
    ap.add_argument("--split-k", type=int, default=0,
                    help="GEMM_OPT_SPLIT_K (0 = chosen per shape, 1 = never, n = n slices)")
    ap.add_argument("--results", default=None,
                    help="with --configs: append one JSON line per finished workload to this file "
                         "and skip workloads already in it")
    ap.add_argument("--ncu-summary", default=None, metavar="REPORT",
                    help="print a Markdown table of the usual metrics from an ncu report (no GPU needed)")
    ap.add_argument("--configs", action="store_true",
                    help="time every specified workload warm and with L2 scrubbed, and the oracle "
                         "on the small ones with 1 and all host threads (one JSON document)")
    ap.add_argument("--ladder-size", type=int, default=4096)
    ap.add_argument("--ladder-steps", default="1,2,3,4,5,6,7,8,101,102")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.ncu_summary:
        return run_ncu_summary(args.ncu_summary)
    ctx = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ctx)
    if args.ladder:
        return run_ladder(args)
    if args.peaks_only:
        import torch
        torch.cuda.set_device(0)
        print(json.dumps(measure_peaks(0, load_peaks()[0]["sm_max_mhz"])))
        return 0
    if args.configs:
        return run_configs(args)

    import torch
    from dense_gemm_sm100_gb300 import gemm
    dev_index = ctx["local"] if ctx else 0
    torch.cuda.set_device(dev_index)
    peaks, peak_note = load_peaks()
    g = gemm.Gemm(dev_index)
    apply_options(g, args)
    rank0 = ctx is None or ctx["rank"] == 0

    sampler = ClockSampler(dev_index) if rank0 else None
    clocks = None
    if sampler:
        sampler.start()
    main_res = bench_workload(g, args.workload, args.steps, args.warmup, ctx, peaks, peak_note,
                              with_e2e=False)
    side = {}
    if not args.no_side_reference:
        side[args.workload] = bench_workload(g, args.workload, min(args.steps, 10), args.warmup, ctx,
                                             peaks, peak_note, with_e2e=False,
                                             side_cublas=True)["cublas_side"]
    if sampler:
        sampler.stop()
        clocks = sampler.summary(*main_res["wall_window"])
        if clocks and clocks.get("sm_mhz"):
            f = clocks["sm_mhz"] / peaks["sm_max_mhz"]
            r = main_res["roofline"]
            r["frac_at_observed_clock"] = round(r["achieved"] / (r["peak"] * f), 4) if f > 0 else None
    e2e = None
    if not args.no_e2e:
        # Right after the headline leg, in the same thermal and power state
        # (after the tensor-core modes' power-capped minutes the SM clock can
        # sit lower); the host-buffer step moves 768 MiB over the host link:
        # 10 steps.
        esampler = ClockSampler(dev_index) if rank0 else None
        if esampler:
            esampler.start()
        t_e0 = time.time()
        r = bench_workload(g, args.workload, min(args.steps, 10), args.warmup, ctx, peaks,
                           peak_note, with_e2e=True)
        t_e1 = time.time()
        e2e = r["e2e"]
        if esampler:
            esampler.stop()
            e2e["clocks"] = esampler.summary(t_e0, t_e1)
    measured = None
    if not args.no_peaks:
        measured = measure_peaks(dev_index, peaks["sm_max_mhz"])
        if measured:
            # the higher of the scalar and packed FMA readings is the FP32 roof
            add_microbench(main_res["roofline"],
                           max(measured.get("ffma_tflops") or 0.0, measured.get("ffma2_tflops") or 0.0))
    modes = []
    if not args.no_modes:
        for name in TC_WORKLOADS + SIMT_WORKLOADS:
            msampler = ClockSampler(dev_index) if rank0 else None
            if msampler:
                msampler.start()
            mode_steps = max(args.steps, MIN_MODE_STEPS.get(name, 0))
            r = bench_workload(g, name, mode_steps, args.warmup, ctx, peaks, peak_note,
                               with_e2e=False, side_cublas=not args.no_side_reference)
            m = {k: r[k] for k in ("workload", "description", "dtype", "value",
                                   "ms_per_step", "kernel_ms", "kernel_ms_median", "path", "roofline")}
            m["steps"], m["warmup"] = r["steps"], args.warmup
            m["l2"] = l2_note(r)
            if r["dtype"] == "f32" and measured:
                add_microbench(m["roofline"], max(measured.get("ffma_tflops") or 0.0,
                                                  measured.get("ffma2_tflops") or 0.0))
            elif measured:
                mb = measured.get(f"mma_{r['dtype']}_tflops")
                if r["dtype"] == "f32x3" and measured.get("mma_tf32_tflops"):
                    mb = measured["mma_tf32_tflops"] / 3
                add_microbench(m["roofline"], mb)
            if "cublas_side" in r:
                m["cublas_side"] = r["cublas_side"]
            if "graph" in r:
                m["graph"] = r["graph"]
            if msampler:
                msampler.stop()
                m["clocks"] = msampler.summary(*r["wall_window"])
                if m["clocks"] and m["clocks"].get("sm_mhz"):
                    # the same peak scaled to the SM clock seen while this mode ran
                    f = m["clocks"]["sm_mhz"] / peaks["sm_max_mhz"]
                    m["roofline"]["frac_at_observed_clock"] = round(
                        m["roofline"]["achieved"] / (m["roofline"]["peak"] * f), 4) if f > 0 else None
            modes.append(m)
    cpu = None
    if rank0 and ctx is None and not args.no_cpu_baseline:
        A64, B64, w, rows, threads = oracle_sample(args.workload, target_s=args.cpu_seconds)
        value, dt = time_oracle(A64, B64, w, rows)
        cpu = {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of A times all of B ({rows}x{w.N}x{w.K} of the "
                         f"{w.M}x{w.N}x{w.K} product), {dt:.1f} s, FP64 with |a*b| sums"}
    g.close()
    if not rank0:
        return 0
    n = ctx["world"] if ctx else 1
    line = {
        "metric": METRIC, "value": main_res["value"], "unit": UNIT, "n_gpus": n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": main_res["dtype"], "data": "synthetic",
        "config": {"workload": main_res["description"], "M": main_res["M"], "N": main_res["N"],
                   "K": main_res["K"], "layout_b": main_res["layout_b"], "path": main_res["path"],
                   "l2": l2_note(main_res),
                   "parallelism": f"replicas{n}" if n > 1 else "single-gpu"},
        "roofline": main_res["roofline"],
        "kernel_ms": main_res["kernel_ms"],
        "kernel_ms_median": main_res["kernel_ms_median"],
        "kernel_ms_min": main_res["kernel_ms_min"],
        "gpu_launches": main_res["launches_timed"],
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "modes": modes,
        "cublas_side": side.get(args.workload),
        "peaks_measured": measured,
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
