"""Python binding of the C ABI in include/gemm.h (argument marshalling only).

The functions ``gemm_create``, ``gemm_run``, ``gemm_run_host``,
``gemm_destroy``, ``gemm_validate``, ``gemm_sync_status``,
``gemm_set_option``, ``gemm_last_error_string``, ``gemm_status_string``,
``gemm_last_path``, ``gemm_launch_count``, ``gemm_version``,
``gemm_run_noalloc``, ``gemm_ladder_run``, ``gemm_ladder_name``,
``gemm_peak_fma_run`` and ``gemm_peak_mma_run`` take and return the same
plain values as their C counterparts (pointers as ints; the FLOP-count
out-parameter of the peak calls is returned as a second value).  ``Gemm``
wraps a handle for torch tensors.  Every GEMM step runs in the library's CUDA
kernels; there is no other code path, and calling anything here without the
built library raises ``GemmLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GEMM_B_ROW_MAJOR = 0
GEMM_B_COL_MAJOR = 1
GEMM_F32 = 0
GEMM_TF32 = 1
GEMM_BF16 = 2
GEMM_F32_3XTF32 = 3

GEMM_OK = 0
GEMM_ERR_INVALID = -1
GEMM_ERR_ALIGNMENT = -2
GEMM_ERR_CUDA = -3
GEMM_ERR_TIMEOUT = -4
GEMM_ERR_DEVICE = -5
GEMM_ERR_NOMEM = -6

GEMM_OPT_FORCE_REPACK = 1
GEMM_OPT_WAIT_TIMEOUT_NS = 2
GEMM_OPT_SIMT_GROUP_M = 3
GEMM_OPT_TC_GROUP_M = 4
GEMM_OPT_MAX_CTAS = 5
GEMM_OPT_SIMT_CONFIG = 6
GEMM_OPT_SPLIT_K = 7
GEMM_OPT_TC_CLUSTER = 8
GEMM_OPT_TC_TMA_STORE = 9
GEMM_OPT_DEBUG_DROP_LOAD = 10
GEMM_OPT_ELEMENTWISE = 11
GEMM_OPT_WORKSPACE_LIMIT = 12
GEMM_OPT_TC_STAGE_SLICES = 13
GEMM_OPT_STREAM_K = 14
GEMM_OPT_SIMT_SMALL = 15

DTYPES = {"f32": GEMM_F32, "tf32": GEMM_TF32, "bf16": GEMM_BF16, "f32x3": GEMM_F32_3XTF32}
LAYOUTS = {"row": GEMM_B_ROW_MAJOR, "col": GEMM_B_COL_MAJOR}

LIB_PATH = _build.LIB_PATH


class GemmLibraryMissing(RuntimeError):
    """The CUDA library has not been built (run ``__graft_entry__.build()``)."""


class GemmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{gemm_status_string(code)}: {message}")
        self.code = code


_lock = threading.Lock()
_lib = None


def load_library():
    """Load ``libdense_gemm_gb300.so`` (raises GemmLibraryMissing if absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise GemmLibraryMissing(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        run_args = [vp, ci, i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, vp]
        sig = {
            "gemm_create": ([ctypes.POINTER(vp), ci], ci),
            "gemm_destroy": ([vp], ci),
            "gemm_run": (run_args, ci),
            "gemm_run_host": (run_args, ci),
            "gemm_validate": ([ci, i64, i64, i64, vp, i64, vp, i64, vp, i64, ci], ci),
            "gemm_sync_status": ([vp, vp], ci),
            "gemm_set_option": ([vp, ci, i64], ci),
            "gemm_last_error_string": ([vp], ctypes.c_char_p),
            "gemm_status_string": ([ci], ctypes.c_char_p),
            "gemm_last_path": ([vp], ctypes.c_char_p),
            "gemm_launch_count": ([vp], i64),
            "gemm_version": ([], ci),
            "gemm_run_noalloc": ([ci, i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, vp], ci),
            "gemm_noalloc_sync_status": ([vp], ci),
            "gemm_noalloc_set_option": ([ci, i64], ci),
            "gemm_ladder_run": ([ci, i64, i64, i64, vp, vp, vp, vp], ci),
            "gemm_ladder_name": ([ci], ctypes.c_char_p),
            "gemm_peak_fma_run": ([ci, i64, vp, vp, ctypes.POINTER(ctypes.c_double)], ci),
            "gemm_peak_mma_run": ([ci, i64, vp, ctypes.c_uint64, vp, ctypes.POINTER(ctypes.c_double)], ci),
        }
        for name, (argtypes, restype) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = restype
        _lib = lib
        return lib


# ----------------------------------------------------------- C-named functions

def gemm_version() -> int:
    return load_library().gemm_version()


def gemm_status_string(code: int) -> str:
    return load_library().gemm_status_string(code).decode()


def gemm_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    rc = load_library().gemm_create(ctypes.byref(h), device)
    if rc != GEMM_OK:
        raise GemmError(rc, f"gemm_create(device={device}) failed")
    return h.value


def gemm_destroy(handle: int) -> int:
    return load_library().gemm_destroy(handle)


def gemm_run(handle, layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream) -> int:
    return load_library().gemm_run(handle, layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream)


def gemm_run_host(handle, layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream) -> int:
    return load_library().gemm_run_host(handle, layout_b, M, N, K, A, lda, B, ldb, C, ldc,
                                        dtype, stream)


def gemm_validate(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype) -> int:
    return load_library().gemm_validate(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype)


def gemm_sync_status(handle, stream) -> int:
    return load_library().gemm_sync_status(handle, stream)


def gemm_set_option(handle, option, value) -> int:
    return load_library().gemm_set_option(handle, option, value)


def gemm_last_error_string(handle) -> str:
    return load_library().gemm_last_error_string(handle).decode()


def gemm_last_path(handle) -> str:
    return load_library().gemm_last_path(handle).decode()


def gemm_launch_count(handle) -> int:
    return load_library().gemm_launch_count(handle)


def gemm_run_noalloc(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream) -> int:
    """C = A·B with no device allocation (no handle; the current device's
    static scratch holds re-packed operands, at most
    GEMM_NOALLOC_SCRATCH_BYTES).  For callers that cannot allocate."""
    return load_library().gemm_run_noalloc(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype,
                                           stream)


def gemm_noalloc_sync_status(stream) -> int:
    """Waits for `stream`; GEMM_ERR_TIMEOUT if an in-kernel wait of an
    allocation-free call on the current device expired (then cleared)."""
    return load_library().gemm_noalloc_sync_status(stream)


def gemm_noalloc_set_option(option, value) -> int:
    """Process-wide wait limit / test hook of the allocation-free calls."""
    return load_library().gemm_noalloc_set_option(option, value)


GEMM_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

# Labelled benchmark suite (include/gemm_ladder.h): the pages' optimisation
# ladder and the PMPP worked kernels.  Not the library's GEMM path.
GEMM_LADDER_STEPS = {1: "naive", 2: "smem_tiling", 3: "thread_tiling", 4: "vectorized",
                     5: "conflict_free", 6: "warp_tiling", 7: "double_buffer", 8: "cp_async"}
GEMM_LADDER_PMPP_CORNER_TURN = 101
GEMM_LADDER_PMPP_COARSENED = 102


def gemm_ladder_run(step, M, N, K, A, B, C, stream) -> int:
    return load_library().gemm_ladder_run(step, M, N, K, A, B, C, stream)


def gemm_ladder_name(step) -> str:
    return load_library().gemm_ladder_name(step).decode()


# Peak-rate microbenchmarks (include/gemm_peaks.h): the compute roofs.

def gemm_peak_fma_run(packed, iters, sink, stream) -> tuple[int, float]:
    flops = ctypes.c_double(0.0)
    rc = load_library().gemm_peak_fma_run(packed, iters, sink, stream, ctypes.byref(flops))
    return rc, flops.value


def gemm_peak_mma_run(dtype, iters, status, timeout_ns, stream) -> tuple[int, float]:
    flops = ctypes.c_double(0.0)
    rc = load_library().gemm_peak_mma_run(dtype, iters, status, timeout_ns, stream, ctypes.byref(flops))
    return rc, flops.value


def measure_peak(kind: str, iters: int, reps: int = 3, stream=None) -> dict:
    """Time the microbenchmark `kind` ("ffma", "ffma2", "mma_bf16",
    "mma_tf32") with CUDA events on `stream`: one warm-up launch, then the
    best of `reps` launches.  Returns TFLOP/s and the launch time."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    sh = _stream_handle(s)
    sink = torch.zeros(2, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def launch():
        if kind in ("ffma", "ffma2"):
            rc, fl = gemm_peak_fma_run(1 if kind == "ffma2" else 0, iters, sink.data_ptr(), sh)
        else:
            dt = GEMM_BF16 if kind == "mma_bf16" else GEMM_TF32
            rc, fl = gemm_peak_mma_run(dt, iters, status.data_ptr(), 0, sh)
        if rc != GEMM_OK:
            raise GemmError(rc, f"{kind} microbenchmark: {gemm_status_string(rc)}")
        return fl

    launch()
    best_ms, flops = None, 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        flops = launch()
        e1.record(s)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best_ms = ms if best_ms is None else min(best_ms, ms)
    if int(status.item()) != 0:
        raise GemmError(GEMM_ERR_TIMEOUT, f"{kind} microbenchmark: a wait expired")
    return {"tflops": flops / (best_ms * 1e-3) / 1e12, "ms": best_ms, "flops": flops}


# ------------------------------------------------------------- torch wrapper

def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class Gemm:
    """A library handle used with torch tensors.

    ``run(A, B, C, layout_b, dtype)`` computes C = A·B on the GPU: A is (M, K)
    row-major, B is (K, N) for ``layout_b="row"`` or (N, K) for ``"col"``
    (each row holding one column of the logical B), C is (M, N).  Rows may be
    padded (any stride(0) >= columns, stride(1) == 1).  The call is queued on
    ``stream`` (default: torch's current stream) and returns at once.
    """

    def __init__(self, device: int = 0):
        self.device = device
        self.handle = gemm_create(device)

    def close(self):
        if self.handle:
            gemm_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc: int):
        if rc != GEMM_OK:
            raise GemmError(rc, gemm_last_error_string(self.handle))

    def set_option(self, option: int, value: int):
        self._check(gemm_set_option(self.handle, option, int(value)))

    @staticmethod
    def _dims(A, B, layout_b):
        M, K = A.shape
        if layout_b == GEMM_B_ROW_MAJOR:
            Kb, N = B.shape
        else:
            N, Kb = B.shape
        if Kb != K:
            raise ValueError(f"inner dimensions differ: A has K={K}, B has K={Kb}")
        return M, N, K

    @staticmethod
    def _ld(t):
        if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError("operands must be 2-D with unit stride along rows")
        return max(t.stride(0), t.shape[1], 1)

    def run(self, A, B, C, layout_b="row", dtype="f32", stream=None):
        lb = LAYOUTS.get(layout_b, layout_b)
        dt = DTYPES.get(dtype, dtype)
        M, N, K = self._dims(A, B, lb)
        if tuple(C.shape) != (M, N):
            raise ValueError(f"C has shape {tuple(C.shape)}, expected {(M, N)}")
        self._check(gemm_run(self.handle, lb, M, N, K, A.data_ptr(), self._ld(A), B.data_ptr(),
                             self._ld(B), C.data_ptr(), self._ld(C), dt, _stream_handle(stream)))
        return C

    def run_host(self, A, B, C, layout_b="row", dtype="f32", stream=None):
        """As ``run`` with CPU tensors (pinned for asynchronous copies): the
        library copies A and B in, runs, and copies C out on ``stream``."""
        lb = LAYOUTS.get(layout_b, layout_b)
        dt = DTYPES.get(dtype, dtype)
        M, N, K = self._dims(A, B, lb)
        self._check(gemm_run_host(self.handle, lb, M, N, K, A.data_ptr(), self._ld(A),
                                  B.data_ptr(), self._ld(B), C.data_ptr(), self._ld(C), dt,
                                  _stream_handle(stream)))
        return C

    def sync_status(self, stream=None):
        """Wait for ``stream`` and raise GemmError if an in-kernel wait expired."""
        self._check(gemm_sync_status(self.handle, _stream_handle(stream)))

    @property
    def last_path(self) -> str:
        return gemm_last_path(self.handle)

    @property
    def launch_count(self) -> int:
        return gemm_launch_count(self.handle)


def matmul(A, B, layout_b="row", dtype="f32", out=None, stream=None, handle: Gemm | None = None):
    """Allocate C (float32, on A's device) if needed and return C = A·B."""
    import torch
    lb = LAYOUTS.get(layout_b, layout_b)
    M, N, _ = Gemm._dims(A, B, lb)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    g = handle or _default_handle(A.device.index or 0)
    return g.run(A, B, out, lb, dtype, stream)


_handles: dict[int, Gemm] = {}


def _default_handle(device: int) -> Gemm:
    with _lock:
        h = _handles.get(device)
    if h is None:
        h = Gemm(device)
        with _lock:
            _handles[device] = h
    return h
