"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every function include/gemm.h declares, and checks arguments on the host."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")
HEADERS = [HEADER, os.path.join(ROOT, "include", "gemm_ladder.h"),
           os.path.join(ROOT, "include", "gemm_peaks.h")]


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_sm100_gb300 import build, gemm
    build.build()
    return gemm.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(gemm_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("gemm_create", "gemm_run", "gemm_destroy", "gemm_run_host",
                     "gemm_validate", "gemm_sync_status", "gemm_last_error_string",
                     "gemm_run_noalloc", "gemm_ladder_run", "gemm_peak_fma_run", "gemm_peak_mma_run"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_built_for_sm_103a_only():
    from dense_gemm_sm100_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def test_version_and_status_names(lib):
    from dense_gemm_sm100_gb300 import gemm as g
    assert g.gemm_version() == 1
    assert g.gemm_status_string(g.GEMM_OK) == "GEMM_OK"
    assert g.gemm_status_string(g.GEMM_ERR_ALIGNMENT) == "GEMM_ERR_ALIGNMENT"
    assert g.gemm_status_string(-99) == "unknown gemm status"


P = 0x10000  # a fake, 16-byte aligned address: gemm_validate never dereferences


@pytest.mark.parametrize("args,code", [
    ((0, 4, 4, 4, P, 4, P, 4, P, 4, 0), 0),
    ((1, 4, 4, 4, P, 4, P, 4, P, 4, 2), 0),
    ((2, 4, 4, 4, P, 4, P, 4, P, 4, 0), -1),      # bad layout
    ((0, 4, 4, 4, P, 4, P, 4, P, 4, 4), -1),      # bad dtype
    ((0, 4, 4, 4, P, 4, P, 4, P, 4, 3), 0),       # FP32-accurate tensor-core mode
    ((0, -1, 4, 4, P, 4, P, 4, P, 4, 0), -1),     # negative M
    ((0, 4, 4, 4, P, 3, P, 4, P, 4, 0), -1),      # lda < K
    ((0, 4, 5, 4, P, 4, P, 4, P, 5, 0), -1),      # row-major ldb < N
    ((1, 4, 5, 6, P, 6, P, 5, P, 5, 0), -1),      # column-major ldb < K
    ((0, 4, 4, 4, P, 4, P, 4, P, 3, 0), -1),      # ldc < N
    ((0, 4, 4, 4, 0, 4, P, 4, P, 4, 0), -1),      # A NULL
    ((0, 4, 4, 4, P, 4, P, 4, 0, 4, 0), -1),      # C NULL
    ((0, 4, 4, 4, P + 2, 4, P, 4, P, 4, 0), -2),  # FP32 A not 4-byte aligned
    ((0, 4, 4, 4, P + 2, 4, P, 4, P, 4, 2), 0),   # BF16 A 2-byte aligned is fine
    ((0, 4, 4, 4, P + 1, 4, P, 4, P, 4, 2), -2),  # BF16 A odd address
    ((0, 4, 4, 4, P, 4, P, 4, P + 2, 4, 0), -2),  # C not 4-byte aligned
    ((0, 0, 4, 4, 0, 0, 0, 0, 0, 0, 0), 0),       # M = 0: nothing to check
    ((0, 4, 4, 0, 0, 0, 0, 0, P, 4, 0), 0),       # K = 0: A, B unused
    ((0, 4, 4, 7, P, 7, P, 4, P, 4, 0), 0),       # odd ld is re-packed, not rejected
    ((0, 1 << 31, 4, 4, P, 4, P, 4, P, 4, 0), -1),  # dimension too large
])
def test_validate(lib, args, code):
    from dense_gemm_sm100_gb300 import gemm as g
    assert g.gemm_validate(*args) == code


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour without a GPU")
def test_create_without_gpu_reports_device_error(lib):
    from dense_gemm_sm100_gb300 import gemm as g
    h = ctypes.c_void_p()
    assert lib.gemm_create(ctypes.byref(h), 0) == g.GEMM_ERR_DEVICE
    assert h.value is None


def test_ladder_rejects_bad_shapes_without_gpu(lib):
    from dense_gemm_sm100_gb300 import gemm as g
    # argument and shape checks happen before any launch
    assert g.gemm_ladder_run(3, 100, 128, 64, P, P, P, None) == g.GEMM_ERR_INVALID  # M % 128
    assert g.gemm_ladder_run(102, 64, 100, 64, P, P, P, None) == g.GEMM_ERR_INVALID  # N % 128
    assert g.gemm_ladder_run(5, 128, 128, 8, P + 4, P, P, None) == g.GEMM_ERR_ALIGNMENT
    assert g.gemm_ladder_run(999, 128, 128, 8, P, P, P, None) == g.GEMM_ERR_INVALID
    assert g.gemm_ladder_run(1, 0, 4, 4, P, P, P, None) == g.GEMM_ERR_INVALID
    assert g.gemm_ladder_name(2).startswith("2 shared-memory tiling")
    assert g.gemm_ladder_name(77) == ""


def test_peak_microbenchmarks_reject_bad_arguments_without_gpu(lib):
    from dense_gemm_sm100_gb300 import gemm as g
    # argument checks happen before any device call
    assert g.gemm_peak_fma_run(2, 16, P, None)[0] == g.GEMM_ERR_INVALID    # packed not 0/1
    assert g.gemm_peak_fma_run(1, 17, P, None)[0] == g.GEMM_ERR_INVALID    # iters % 16
    assert g.gemm_peak_fma_run(1, 0, P, None)[0] == g.GEMM_ERR_INVALID
    assert g.gemm_peak_fma_run(0, 16, 0, None)[0] == g.GEMM_ERR_INVALID    # no sink
    assert g.gemm_peak_mma_run(g.GEMM_F32, 10, 0, 0, None)[0] == g.GEMM_ERR_INVALID
    assert g.gemm_peak_mma_run(g.GEMM_BF16, 0, 0, 0, None)[0] == g.GEMM_ERR_INVALID


def test_null_handle_calls_are_rejected(lib):
    from dense_gemm_sm100_gb300 import gemm as g
    assert g.gemm_run(None, 0, 4, 4, 4, P, 4, P, 4, P, 4, 0, None) == g.GEMM_ERR_INVALID
    assert g.gemm_destroy(None) == g.GEMM_OK
    assert g.gemm_last_error_string(None) == ""
    assert g.gemm_launch_count(None) == 0


C_CHECK = os.path.join(ROOT, "tests", "c_abi", "gemm_abi_check.c")


def c_abi_build_cmd(out, cuda_home):
    return ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
            "-isystem", os.path.join(cuda_home, "include"), C_CHECK,
            "-L", os.path.join(ROOT, "dense_gemm_sm100_gb300"), "-ldense_gemm_gb300",
            "-L", os.path.join(cuda_home, "lib64"), "-lcudart",
            "-Wl,-rpath," + os.path.join(ROOT, "dense_gemm_sm100_gb300"), "-o", out]


def test_headers_are_plain_c_and_the_library_links(lib, tmp_path):
    """The three public headers compile as C99 with warnings as errors, and a
    C program links against the library (run on the GPU by
    tests/test_c_abi_gpu.py)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    r = subprocess.run(c_abi_build_cmd(str(tmp_path / "abi_check"), cuda_home), capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from dense_gemm_sm100_gb300 import gemm as g
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(g, "_lib", None)
    with pytest.raises(g.GemmLibraryMissing):
        g.load_library()


def test_noalloc_options_are_checked_on_the_host(lib):
    """The allocation-free calls' process-wide settings: only the wait limit
    (1e6..6e10 ns) and the test hook (0/1) exist; nothing touches a GPU."""
    from dense_gemm_sm100_gb300 import gemm as g
    assert g.gemm_noalloc_set_option(g.GEMM_OPT_WAIT_TIMEOUT_NS, 999_999) == g.GEMM_ERR_INVALID
    assert g.gemm_noalloc_set_option(g.GEMM_OPT_WAIT_TIMEOUT_NS, 61_000_000_000) == g.GEMM_ERR_INVALID
    assert g.gemm_noalloc_set_option(g.GEMM_OPT_DEBUG_DROP_LOAD, 2) == g.GEMM_ERR_INVALID
    assert g.gemm_noalloc_set_option(g.GEMM_OPT_SIMT_CONFIG, 1) == g.GEMM_ERR_INVALID
    assert g.gemm_noalloc_set_option(g.GEMM_OPT_WAIT_TIMEOUT_NS, 4_000_000_000) == g.GEMM_OK
    assert g.gemm_noalloc_set_option(g.GEMM_OPT_DEBUG_DROP_LOAD, 0) == g.GEMM_OK
