"""The C ABI from a plain C program (tests/c_abi/gemm_abi_check.c) on the
GPU: FP32 with both B layouts and TF32 through gemm_run, FP32 through
gemm_run_host, exact on integer inputs, and argument errors as codes."""
import os
import shutil
import subprocess

import pytest
import torch

from tests.test_abi_cpu import c_abi_build_cmd

pytestmark = pytest.mark.gpu


def test_c_program_drives_the_library(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    from dense_gemm_sm100_gb300 import build
    build.build()
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "abi_check")
    r = subprocess.run(c_abi_build_cmd(exe, cuda_home), capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI OK" in r.stdout
