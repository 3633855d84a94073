"""GB300-native dense GEMM (C = A·B) behind a C ABI (include/gemm.h).

``dense_gemm_sm100_gb300.gemm`` is the Python binding; ``build`` compiles the
CUDA library in-tree; ``inputs`` draws seeded operands; ``roofline`` holds the
work/traffic model used by the benchmark.
"""
from . import build, inputs, roofline  # noqa: F401
from .gemm import (GEMM_B_COL_MAJOR, GEMM_B_ROW_MAJOR, GEMM_BF16, GEMM_F32,  # noqa: F401
                   GEMM_TF32, Gemm, GemmError, GemmLibraryMissing, matmul)
