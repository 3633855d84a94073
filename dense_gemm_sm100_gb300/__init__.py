"""GB300-native dense GEMM (C = A·B) behind a C ABI; see include/gemm.h."""
