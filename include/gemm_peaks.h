/*
 * Peak-rate microbenchmarks of the arithmetic units the GEMM kernels are
 * bound by: the compute roof of the roofline ("GEMM 性能优化", Roofline 模型;
 * "PMPP Chapter 06: Performance considerations", compute-bound kernels).
 * They calibrate the roofline denominators on the GPU at hand: the FP32
 * SIMT peak that is otherwise derived from SMs x 128 lanes x 2 x clock, and
 * the TF32 tensor rate that is otherwise scaled from BF16 by a nominal ratio.
 *
 * Both calls launch one kernel on `stream` on the current device and return
 * without waiting; the caller times the launch (CUDA events on `stream`) and
 * divides *flops by the time.  Return codes are those of gemm.h.
 */
#ifndef DENSE_GEMM_GB300_PEAKS_H
#define DENSE_GEMM_GB300_PEAKS_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * FP32 multiply-adds on the CUDA cores: 4 CTAs of 256 threads per SM, each
 * thread `iters` rounds of 16 independent multiply-adds, issued as scalar
 * fma.rn.f32 (packed = 0) or as 8 packed fma.rn.f32x2 (packed = 1).
 * iters > 0 and a multiple of 16.  sink: device float[2] that receives a
 * value from the chains (so the compiler keeps them).  *flops (may be NULL):
 * floating-point operations of the launch (2 per multiply-add).
 * GEMM_ERR_INVALID for bad arguments, GEMM_ERR_CUDA if the launch fails.
 */
int gemm_peak_fma_run(int packed, int64_t iters, float *sink, cudaStream_t stream, double *flops);

/*
 * tcgen05 MMAs (M = 128, N = 256, FP32 accumulation in tensor memory), one
 * CTA per SM, operands resident in shared memory (K-major, 128-byte swizzle),
 * `iters` rounds of one 128-byte K slice each (4 instructions: K = 64 BF16 or
 * 32 TF32 elements).  dtype: GEMM_BF16 or GEMM_TF32.  status: device int
 * (may be NULL) that receives 0x100 | 6 if the final wait for the MMAs
 * expires after timeout_ns (0 = 4 s); tensor memory is freed either way.
 * *flops (may be NULL): floating-point operations of the launch.
 */
int gemm_peak_mma_run(int dtype, int64_t iters, int *status, uint64_t timeout_ns, cudaStream_t stream,
                      double *flops);

#ifdef __cplusplus
}
#endif

#endif
