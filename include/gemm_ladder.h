/*
 * Labelled benchmark suite: the optimisation ladder of "GEMM 性能优化"
 * (section 八个台阶, steps 1-7; step 8, SASS tuning, is not reproduced) and the
 * two worked kernels of "PMPP Chapter 06: Performance considerations"
 * (section 1, corner turning; section 3, thread coarsening), built for
 * sm_103a.  These kernels are NOT the library's GEMM path (that is gemm_run
 * in gemm.h); they exist to measure each step of the pages' ladder on this
 * GPU and to compare measured global-load traffic with the pages' formulas.
 *
 * Every kernel computes C = A·B with A (M x K), B (K x N) and C (M x N)
 * row-major with tight pitches (lda = K, ldb = N, ldc = N), all device
 * pointers, except GEMM_LADDER_PMPP_CORNER_TURN, whose B is column-major
 * (element (k, j) at B[j*K + k]).  The call is asynchronous on `stream`.
 *
 * Size rules (else GEMM_ERR_INVALID, nothing launched): steps 1, 2 and the
 * corner-turning kernel take any positive sizes; steps 3-8 need M and N
 * multiples of 128 and K a multiple of 8, and steps 4-8 16-byte-aligned
 * pointers (else GEMM_ERR_ALIGNMENT); the coarsening kernel needs M and K
 * multiples of 32 and N a multiple of 128.  Return codes are gemm.h's.
 */
#ifndef DENSE_GEMM_SM100_GB300_GEMM_LADDER_H
#define DENSE_GEMM_SM100_GB300_GEMM_LADDER_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_LADDER_NAIVE 1            /* one thread per element of C */
#define GEMM_LADDER_SMEM_TILING 2      /* 32x32 shared-memory tiles along K */
#define GEMM_LADDER_THREAD_TILING 3    /* 128x128 tile, 8x8 register outer product */
#define GEMM_LADDER_VECTORIZED 4       /* + float4 loads, A transposed in shared memory */
#define GEMM_LADDER_CONFLICT_FREE 5    /* + padded A tile, split B columns */
#define GEMM_LADDER_WARP_TILING 6      /* + 4x8 lanes per warp */
#define GEMM_LADDER_DOUBLE_BUFFER 7    /* + two shared buffers, register prefetch */
#define GEMM_LADDER_CP_ASYNC 8         /* + cp.async 3-stage pipeline */
#define GEMM_LADDER_PMPP_CORNER_TURN 101 /* 16x16 tiles, column-major B read along K, turned in shared memory */
#define GEMM_LADDER_PMPP_COARSENED 102   /* 32x32 tiles, 4 output tiles per block (one A tile per phase) */

/* Run one kernel of the suite.  Returns GEMM_OK or a GEMM_ERR_* code. */
int gemm_ladder_run(int step, int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                    float *C, cudaStream_t stream);

/* Human-readable name of a kernel of the suite ("" for an unknown id). */
const char *gemm_ladder_name(int step);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_SM100_GB300_GEMM_LADDER_H */
