/*
 * dense_gemm_sm100_gb300 — single-GPU dense GEMM C = A·B for NVIDIA GB300
 * (sm_103a), behind a plain C ABI.
 *
 * The operation (its definition and the layouts) comes from two pages:
 *
 *  - "GEMM 性能优化", section 指标与目标 and 台阶 1 (Shared Memory Tiling):
 *    C = A·B accumulates along K; 2·M·N·K flops; TFLOPS = 2MNK / (t·1e12).
 *  - "PMPP Chapter 06: Performance considerations", section 1 (Corner
 *    Turning example): A and C row-major, B column-major with element (k, j)
 *    at B[j*K + k]; out-of-range tile elements count as zero and only the
 *    C elements inside M x N are written.
 *
 * Semantics of every run entry point:
 *
 *     C[i*ldc + j] = sum_{k < K} A[i*lda + k] * B(k, j)   for i < M, j < N
 *     B(k, j) = B[k*ldb + j]   (GEMM_B_ROW_MAJOR)
 *     B(k, j) = B[j*ldb + k]   (GEMM_B_COL_MAJOR, the corner-turning case)
 *
 * C is overwritten (no alpha/beta); C elements outside the M x N box (the
 * ldc padding) are never touched.  Leading dimensions count elements.  K = 0
 * writes C = 0 (the empty sum).  M = 0 or N = 0 does nothing and succeeds.
 * C must not overlap A or B.  The order of the additions inside a sum is the
 * library's choice but fixed: repeated calls give bit-identical results.
 *
 * Compute modes (the `dtype` argument):
 *
 *   GEMM_F32   A, B, C float.  FP32 fused multiply-adds on the CUDA cores
 *              (SIMT), accumulation in FP32.
 *   GEMM_TF32  A, B, C float.  Tensor cores (tcgen05.mma kind::tf32): the
 *              operands enter the multiplier as TF32 (10-bit mantissa);
 *              products accumulate in FP32.
 *   GEMM_BF16  A, B bfloat16 (uint16 bit patterns), C float.  Tensor cores
 *              (tcgen05.mma kind::f16 with BF16 inputs), FP32 accumulation.
 *   GEMM_F32_3XTF32  A, B, C float; FP32-level accuracy on the tensor cores.
 *              Each operand is split into a TF32 part and the FP32 rest
 *              (x = hi + lo) in the workspace, three times along K, and one
 *              TF32 product over 3K computes hi(A)hi(B) + hi(A)lo(B) +
 *              lo(A)hi(B): A·B up to the lo(A)lo(B) term, about 2^-22 of
 *              |a·b|, within the FP32 mode's error bound.  Needs 3 (M + N) K
 *              floats of workspace; finite inputs (an infinity gives NaN).
 *
 * Ownership and threading: the caller owns A, B, C and the stream.  A handle
 * owns a small device status word and a device workspace that grows on
 * demand (used to re-pack operands whose address or leading dimension is not
 * a multiple of 16 bytes, for the K-slice partial products of small FP32
 * problems, and by gemm_run_host).  Calls on one handle must be
 * issued from one host thread at a time and be ordered on the GPU (one
 * stream, or streams the caller orders), because they share the workspace.
 * Growth is stream-ordered on the calling stream (cudaFreeAsync of the old
 * buffer after the last call that used it, then cudaMallocAsync from the
 * device's default memory pool): it neither synchronises the device nor
 * waits on the host.  gemm_destroy synchronises the device.
 *
 * Errors: every function returns GEMM_OK (0) or a negative GEMM_ERR_* code.
 * Argument errors are detected on the host before anything is launched.
 * gemm_last_error_string() describes the last failure on a handle.
 */
#ifndef DENSE_GEMM_SM100_GB300_GEMM_H
#define DENSE_GEMM_SM100_GB300_GEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_VERSION 1

/* Storage of B (the logical K x N operand). */
#define GEMM_B_ROW_MAJOR 0 /* B[k*ldb + j], ldb >= N */
#define GEMM_B_COL_MAJOR 1 /* B[j*ldb + k], ldb >= K (corner-turning case) */

/* Compute modes, see above. */
#define GEMM_F32 0
#define GEMM_TF32 1
#define GEMM_BF16 2
#define GEMM_F32_3XTF32 3

/* Return codes. */
#define GEMM_OK 0
#define GEMM_ERR_INVALID (-1)   /* null pointer, negative size, ld too small, unknown enum */
#define GEMM_ERR_ALIGNMENT (-2) /* a pointer not aligned to its element size */
#define GEMM_ERR_CUDA (-3)      /* a CUDA call failed; see gemm_last_error_string */
#define GEMM_ERR_TIMEOUT (-4)   /* a kernel's bounded wait expired (reported by gemm_sync_status) */
#define GEMM_ERR_DEVICE (-5)    /* no usable device, or not a compute capability 10.3 GPU */
#define GEMM_ERR_NOMEM (-6)     /* workspace or host bookkeeping allocation failed */

/* Options for gemm_set_option. */
#define GEMM_OPT_FORCE_REPACK 1   /* 1: always stage A and B through the workspace (tests) */
#define GEMM_OPT_WAIT_TIMEOUT_NS 2 /* limit of every in-kernel wait, nanoseconds (default 4e9) */
#define GEMM_OPT_SIMT_GROUP_M 3   /* tile-order group height in tiles for the FP32 kernel */
#define GEMM_OPT_TC_GROUP_M 4     /* tile-order group height in tiles for the tensor-core kernel */
#define GEMM_OPT_MAX_CTAS 5       /* cap on persistent CTAs (0 = SMs x resident CTAs per SM) */
/* FP32 tile configuration: 0 = chosen per shape (least estimated time), else
 * 1..8 = 128x128, 128x128 scalar FMA, 64x128, 64x64, 128x256 (8x16 per
 * thread), 192x128 (12 consumer warps, the usual row-major choice), 128x128
 * with 16 consumer warps, 256x128 with 16 consumer warps.  A configuration
 * the device cannot run is refused with GEMM_ERR_INVALID. */
#define GEMM_OPT_SIMT_CONFIG 6
/* K slices.  0 = chosen per shape.  FP32: the tiles of a partial last wave
 * (all tiles when they fill less than one wave) are cut into K slices;
 * tensor cores (one-CTA and pair modes): all tiles when they fill less than
 * one wave.  A second kernel adds the slices in slice order.  1 = never.
 * 2..64 = every tile cut into that many slices (fewer if K is short). */
#define GEMM_OPT_SPLIT_K 7
#define GEMM_OPT_TC_CLUSTER 8     /* tensor-core mode: 1 one CTA per tile, 3 pair MMA (cta_group::2, default); other values are GEMM_ERR_INVALID */
#define GEMM_OPT_TC_TMA_STORE 9   /* 1 (default): tensor-core epilogue stores C by TMA when aligned */
/* Test hook for failure detection, 0 by default.  1: in the next runs, CTA 0
 * of the GEMM kernel skips the copies of its first stage while still
 * expecting their bytes, so every wait that depends on them expires after
 * GEMM_OPT_WAIT_TIMEOUT_NS; the kernel then leaves C incomplete, ends, and
 * gemm_sync_status reports GEMM_ERR_TIMEOUT.  The context stays usable. */
#define GEMM_OPT_DEBUG_DROP_LOAD 10
/* FP32 with row-major B and an operand TMA cannot address (base or pitch not
 * a multiple of 16 bytes): 0 (default) = re-pack the operand into the
 * workspace first, then TMA; 1 = the producer warps copy A and B element by
 * element with 4-byte cp.async into the shared-memory ring (no workspace for
 * the operands, but 2-4x slower: the copies cannot keep the ring fed).
 * Tensor-core modes and column-major B always re-pack. */
#define GEMM_OPT_ELEMENTWISE 11
/* Cap on the handle's workspace in bytes (0 = none, the default).  A run
 * that would need more (re-packed operands, split-K partial tiles, staged
 * host buffers) fails with GEMM_ERR_NOMEM before launching anything; an
 * allocation already made is kept. */
#define GEMM_OPT_WORKSPACE_LIMIT 12
/* Pair-MMA tensor-core mode without a K split: 128-byte K slices per stage
 * of its shared-memory ring.  1 = six stages of one slice; 2 = three stages
 * of two slices (the same bytes in flight, half the barrier round trips per
 * MMA instruction); 0 (default) = the library's choice, at present six
 * stages of one slice (faster on every shape measured).  Same results. */
#define GEMM_OPT_TC_STAGE_SLICES 13
/* FP32: how the tiles of a partial last wave share the CTAs, when
 * GEMM_OPT_SPLIT_K is 0.  0 (default) = whichever of the two the wave model
 * rates shorter; 1 = K slices of equal length per tile; 2 = stream-K: the
 * tail tiles' 32-wide k steps, tile after tile, cut into one contiguous range
 * per CTA (at least four steps each), crossing tile boundaries (a second
 * kernel adds each tile's pieces in k order).  Same results up to the order
 * of the additions.  Configurations without stream-K kernels
 * (GEMM_OPT_SIMT_CONFIG 2, 5, 7, 8) and the element-wise producer
 * (GEMM_OPT_ELEMENTWISE) always take slices. */
#define GEMM_OPT_STREAM_K 14
/* FP32 small-problem kernel (one 32 x 32 tile of C per CTA of 1024 threads in
 * four K groups, 2 x 2 outputs per thread, the groups' partial tiles added in
 * order in shared memory; A and B read at any pitch and alignment, no
 * workspace): 0
 * (default) = used for problems of at most one tile per SM and K <= 384
 * when GEMM_OPT_SIMT_CONFIG, GEMM_OPT_MAX_CTAS and GEMM_OPT_SPLIT_K are 0;
 * 1 = never; 2 = for every FP32 problem (tests). */
#define GEMM_OPT_SIMT_SMALL 15

typedef struct gemm_ctx *gemm_handle_t;

/*
 * Create a handle bound to CUDA device `device` (which becomes current on the
 * calling thread).  Fails with GEMM_ERR_DEVICE when the device is missing or
 * is not compute capability 10.3 (GB300).  *out is set only on success.
 */
int gemm_create(gemm_handle_t *out, int device);

/* Release the handle and its device memory.  NULL is accepted. */
int gemm_destroy(gemm_handle_t h);

/*
 * C = A·B on `stream` (device pointers; see the semantics above).
 * Asynchronous: returns once the work is queued.  A, B and C must stay valid
 * until the stream has executed it.  For GEMM_F32/GEMM_TF32, A, B and C are
 * float*; for GEMM_BF16, A and B point to bfloat16 values.  A and B must be
 * aligned to their element size, C to 4 bytes (else GEMM_ERR_ALIGNMENT).
 * Operands whose pointer or leading dimension is not a multiple of 16 bytes
 * are first re-packed into the handle's workspace by a device kernel (part of
 * the queued work).  A wait that expires inside a kernel is reported by
 * gemm_sync_status, not here.
 */
int gemm_run(gemm_handle_t h, int layout_b, int64_t M, int64_t N, int64_t K,
             const void *A, int64_t lda, const void *B, int64_t ldb,
             float *C, int64_t ldc, int dtype, cudaStream_t stream);

/*
 * As gemm_run, but A, B and C are HOST pointers.  The call stages A and B in
 * the handle's workspace, runs the GEMM and copies C back, and returns
 * without waiting: the host buffers must stay valid and C must not be read
 * until `stream` has been synchronised.  For large problems C is computed in
 * blocks (row panels of A times column panels of B, each a whole number of
 * persistent waves), and the copies of the next block's operands in and the
 * previous block's C out run on two internal streams of the handle while a
 * block computes; events order the copies after the work already queued on
 * `stream` and make `stream` wait for the last copy, so the call behaves as
 * one operation on `stream`.  Each block is a GEMM over the whole of K, but
 * a block's partial last wave may be cut along K (slices or stream-K) where
 * one call over the whole of C would cut other tiles, or none: the result
 * then differs from gemm_run's by rounding only (the mode's tolerance), and
 * is bit-identical where neither cuts a tile along K and on integer data.
 * Pinned (page-locked) host memory makes the copies asynchronous; pageable
 * memory works but the copies block.
 */
int gemm_run_host(gemm_handle_t h, int layout_b, int64_t M, int64_t N, int64_t K,
                  const void *A_host, int64_t lda, const void *B_host, int64_t ldb,
                  float *C_host, int64_t ldc, int dtype, cudaStream_t stream);

/*
 * Check the arguments of a run without touching the GPU: returns GEMM_OK,
 * GEMM_ERR_INVALID or GEMM_ERR_ALIGNMENT exactly as gemm_run would.
 */
int gemm_validate(int layout_b, int64_t M, int64_t N, int64_t K,
                  const void *A, int64_t lda, const void *B, int64_t ldb,
                  const float *C, int64_t ldc, int dtype);

/*
 * Wait for `stream`, then read and clear the handle's device status word.
 * Returns GEMM_OK, GEMM_ERR_TIMEOUT when an in-kernel wait expired since the
 * last check (the kernel then left C incomplete and returned), or
 * GEMM_ERR_CUDA when the stream reports an error.
 */
int gemm_sync_status(gemm_handle_t h, cudaStream_t stream);

/* Set an option (GEMM_OPT_*).  Returns GEMM_ERR_INVALID for an unknown
 * option or an out-of-range value. */
int gemm_set_option(gemm_handle_t h, int option, int64_t value);

/* Human-readable description of the last failure on `h` ("" if none). */
const char *gemm_last_error_string(gemm_handle_t h);

/* Name of a GEMM_OK / GEMM_ERR_* code. */
const char *gemm_status_string(int code);

/* Name of the kernel path the last successful run on `h` queued, e.g.
 * "simt_f32_128x128_rowB" or "tc_bf16_128x256_rowB+repack". */
const char *gemm_last_path(gemm_handle_t h);

/* Number of kernels this handle has launched so far (all paths). */
int64_t gemm_launch_count(gemm_handle_t h);

/* GEMM_VERSION of the library. */
int gemm_version(void);

/*
 * C = A·B without allocating anything.  The pages have no counterpart of this
 * entry point; it exists for callers that cannot call cudaMalloc: code whose
 * device memory is owned by a framework's memory manager (every allocation
 * must go through it, or the budget is reserved up front), and
 * latency-critical threads that must not take cudaMalloc's implicit device
 * synchronisation.  gemm_create and gemm_run allocate, so they are not usable
 * there.
 *
 * Arguments, semantics, errors and asynchrony are those of gemm_run, without
 * the handle: the call runs on the calling thread's current device, and
 * `stream` must belong to that device.  Operands whose address or pitch is
 * not a multiple of 16 bytes are re-packed into a scratch array of
 * GEMM_NOALLOC_SCRATCH_BYTES that the library reserves as a static device
 * array on every GPU that loads it, until the process exits.  When the
 * re-packed A and B together need more than that, the call returns
 * GEMM_ERR_INVALID and launches nothing (aligned operands need no scratch and
 * have no such limit).  GEMM_F32_3XTF32, whose split operands always need
 * workspace, is refused the same way.
 *
 * The first call on a device does a one-time set-up there (device check,
 * kernel attributes, lookup of the scratch array's device address); make
 * that first call before any stream capture.  All calls on a device share
 * the scratch array and it keeps the last call's contents; nothing in it has
 * to start at zero, because each call writes every element it reads.  Calls
 * that overlap on the GPU (unordered streams, or several host threads) race
 * on the array: order them.  An in-kernel wait that expires ends the kernel
 * with C incomplete and sets a per-device status word (a static device
 * variable beside the scratch array); gemm_noalloc_sync_status reports it.
 * The call makes no cudaMalloc, cudaFree or other allocating call.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int gemm_run_noalloc(int layout_b, int64_t M, int64_t N, int64_t K,
                     const void *A, int64_t lda, const void *B, int64_t ldb,
                     float *C, int64_t ldc, int dtype, cudaStream_t stream);

/*
 * Status of the allocation-free calls on the current device: waits for
 * `stream`, then returns GEMM_ERR_TIMEOUT if an in-kernel wait of an earlier
 * gemm_run_noalloc call on this device expired (C of that call is
 * incomplete) and clears the report, else GEMM_OK.  The status word is shared
 * by every allocation-free call on the device, whatever its stream.
 * Allocates nothing (a 4-byte device-to-host copy).
 */
int gemm_noalloc_sync_status(cudaStream_t stream);

/*
 * Process-wide settings of the allocation-free calls (they have no handle):
 * GEMM_OPT_WAIT_TIMEOUT_NS (limit of every in-kernel wait, 1e6..6e10 ns,
 * default 4e9) and the test hook GEMM_OPT_DEBUG_DROP_LOAD (0 or 1, as for a
 * handle).  Other options are GEMM_ERR_INVALID.  Applies to later calls.
 */
int gemm_noalloc_set_option(int option, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_SM100_GB300_GEMM_H */
