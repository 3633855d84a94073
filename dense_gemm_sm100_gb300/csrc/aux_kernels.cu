// Small bandwidth-bound helpers of the GEMM path.
//
//  * repack: copies an operand whose base address or leading dimension is not
//    a multiple of 16 bytes into a workspace with a 16-byte-multiple leading
//    dimension, so the GEMM kernels can read it with TMA (a TMA tensor needs
//    16-byte aligned rows).  One CTA walks whole rows: reads and writes are
//    both row-contiguous, so every warp access is coalesced ("PMPP Chapter 06:
//    Performance considerations", section 1, coalescing).
//  * zero fill: C = 0 for K = 0 (the empty sum).
#include <cstdint>

#include "gemm_internal.h"

namespace dg {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) repack_rows_kernel(const T *__restrict__ src, long long lds,
                                                          T *__restrict__ dst, long long ldd,
                                                          long long rows, long long cols)
{
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const T *s = src + r * lds;
        T *d = dst + r * ldd;
        for (long long c = threadIdx.x; c < cols; c += blockDim.x) d[c] = s[c];
    }
}

__global__ void __launch_bounds__(256) zero_fill_kernel(float *__restrict__ C, long long ldc,
                                                        long long M, long long N)
{
    for (long long r = blockIdx.x; r < M; r += gridDim.x) {
        float *c = C + r * ldc;
        for (long long j = threadIdx.x; j < N; j += blockDim.x) c[j] = 0.0f;
    }
}

int rows_grid(long long rows, int sm_count)
{
    const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;
    return static_cast<int>(rows < cap ? rows : cap);
}

}  // namespace

cudaError_t launch_repack(const void *src, int64_t lds, void *dst, int64_t ldd, int64_t rows,
                          int64_t cols, int elem_bytes, int sm_count, cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int grid = rows_grid(rows, sm_count);
    if (elem_bytes == 4)
        repack_rows_kernel<uint32_t><<<grid, 256, 0, stream>>>(
            static_cast<const uint32_t *>(src), lds, static_cast<uint32_t *>(dst), ldd, rows, cols);
    else
        repack_rows_kernel<uint16_t><<<grid, 256, 0, stream>>>(
            static_cast<const uint16_t *>(src), lds, static_cast<uint16_t *>(dst), ldd, rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(float *C, int64_t ldc, int64_t M, int64_t N, int sm_count,
                             cudaStream_t stream)
{
    if (M <= 0 || N <= 0) return cudaSuccess;
    zero_fill_kernel<<<rows_grid(M, sm_count), 256, 0, stream>>>(C, ldc, M, N);
    return cudaGetLastError();
}

}  // namespace dg
