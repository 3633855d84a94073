// Small bandwidth-bound helpers of the GEMM path.
//
//  * repack: copies an operand whose base address or leading dimension is not
//    a multiple of 16 bytes into a workspace with a 16-byte-multiple leading
//    dimension, so the GEMM kernels can read it with TMA (a TMA tensor needs
//    16-byte aligned rows).  One CTA walks whole rows: reads and writes are
//    both row-contiguous, so every warp access is coalesced ("PMPP Chapter 06:
//    Performance considerations", section 1, coalescing).
//  * tile split reduction: C = the K-slice partial tiles of the tensor-core
//    kernels added in slice order ("GEMM 性能优化", 台阶 1: partial sums over K
//    slices add up to the product).
//  * zero fill: C = 0 for K = 0 (the empty sum).
//  * three-part split of an FP32 operand for the FP32-accurate tensor-core
//    mode: x = hi + lo with hi = x with its low 13 mantissa bits cleared (a
//    TF32 value, exactly what the tensor core reads of hi) and lo = x - hi
//    (exact in FP32).  The operand is written three times along K, so one
//    TF32 product over 3K gives hi(A)hi(B) + hi(A)lo(B) + lo(A)hi(B), which
//    is A·B up to the lo(A)lo(B) term (about 2^-22 of |a·b|).
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

// x split into its TF32 part and the FP32 rest.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo)
{
    hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    lo = x - hi;
}

// K runs along the rows (`along_rows` = 0: A, or column-major B, K is the
// contiguous dimension) or down the columns (1: row-major B, K counts rows).
// Part p of 3 of the output holds hi, hi, lo (first = 0: A) or hi, lo, hi
// (first = 1: B), so the K-concatenated product pairs hi(A) with hi(B) and
// lo(B), and lo(A) with hi(B).  One thread per input element, rows walked by
// CTAs, columns by threads (coalesced reads and writes).
__global__ void __launch_bounds__(256) split3_kernel(const float *__restrict__ src, long long lds,
                                                     float *__restrict__ dst, long long ldd, long long rows,
                                                     long long cols, int along_rows, int b_side)
{
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *sr = src + r * lds;
        for (long long c = threadIdx.x; c < cols; c += blockDim.x) {
            float hi, lo;
            split_tf32(sr[c], hi, lo);
            const float p0 = hi, p1 = b_side ? lo : hi, p2 = b_side ? hi : lo;
            if (along_rows) {  // K = rows: parts are row blocks
                dst[r * ldd + c] = p0;
                dst[(r + rows) * ldd + c] = p1;
                dst[(r + 2 * rows) * ldd + c] = p2;
            } else {  // K = cols: parts are column blocks of one row
                float *dr = dst + r * ldd;
                dr[c] = p0;
                dr[c + cols] = p1;
                dr[c + 2 * cols] = p2;
            }
        }
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

// One thread per 4 consecutive columns of a tile row; slices added in order.
__global__ void __launch_bounds__(256) tile_split_reduce_kernel(const float *__restrict__ P, int splits,
                                                                long long tiles_m, long long tiles_n, int bm,
                                                                int bn, float *__restrict__ C, long long ldc,
                                                                long long M, long long N, int c_vec4)
{
    const long long tile = (long long)bm * bn;
    const long long quads = tiles_m * tiles_n * (tile / 4);
    const long long slice = tiles_m * tiles_n * tile;
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < quads;
         q += (long long)gridDim.x * blockDim.x) {
        const long long t = q / (tile / 4);
        const long long e = (q - t * (tile / 4)) * 4;
        const long long mb = t / tiles_n, nb = t - (t / tiles_n) * tiles_n;
        const long long m = mb * bm + e / bn;
        const long long n = nb * bn + e % bn;
        if (m >= M || n >= N) continue;
        const float *src = P + t * tile + e;
        float4 acc = *reinterpret_cast<const float4 *>(src);
        for (int s = 1; s < splits; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(src + s * slice);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        float *c = C + m * ldc + n;
        if (c_vec4 && n + 3 < N) {
            *reinterpret_cast<float4 *>(c) = acc;
        } else {
            c[0] = acc.x;
            if (n + 1 < N) c[1] = acc.y;
            if (n + 2 < N) c[2] = acc.z;
            if (n + 3 < N) c[3] = acc.w;
        }
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

cudaError_t launch_split3(const float *src, int64_t lds, float *dst, int64_t ldd, int64_t rows, int64_t cols,
                          bool along_rows, bool b_side, int sm_count, cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    split3_kernel<<<rows_grid(rows, sm_count), 256, 0, stream>>>(src, lds, dst, ldd, rows, cols, along_rows ? 1 : 0,
                                                                 b_side ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_tile_split_reduce(const float *partials, int splits, int64_t tiles_m, int64_t tiles_n, int bm,
                                     int bn, float *C, int64_t ldc, int64_t M, int64_t N, bool c_vec4, int sm_count,
                                     cudaStream_t stream)
{
    if (M <= 0 || N <= 0 || splits < 1) return cudaSuccess;
    const long long quads = tiles_m * tiles_n * ((long long)bm * bn / 4);
    long long blocks = (quads + 255) / 256;
    const long long cap = 8LL * (sm_count > 0 ? sm_count : 1);
    if (blocks > cap) blocks = cap;
    tile_split_reduce_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(partials, splits, tiles_m, tiles_n, bm, bn,
                                                                            C, ldc, M, N, c_vec4 ? 1 : 0);
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
