// FP32 GEMM for small problems: a few 32 x 32 tiles of C and a short K.
//
// The persistent TMA kernels (sgemm_simt.cu) give each thread an 8 x 8 (or
// wider) tile of C, so a problem of a handful of tiles leaves most of the GPU
// idle and each thread runs a long chain of multiply-adds ("GEMM 性能优化",
// Wave 模型: an under-filled launch is bounded by one CTA's serial work).
// This kernel cuts C into 32 x 32 tiles, one per CTA of 256 threads, each
// thread owning 2 x 2 outputs, and stages A and B through shared memory one
// 32-wide K step at a time ("GEMM 性能优化", 台阶 2: shared-memory tiling),
// with the next step's global loads in flight while the current one is
// multiplied (台阶 6, double buffering in registers).  A is read along its
// rows and written to shared memory K-major; B, row-major or column-major, is
// read along its contiguous direction and turned in shared memory where
// needed ("PMPP Chapter 06: Performance considerations", §1, corner
// turning).  Any pitch and alignment: 16-byte loads where the rows allow,
// else element loads; zero fill outside the matrices.
#include <cstdint>

#include "gemm_internal.h"

namespace dg {
namespace {

constexpr int SB = 32;    // tile rows and columns
constexpr int SBK = 32;   // K per step
constexpr int ST = 256;   // threads: 16 x 16, each 2 x 2 outputs

// Four consecutive elements of row `r` (length `len`, pitch `ld`) starting at
// column `c`, zero past the end.  VEC: the row start and pitch are 16-byte
// aligned, so a whole in-range group is one 16-byte load.
template <bool VEC>
__device__ __forceinline__ float4 load4(const float *__restrict__ P, long long ld, long long r, long long rows, int c,
                                        int len)
{
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (r >= rows) return v;
    const float *row = P + r * ld;
    if (VEC && c + 3 < len) return *reinterpret_cast<const float4 *>(row + c);
    if (c < len) v.x = row[c];
    if (c + 1 < len) v.y = row[c + 1];
    if (c + 2 < len) v.z = row[c + 2];
    if (c + 3 < len) v.w = row[c + 3];
    return v;
}

template <int LAYOUT_B, bool VEC>
__global__ void __launch_bounds__(ST) sgemm_small_kernel(const float *__restrict__ A, long long lda,
                                                         const float *__restrict__ B, long long ldb,
                                                         float *__restrict__ C, long long ldc, int M, int N, int K)
{
    __shared__ float As[SBK][SB + 1];  // As[k][m]: a K step of the tile's rows
    __shared__ __align__(16) float Bs[SBK][SB + 4];  // Bs[k][n]: rows of 36 floats keep 16-byte stores aligned
    const int tid = threadIdx.x;
    const long long m0 = (long long)blockIdx.y * SB;
    const int n0 = blockIdx.x * SB;
    const int ty = tid >> 4, tx = tid & 15;  // outputs: rows 2ty, 2ty + 1; columns 2tx, 2tx + 1
    const int lr = tid >> 3, lc = tid & 7;   // loads: line lr, elements 4lc .. 4lc + 3

    // A: row m0 + lr, k0 + 4lc.  B row-major: row k0 + lr, columns n0 + 4lc;
    // column-major: column n0 + lr (a row of the N x K storage), k0 + 4lc.
    auto load_a = [&](int k0) { return load4<VEC>(A, lda, m0 + lr, M, k0 + 4 * lc, K); };
    auto load_b = [&](int k0) {
        if (LAYOUT_B == 0) return load4<VEC>(B + n0, ldb, (long long)k0 + lr, K, 4 * lc, N - n0);
        return load4<VEC>(B, ldb, (long long)n0 + lr, N, k0 + 4 * lc, K);
    };

    float acc00 = 0.0f, acc01 = 0.0f, acc10 = 0.0f, acc11 = 0.0f;
    float4 ra = load_a(0), rb = load_b(0);
    for (int k0 = 0; k0 < K; k0 += SBK) {
        // stage this step: A (and column-major B) turned to K-major
        As[4 * lc + 0][lr] = ra.x;
        As[4 * lc + 1][lr] = ra.y;
        As[4 * lc + 2][lr] = ra.z;
        As[4 * lc + 3][lr] = ra.w;
        if (LAYOUT_B == 0) {
            *reinterpret_cast<float4 *>(&Bs[lr][4 * lc]) = rb;
        } else {
            Bs[4 * lc + 0][lr] = rb.x;
            Bs[4 * lc + 1][lr] = rb.y;
            Bs[4 * lc + 2][lr] = rb.z;
            Bs[4 * lc + 3][lr] = rb.w;
        }
        __syncthreads();
        if (k0 + SBK < K) {  // the next step's loads fly while this one is multiplied
            ra = load_a(k0 + SBK);
            rb = load_b(k0 + SBK);
        }
#pragma unroll
        for (int k = 0; k < SBK; ++k) {
            const float a0 = As[k][2 * ty], a1 = As[k][2 * ty + 1];
            const float b0 = Bs[k][2 * tx], b1 = Bs[k][2 * tx + 1];
            acc00 = fmaf(a0, b0, acc00);
            acc01 = fmaf(a0, b1, acc01);
            acc10 = fmaf(a1, b0, acc10);
            acc11 = fmaf(a1, b1, acc11);
        }
        __syncthreads();
    }
    const long long m = m0 + 2 * ty;
    const int n = n0 + 2 * tx;
    if (m < M) {
        if (n < N) C[m * ldc + n] = acc00;
        if (n + 1 < N) C[m * ldc + n + 1] = acc01;
    }
    if (m + 1 < M) {
        if (n < N) C[(m + 1) * ldc + n] = acc10;
        if (n + 1 < N) C[(m + 1) * ldc + n + 1] = acc11;
    }
}

template <int L, bool V>
cudaError_t launch(const float *A, int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc, int M, int N,
                   int K, cudaStream_t stream)
{
    const dim3 grid(static_cast<unsigned>((N + SB - 1) / SB), static_cast<unsigned>((M + SB - 1) / SB), 1);
    sgemm_small_kernel<L, V><<<grid, ST, 0, stream>>>(A, lda, B, ldb, C, ldc, M, N, K);
    return cudaGetLastError();
}

}  // namespace

bool simt_small_fits(int64_t M, int64_t N, int64_t K, int sm_count)
{
    // A few tiles and a short K: at most one 32 x 32 tile per SM and at most
    // 256 along K.  Measured per call in CUDA-graph replays: 128^3 4.3 us
    // against 8.4 for the 64 x 64 persistent kernel (column-major B 4.0
    // against 13.3), 256^3 7.6 against 8.8; with K = 384 or more the
    // persistent kernels' K split wins (384^3 9.5 against 10.6, 256 x 256 x
    // 1024 9.5 against 25.6).
    const int64_t tiles = ((M + SB - 1) / SB) * ((N + SB - 1) / SB);
    return M > 0 && N > 0 && K > 0 && K <= 256 && tiles <= sm_count;
}

cudaError_t launch_simt_small(int layout_b, const float *A, int64_t lda, const float *B, int64_t ldb, float *C,
                              int64_t ldc, int M, int N, int K, cudaStream_t stream)
{
    if ((M + SB - 1) / SB > 65535) return cudaErrorInvalidValue;  // grid rows
    const bool vec = (reinterpret_cast<uintptr_t>(A) & 15) == 0 && (reinterpret_cast<uintptr_t>(B) & 15) == 0 &&
                     lda % 4 == 0 && ldb % 4 == 0;
    if (layout_b == 0)
        return vec ? launch<0, true>(A, lda, B, ldb, C, ldc, M, N, K, stream)
                   : launch<0, false>(A, lda, B, ldb, C, ldc, M, N, K, stream);
    return vec ? launch<1, true>(A, lda, B, ldb, C, ldc, M, N, K, stream)
               : launch<1, false>(A, lda, B, ldb, C, ldc, M, N, K, stream);
}

}  // namespace dg
