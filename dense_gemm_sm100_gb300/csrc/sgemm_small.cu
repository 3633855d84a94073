// FP32 GEMM for small problems: a few 32 x 32 tiles of C and a short K.
//
// The persistent TMA kernels (sgemm_simt.cu) give each thread an 8 x 8 (or
// wider) tile of C, so a problem of a handful of tiles leaves most of the GPU
// idle and each thread runs a long chain of multiply-adds ("GEMM 性能优化",
// Wave 模型: an under-filled launch is bounded by one CTA's serial work).
// This kernel cuts C into 32 x 32 tiles, one per CTA of 1024 threads, and
// shortens the CTA's serial work four ways: the threads form four K groups,
// each multiplying a quarter of every staged K chunk into 2 x 2 outputs per
// thread, and the groups' partial tiles are added in group order at the end
// ("GEMM 性能优化", 台阶 1: K may be cut into slices whose partial products
// add up to the product).  A and B go through shared memory 128 K at a time
// (台阶 1: shared-memory tiling), each thread keeps its outputs in registers
// (台阶 2: thread tiling), and the next chunk's global loads are in flight
// while the current one is multiplied (台阶 6, double buffering in
// registers).  Each operand is staged in its own orientation, A and
// column-major B K-contiguous and row-major B N-contiguous, so staging is a
// straight copy and the multiply reads 16-byte vectors along K (8-byte pairs
// along N for row-major B) ("PMPP Chapter 06: Performance considerations",
// §1: a column-major B is read along its contiguous K direction).  Any pitch
// and alignment: 16-byte loads where the rows allow, else element loads;
// zero fill outside the matrices.
#include <cstdint>

#include "gemm_internal.h"

namespace dg {
namespace {

constexpr int SB = 32;       // tile rows and columns
constexpr int KC = 128;      // K per staged chunk
constexpr int KG = 4;        // K groups
constexpr int KQ = KC / KG;  // K per group per chunk
constexpr int ST = 1024;     // threads: KG groups of 16 x 16, each thread 2 x 2 outputs
constexpr int PK = KC + 4;   // pitch of K-contiguous rows: 16-byte aligned; rows 2 apart
                             // start in different 16-byte bank groups

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
    // As[m * PK + k]: the chunk's 32 rows of A.  Bs: row-major B as
    // [k * SB + n] (KC x 32), column-major B as [n * PK + k] (32 x KC).  After
    // the last chunk the same storage holds the K groups' partial tiles.
    __shared__ __align__(16) float smem[2 * SB * PK];
    float *As = smem;
    float *Bs = smem + SB * PK;
    const int tid = threadIdx.x;
    const long long m0 = (long long)blockIdx.y * SB;
    const int n0 = blockIdx.x * SB;
    // loads, one float4 of A and one of B per thread per chunk: A (and
    // column-major B) line lr, K offset lk; row-major B K row bk, columns bn
    const int lr = tid >> 5, lk = (tid & 31) * 4;
    const int bk = tid >> 3, bn = (tid & 7) * 4;
    // multiply: K group kg (K offsets kg * KQ .. + KQ - 1 of each chunk), rows
    // 2ty and 2ty + 1, columns 2tx and 2tx + 1 (row-major B) or tx and tx + 16
    // (column-major B: 16 K-contiguous rows in distinct bank groups per load)
    const int kg = tid >> 8, ty = (tid >> 4) & 15, tx = tid & 15;
    const int c0 = LAYOUT_B == 0 ? 2 * tx : tx;
    const int c1 = LAYOUT_B == 0 ? 2 * tx + 1 : tx + 16;

    auto load_a = [&](int k0) { return load4<VEC>(A, lda, m0 + lr, M, k0 + lk, K); };
    auto load_b = [&](int k0) {
        if (LAYOUT_B == 0) return load4<VEC>(B + n0, ldb, (long long)k0 + bk, K, bn, N - n0);
        return load4<VEC>(B, ldb, (long long)n0 + lr, N, k0 + lk, K);
    };

    float acc00 = 0.0f, acc01 = 0.0f, acc10 = 0.0f, acc11 = 0.0f;
    float4 ra = load_a(0), rb = load_b(0);
    for (int k0 = 0; k0 < K; k0 += KC) {
        *reinterpret_cast<float4 *>(&As[lr * PK + lk]) = ra;
        if (LAYOUT_B == 0)
            *reinterpret_cast<float4 *>(&Bs[bk * SB + bn]) = rb;
        else
            *reinterpret_cast<float4 *>(&Bs[lr * PK + lk]) = rb;
        __syncthreads();
        if (k0 + KC < K) {  // the next chunk's loads fly while this one is multiplied
            ra = load_a(k0 + KC);
            rb = load_b(k0 + KC);
        }
        const float *a0p = &As[2 * ty * PK + kg * KQ];
        const float *a1p = a0p + PK;
#pragma unroll
        for (int kk = 0; kk < KQ; kk += 4) {
            const float4 a0 = *reinterpret_cast<const float4 *>(a0p + kk);
            const float4 a1 = *reinterpret_cast<const float4 *>(a1p + kk);
            float b0[4], b1[4];
            if (LAYOUT_B == 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 v = *reinterpret_cast<const float2 *>(&Bs[(kg * KQ + kk + j) * SB + c0]);
                    b0[j] = v.x;
                    b1[j] = v.y;
                }
            } else {
                const float4 v0 = *reinterpret_cast<const float4 *>(&Bs[c0 * PK + kg * KQ + kk]);
                const float4 v1 = *reinterpret_cast<const float4 *>(&Bs[c1 * PK + kg * KQ + kk]);
                b0[0] = v0.x, b0[1] = v0.y, b0[2] = v0.z, b0[3] = v0.w;
                b1[0] = v1.x, b1[1] = v1.y, b1[2] = v1.z, b1[3] = v1.w;
            }
            const float x0[4] = {a0.x, a0.y, a0.z, a0.w};
            const float x1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // k order within the group
                acc00 = fmaf(x0[j], b0[j], acc00);
                acc01 = fmaf(x0[j], b1[j], acc01);
                acc10 = fmaf(x1[j], b0[j], acc10);
                acc11 = fmaf(x1[j], b1[j], acc11);
            }
        }
        __syncthreads();
    }
    // The K groups' partial tiles, red[g][m][n], then their sum in group
    // order, one output per thread, rows of 32 consecutive columns per warp.
    float *red = smem;
    red[(kg * SB + 2 * ty) * SB + c0] = acc00;
    red[(kg * SB + 2 * ty) * SB + c1] = acc01;
    red[(kg * SB + 2 * ty + 1) * SB + c0] = acc10;
    red[(kg * SB + 2 * ty + 1) * SB + c1] = acc11;
    __syncthreads();
    const int om = tid >> 5, on = tid & 31;
    float c = red[om * SB + on];
#pragma unroll
    for (int g = 1; g < KG; ++g) c += red[(g * SB + om) * SB + on];
    const long long m = m0 + om;
    const int n = n0 + on;
    if (m < M && n < N) C[m * ldc + n] = c;
}

static_assert(SB * KC / 4 == ST, "staging: one float4 of A and one of B per thread per chunk");
static_assert(KC / 4 == 32 && SB / 4 == 8, "load indices lr, lk, bk, bn");
static_assert(KG * 256 == ST && KQ % 4 == 0, "K groups of 16 x 16 threads, float4 steps along K");
static_assert(KG * SB * SB <= 2 * SB * PK, "partial tiles fit in the staging storage");

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
    // 384 along K.  Measured per call in CUDA-graph replays: 128^3 3.4 us
    // against 8.0 for the 64 x 64 persistent kernel and 4.4 for cuBLAS
    // (column-major B 3.6 against 11.9), 256^3 5.6 against 8.8, 256 x 256 x
    // 384 7.5 against 8.8, 384^3 7.6 against 9.3; from K = 512 the persistent
    // kernels' K split wins (256 x 256 x 512 9.4 against 8.8, 256 x 256 x
    // 1024 17.0 against 9.2).
    const int64_t tiles = ((M + SB - 1) / SB) * ((N + SB - 1) / SB);
    return M > 0 && N > 0 && K > 0 && K <= 384 && tiles <= sm_count;
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
