// The optimisation ladder of "GEMM 性能优化" (八个台阶) and the two worked
// kernels of "PMPP Chapter 06: Performance considerations", written for
// sm_103a as a labelled benchmark suite.  None of these kernels is on the
// library's GEMM path; they exist to measure each step of the pages' ladder
// on GB300 (as % of cuBLAS) and to check the pages' global-traffic formulas
// against ncu counters.  All compute C = A·B with A, B, C row-major (tight
// pitches), except the corner-turning kernel, whose B is column-major.
//
//   1 naive            one thread per C element, operands from global memory
//   2 smem tiling      32x32 tiles along K in shared memory (台阶 1)
//   3 thread tiling    128x128 tile, 8x8 register outer product (台阶 2)
//   4 vectorised       float4 global loads, A stored transposed (台阶 3)
//   5 conflict-free    padded A tile, split B columns (台阶 4)
//   6 warp tiling      4x8 lanes per warp (台阶 5)
//   7 double buffer    two shared buffers + register prefetch (台阶 6)
//   8 multistage       cp.async 3-stage pipeline (台阶 7)
//   101 PMPP corner turning   16x16 tiles, column-major B loaded along K
//   102 PMPP coarsening       32x32 tiles, 4 output tiles per block
#include <cstdint>

#include "../../include/gemm.h"
#include "../../include/gemm_ladder.h"

namespace {

// ---------------------------------------------------------------- step 1
__global__ void __launch_bounds__(256) k_naive(const float *__restrict__ A, const float *__restrict__ B,
                                               float *__restrict__ C, int M, int N, int K)
{
    const int col = blockIdx.x * 32 + threadIdx.x;
    const int row = blockIdx.y * 8 + threadIdx.y;
    if (row >= M || col >= N) return;
    float acc = 0.0f;
    for (int k = 0; k < K; ++k) acc = fmaf(A[(long long)row * K + k], B[(long long)k * N + col], acc);
    C[(long long)row * N + col] = acc;
}

// ---------------------------------------------------------------- step 2
// Square tiles of T along K; out-of-range elements load as zero.
template <int T>
__global__ void __launch_bounds__(T *T) k_tiled(const float *__restrict__ A, const float *__restrict__ B,
                                                float *__restrict__ C, int M, int N, int K)
{
    __shared__ float As[T][T];
    __shared__ float Bs[T][T];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int row = blockIdx.y * T + ty, col = blockIdx.x * T + tx;
    float acc = 0.0f;
    for (int k0 = 0; k0 < K; k0 += T) {
        As[ty][tx] = (row < M && k0 + tx < K) ? A[(long long)row * K + k0 + tx] : 0.0f;
        Bs[ty][tx] = (k0 + ty < K && col < N) ? B[(long long)(k0 + ty) * N + col] : 0.0f;
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < T; ++kk) acc = fmaf(As[ty][kk], Bs[kk][tx], acc);
        __syncthreads();
    }
    if (row < M && col < N) C[(long long)row * N + col] = acc;
}

// ---------------------------------------------------------------- steps 3-7
// 128x128 tile, BK = 8, 256 threads, 8x8 per thread.  M, N multiples of 128,
// K a multiple of 8.
constexpr int LBM = 128, LBN = 128, LBK = 8;

// step 3: scalar loads, A kept row-major in shared memory
__global__ void __launch_bounds__(256) k_thread_tile(const float *__restrict__ A, const float *__restrict__ B,
                                                     float *__restrict__ C, int M, int N, int K)
{
    __shared__ float As[LBM][LBK];
    __shared__ float Bs[LBK][LBN];
    const int t = threadIdx.x, tx = t % 16, ty = t / 16;
    const float *Ab = A + (long long)blockIdx.y * LBM * K;
    const float *Bb = B + (long long)blockIdx.x * LBN;
    float acc[8][8] = {};
    for (int k0 = 0; k0 < K; k0 += LBK) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = t + 256 * r;  // 1024 elements of each tile
            As[e / LBK][e % LBK] = Ab[(long long)(e / LBK) * K + k0 + e % LBK];
            Bs[e / LBN][e % LBN] = Bb[(long long)(k0 + e / LBN) * N + e % LBN];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < LBK; ++k) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = As[ty * 8 + i][k];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = Bs[k][tx * 8 + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *Cb = C + (long long)(blockIdx.y * LBM + ty * 8) * N + blockIdx.x * LBN + tx * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) Cb[(long long)i * N + j] = acc[i][j];
}

// Steps 4-6 share one body:
//   PAD  = padding of the transposed A tile (step 5 removes conflicts)
//   SPLIT: a thread's 8 columns are two float4 64 apart instead of 8
//          consecutive (step 5)
//   WARP: threads laid out as 4x8 lanes per warp, 2x4 warps (step 6)
template <int PAD, bool SPLIT, bool WARP>
__global__ void __launch_bounds__(256) k_vec(const float *__restrict__ A, const float *__restrict__ B,
                                             float *__restrict__ C, int M, int N, int K)
{
    __shared__ __align__(16) float As[LBK][LBM + PAD];  // A transposed: As[k][m]
    __shared__ __align__(16) float Bs[LBK][LBN];
    const int t = threadIdx.x;
    int tx, ty;  // thread's column group (0..15) and row group (0..15)
    if (WARP) {
        const int warp = t / 32, lane = t % 32;
        ty = (warp / 4) * 8 + (lane / 8) * 2 + 0;  // rows: 2 warp rows x 4 lane rows x 2
        tx = (warp % 4) * 4 + (lane % 8) / 2;
        ty += lane % 2;
    } else {
        tx = t % 16;
        ty = t / 16;
    }
    const float *Ab = A + (long long)blockIdx.y * LBM * K;
    const float *Bb = B + (long long)blockIdx.x * LBN;
    // one float4 of A (row t/2, k-half t%2) and one of B (row t/32, cols 4*(t%32))
    const int ar = t / 2, ac = (t % 2) * 4;
    const int br = t / 32, bc = (t % 32) * 4;
    float acc[8][8] = {};
    for (int k0 = 0; k0 < K; k0 += LBK) {
        const float4 av = *reinterpret_cast<const float4 *>(Ab + (long long)ar * K + k0 + ac);
        const float4 bv = *reinterpret_cast<const float4 *>(Bb + (long long)(k0 + br) * N + bc);
        As[ac + 0][ar] = av.x;
        As[ac + 1][ar] = av.y;
        As[ac + 2][ar] = av.z;
        As[ac + 3][ar] = av.w;
        *reinterpret_cast<float4 *>(&Bs[br][bc]) = bv;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < LBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[k][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[k][ty * 8 + 4]);
            float4 b0, b1;
            if (SPLIT) {
                b0 = *reinterpret_cast<const float4 *>(&Bs[k][tx * 4]);
                b1 = *reinterpret_cast<const float4 *>(&Bs[k][tx * 4 + 64]);
            } else {
                b0 = *reinterpret_cast<const float4 *>(&Bs[k][tx * 8]);
                b1 = *reinterpret_cast<const float4 *>(&Bs[k][tx * 8 + 4]);
            }
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    const long long r0 = (long long)blockIdx.y * LBM + ty * 8;
    const int c0 = blockIdx.x * LBN;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float *crow = C + (r0 + i) * N + c0;
        if (SPLIT) {
            *reinterpret_cast<float4 *>(crow + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            *reinterpret_cast<float4 *>(crow + tx * 4 + 64) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        } else {
            *reinterpret_cast<float4 *>(crow + tx * 8) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            *reinterpret_cast<float4 *>(crow + tx * 8 + 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
    }
}

// step 7: step 6 plus two shared-memory buffers (the next tile is fetched into
// registers while the current one is multiplied) and fragment double
// buffering across k
__global__ void __launch_bounds__(256) k_double_buffer(const float *__restrict__ A, const float *__restrict__ B,
                                                       float *__restrict__ C, int M, int N, int K)
{
    constexpr int PAD = 4;
    __shared__ __align__(16) float As[2][LBK][LBM + PAD];
    __shared__ __align__(16) float Bs[2][LBK][LBN];
    const int t = threadIdx.x;
    const int warp = t / 32, lane = t % 32;
    const int ty = (warp / 4) * 8 + (lane / 8) * 2 + lane % 2;
    const int tx = (warp % 4) * 4 + (lane % 8) / 2;
    const float *Ab = A + (long long)blockIdx.y * LBM * K;
    const float *Bb = B + (long long)blockIdx.x * LBN;
    const int ar = t / 2, ac = (t % 2) * 4;
    const int br = t / 32, bc = (t % 32) * 4;
    auto stash = [&](int buf, const float4 &av, const float4 &bv) {
        As[buf][ac + 0][ar] = av.x;
        As[buf][ac + 1][ar] = av.y;
        As[buf][ac + 2][ar] = av.z;
        As[buf][ac + 3][ar] = av.w;
        *reinterpret_cast<float4 *>(&Bs[buf][br][bc]) = bv;
    };
    float acc[8][8] = {};
    float4 av = *reinterpret_cast<const float4 *>(Ab + (long long)ar * K + ac);
    float4 bv = *reinterpret_cast<const float4 *>(Bb + (long long)br * N + bc);
    stash(0, av, bv);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += LBK) {
        const bool more = k0 + LBK < K;
        if (more) {
            av = *reinterpret_cast<const float4 *>(Ab + (long long)ar * K + k0 + LBK + ac);
            bv = *reinterpret_cast<const float4 *>(Bb + (long long)(k0 + LBK + br) * N + bc);
        }
        float4 fa[2][2], fb[2][2];
        fa[0][0] = *reinterpret_cast<const float4 *>(&As[buf][0][ty * 8]);
        fa[0][1] = *reinterpret_cast<const float4 *>(&As[buf][0][ty * 8 + 4]);
        fb[0][0] = *reinterpret_cast<const float4 *>(&Bs[buf][0][tx * 4]);
        fb[0][1] = *reinterpret_cast<const float4 *>(&Bs[buf][0][tx * 4 + 64]);
#pragma unroll
        for (int k = 0; k < LBK; ++k) {
            const int cur = k & 1, nxt = cur ^ 1;
            if (k + 1 < LBK) {
                fa[nxt][0] = *reinterpret_cast<const float4 *>(&As[buf][k + 1][ty * 8]);
                fa[nxt][1] = *reinterpret_cast<const float4 *>(&As[buf][k + 1][ty * 8 + 4]);
                fb[nxt][0] = *reinterpret_cast<const float4 *>(&Bs[buf][k + 1][tx * 4]);
                fb[nxt][1] = *reinterpret_cast<const float4 *>(&Bs[buf][k + 1][tx * 4 + 64]);
            }
            const float a[8] = {fa[cur][0].x, fa[cur][0].y, fa[cur][0].z, fa[cur][0].w,
                                fa[cur][1].x, fa[cur][1].y, fa[cur][1].z, fa[cur][1].w};
            const float b[8] = {fb[cur][0].x, fb[cur][0].y, fb[cur][0].z, fb[cur][0].w,
                                fb[cur][1].x, fb[cur][1].y, fb[cur][1].z, fb[cur][1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) stash(buf ^ 1, av, bv);
        __syncthreads();
        buf ^= 1;
    }
    const long long r0 = (long long)blockIdx.y * LBM + ty * 8;
    const int c0 = blockIdx.x * LBN;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float *crow = C + (r0 + i) * N + c0;
        *reinterpret_cast<float4 *>(crow + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        *reinterpret_cast<float4 *>(crow + tx * 4 + 64) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
}

// ---------------------------------------------------------------- step 8
// cp.async N-stage pipeline (台阶 7): 16-byte asynchronous copies of A (kept
// K-major, row pitch BK + 4) and B into a 3-stage ring; commit/wait groups.
constexpr int CP_STAGES = 3, CP_BK = 8;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__global__ void __launch_bounds__(256) k_cp_async(const float *__restrict__ A, const float *__restrict__ B,
                                                  float *__restrict__ C, int M, int N, int K)
{
    __shared__ __align__(16) float As[CP_STAGES][LBM][CP_BK + 4];
    __shared__ __align__(16) float Bs[CP_STAGES][CP_BK][LBN];
    const int t = threadIdx.x;
    const int warp = t / 32, lane = t % 32;
    const int ty = (warp / 4) * 8 + (lane / 8) * 2 + lane % 2;
    const int tx = (warp % 4) * 4 + (lane % 8) / 2;
    const float *Ab = A + (long long)blockIdx.y * LBM * K;
    const float *Bb = B + (long long)blockIdx.x * LBN;
    auto load = [&](int st, int k0) {
        // A: 128 x 8 = 256 float4, B: 8 x 128 = 256 float4; one each per thread
        const int am = t / 2, ak = (t % 2) * 4;
        cp_async16(&As[st][am][ak], Ab + (long long)am * K + k0 + ak);
        const int bk = t / 32, bn = (t % 32) * 4;
        cp_async16(&Bs[st][bk][bn], Bb + (long long)(k0 + bk) * N + bn);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    const int kt = K / CP_BK;
    for (int s = 0; s < CP_STAGES - 1; ++s) {
        if (s < kt)
            load(s, s * CP_BK);
        else
            asm volatile("cp.async.commit_group;" ::: "memory");
    }
    float acc[8][8] = {};
    for (int i = 0; i < kt; ++i) {
        asm volatile("cp.async.wait_group %0;" ::"n"(CP_STAGES - 2) : "memory");
        __syncthreads();
        const int nxt = i + CP_STAGES - 1;
        if (nxt < kt)
            load(nxt % CP_STAGES, nxt * CP_BK);
        else
            asm volatile("cp.async.commit_group;" ::: "memory");
        const int st = i % CP_STAGES;
#pragma unroll
        for (int k = 0; k < CP_BK; ++k) {
            float a[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) a[r] = As[st][ty * 8 + r][k];
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[st][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[st][k][tx * 4 + 64]);
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[r][j] = fmaf(a[r], b[j], acc[r][j]);
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    const long long r0 = (long long)blockIdx.y * LBM + ty * 8;
    const int c0 = blockIdx.x * LBN;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float *crow = C + (r0 + i) * N + c0;
        *reinterpret_cast<float4 *>(crow + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        *reinterpret_cast<float4 *>(crow + tx * 4 + 64) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
}

// ---------------------------------------------------------------- PMPP
// The two worked examples of "PMPP Chapter 06: Performance considerations",
// written from the section 1 and section 3 traffic analysis: what fixes
// their global traffic is which tiles a block brings into shared memory and
// how often, so each kernel below loads every element of its tiles exactly
// once per phase, with consecutive lanes on consecutive addresses; the
// thread-to-output mapping is this file's own.
//
// Corner turning (section 1): B is column-major (element (k, j) at
// B[j*K + k]), so its contiguous direction is k.  A 64-thread block owns a
// 16 x 16 tile of C.  Per 16-wide phase along K it loads the 16 x 16 tile of
// A and of B by element index e = thread + 64*i: element e is (row e/16,
// k e%16) of A and (column e/16, k e%16) of B, so lanes 0-15 of a warp read
// 16 consecutive floats of one row of A or one column of B (coalesced for
// both).  B is stored into shared memory transposed, Bt[k][column] (the
// turn: the transpose happens between the coalesced global read and the
// shared-memory write, not in the global access), and each thread then
// computes a 2 x 2 block of C from two rows of A and two columns of Bt.
// Global loads: 2*16*16 floats per block-phase, i.e. 8*m*n*k/16 bytes.
__global__ void __launch_bounds__(64) k_pmpp_corner_turn(const float *__restrict__ A,
                                                         const float *__restrict__ Bcol,
                                                         float *__restrict__ C, int M, int N, int K)
{
    constexpr int T = 16;
    __shared__ float As[T][T + 1];  // [row][k]; the pad keeps column walks conflict-free
    __shared__ float Bt[T][T + 1];  // [k][column]
    const int t = threadIdx.x;
    const int m0 = blockIdx.y * T, n0 = blockIdx.x * T;
    const int r = 2 * (t >> 3), c = 2 * (t & 7);  // this thread's 2 x 2 block of the tile
    float c00 = 0.0f, c01 = 0.0f, c10 = 0.0f, c11 = 0.0f;
    for (int k0 = 0; k0 < K; k0 += T) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = t + 64 * i, outer = e >> 4, kk = e & 15;
            const int gk = k0 + kk;
            const int gm = m0 + outer, gn = n0 + outer;
            As[outer][kk] = (gm < M && gk < K) ? A[(long long)gm * K + gk] : 0.0f;
            Bt[kk][outer] = (gn < N && gk < K) ? Bcol[(long long)gn * K + gk] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < T; ++kk) {
            const float a0 = As[r][kk], a1 = As[r + 1][kk];
            const float b0 = Bt[kk][c], b1 = Bt[kk][c + 1];
            c00 = fmaf(a0, b0, c00);
            c01 = fmaf(a0, b1, c01);
            c10 = fmaf(a1, b0, c10);
            c11 = fmaf(a1, b1, c11);
        }
        __syncthreads();
    }
    const int gm = m0 + r, gn = n0 + c;
    if (gm < M) {
        if (gn < N) C[(long long)gm * N + gn] = c00;
        if (gn + 1 < N) C[(long long)gm * N + gn + 1] = c01;
    }
    if (gm + 1 < M) {
        if (gn < N) C[(long long)(gm + 1) * N + gn] = c10;
        if (gn + 1 < N) C[(long long)(gm + 1) * N + gn + 1] = c11;
    }
}

// Thread coarsening (section 3), tile width T = 32, coarsening factor CF:
// a 256-thread block owns CF horizontally adjacent 32 x 32 tiles of C (a
// 32 x 32*CF strip).  Per phase it loads the strip's one A tile once and its
// CF B tiles, by element index (consecutive lanes along k for A, along the
// columns for B: both coalesced), then synchronises once.  Thread t owns
// row t/8 of the strip and the 4*CF columns (t%8) + 8*j: every A value it
// reads from shared memory serves 4*CF multiply-adds across all CF tiles.
// Global loads per block-phase: 32*32*(1 + CF) floats, i.e.
// 4*m*n*k*(1 + 1/CF)/32 bytes in total.  M, K multiples of 32, N a multiple
// of 32*CF.
template <int CF>
__global__ void __launch_bounds__(256) k_pmpp_coarsened(const float *__restrict__ A, const float *__restrict__ B,
                                                        float *__restrict__ C, int M, int N, int K)
{
    constexpr int T = 32, W = T * CF;
    __shared__ float As[T][T + 1];  // [row][k]
    __shared__ float Bs[T][W];      // [k][column of the strip]
    const int t = threadIdx.x;
    const int m0 = blockIdx.y * T, n0 = blockIdx.x * W;
    const int row = t >> 3, lane_col = t & 7;
    float acc[4 * CF];
#pragma unroll
    for (int j = 0; j < 4 * CF; ++j) acc[j] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += T) {
#pragma unroll
        for (int i = 0; i < T * T / 256; ++i) {
            const int e = t + 256 * i;
            As[e >> 5][e & 31] = A[(long long)(m0 + (e >> 5)) * K + k0 + (e & 31)];
        }
#pragma unroll
        for (int i = 0; i < T * W / 256; ++i) {
            const int e = t + 256 * i;
            Bs[e / W][e % W] = B[(long long)(k0 + e / W) * N + n0 + e % W];
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < T; ++kk) {
            const float a = As[row][kk];
#pragma unroll
            for (int j = 0; j < 4 * CF; ++j) acc[j] = fmaf(a, Bs[kk][lane_col + 8 * j], acc[j]);
        }
        __syncthreads();
    }
    float *crow = C + (long long)(m0 + row) * N + n0 + lane_col;
#pragma unroll
    for (int j = 0; j < 4 * CF; ++j) crow[8 * j] = acc[j];
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

extern "C" const char *gemm_ladder_name(int step)
{
    switch (step) {
    case GEMM_LADDER_NAIVE: return "1 naive";
    case GEMM_LADDER_SMEM_TILING: return "2 shared-memory tiling (32x32)";
    case GEMM_LADDER_THREAD_TILING: return "3 thread tiling (8x8 registers)";
    case GEMM_LADDER_VECTORIZED: return "4 float4 loads, A transposed";
    case GEMM_LADDER_CONFLICT_FREE: return "5 bank conflicts removed";
    case GEMM_LADDER_WARP_TILING: return "6 warp tiling (4x8)";
    case GEMM_LADDER_DOUBLE_BUFFER: return "7 double buffering";
    case GEMM_LADDER_CP_ASYNC: return "8 cp.async 3-stage pipeline";
    case GEMM_LADDER_PMPP_CORNER_TURN: return "PMPP corner turning (16x16 tiles, B column-major, 2x2 per thread)";
    case GEMM_LADDER_PMPP_COARSENED: return "PMPP thread coarsening (32x32 tiles, factor 4, 16 outputs per thread)";
    default: return "";
    }
}

extern "C" int gemm_ladder_run(int step, int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                               float *C, cudaStream_t stream)
{
    if (M <= 0 || N <= 0 || K <= 0 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30) || !A || !B || !C)
        return GEMM_ERR_INVALID;
    const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
    const bool tiled128 = M % 128 == 0 && N % 128 == 0;
    switch (step) {
    case GEMM_LADDER_NAIVE:
        k_naive<<<dim3((n + 31) / 32, (m + 7) / 8), dim3(32, 8), 0, stream>>>(A, B, C, m, n, k);
        break;
    case GEMM_LADDER_SMEM_TILING:
        k_tiled<32><<<dim3((n + 31) / 32, (m + 31) / 32), dim3(32, 32), 0, stream>>>(A, B, C, m, n, k);
        break;
    case GEMM_LADDER_THREAD_TILING:
        if (!tiled128 || K % 8) return GEMM_ERR_INVALID;
        k_thread_tile<<<dim3(n / 128, m / 128), 256, 0, stream>>>(A, B, C, m, n, k);
        break;
    case GEMM_LADDER_VECTORIZED:
    case GEMM_LADDER_CONFLICT_FREE:
    case GEMM_LADDER_WARP_TILING:
    case GEMM_LADDER_DOUBLE_BUFFER:
        if (!tiled128 || K % 8) return GEMM_ERR_INVALID;
        if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_ALIGNMENT;
        if (step == GEMM_LADDER_VECTORIZED)
            k_vec<0, false, false><<<dim3(n / 128, m / 128), 256, 0, stream>>>(A, B, C, m, n, k);
        else if (step == GEMM_LADDER_CONFLICT_FREE)
            k_vec<4, true, false><<<dim3(n / 128, m / 128), 256, 0, stream>>>(A, B, C, m, n, k);
        else if (step == GEMM_LADDER_WARP_TILING)
            k_vec<4, true, true><<<dim3(n / 128, m / 128), 256, 0, stream>>>(A, B, C, m, n, k);
        else
            k_double_buffer<<<dim3(n / 128, m / 128), 256, 0, stream>>>(A, B, C, m, n, k);
        break;
    case GEMM_LADDER_CP_ASYNC:
        if (!tiled128 || K % CP_BK) return GEMM_ERR_INVALID;
        if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_ALIGNMENT;
        k_cp_async<<<dim3(n / 128, m / 128), 256, 0, stream>>>(A, B, C, m, n, k);
        break;
    case GEMM_LADDER_PMPP_CORNER_TURN:
        k_pmpp_corner_turn<<<dim3((n + 15) / 16, (m + 15) / 16), 64, 0, stream>>>(A, B, C, m, n, k);
        break;
    case GEMM_LADDER_PMPP_COARSENED:
        if (M % 32 || K % 32 || N % 128) return GEMM_ERR_INVALID;
        k_pmpp_coarsened<4><<<dim3(n / 128, m / 32), 256, 0, stream>>>(A, B, C, m, n, k);
        break;
    default:
        return GEMM_ERR_INVALID;
    }
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
