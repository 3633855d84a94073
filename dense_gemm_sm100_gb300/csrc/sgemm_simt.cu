// FP32 SIMT GEMM for sm_103a: C = A·B with FP32 fused multiply-adds on the
// CUDA cores.
//
// Design, restating the optimisation steps of "GEMM 性能优化" (八个台阶) for
// Blackwell:
//  * 台阶 1 (shared-memory tiling along K): each CTA owns a 128x128 tile of C
//    and walks K in 32-element slices staged in shared memory.
//  * 台阶 2 (thread tiling): every consumer thread keeps an 8x8 block of C in
//    registers and does 64 FMAs per k from 8 A and 8 B values.
//  * 台阶 3/4 (vector loads, bank conflicts): the Tensor Memory Accelerator
//    writes each stage with a 128-byte XOR swizzle; every shared load is a
//    16-byte vector and the thread-to-data mapping below makes each warp-wide
//    load hit 32 distinct banks (or broadcast).
//  * 台阶 5 (warp tiling): a warp covers 64 rows x 64 columns of the tile
//    through 4x8 lanes; lanes that share a row group share A loads.
//  * 台阶 6/7 (double buffering, asynchronous copies): a dedicated producer
//    warp issues TMA copies into a 6-stage ring guarded by mbarriers, so
//    global loads overlap the math; register fragments of the next k group
//    are loaded while the current one is multiplied.
//  * 台阶 8 (SASS tuning) is replaced by source-level structure: compile-time
//    power-of-two tiles, offsets precomputed per thread so every shared load
//    is base + immediate, and __launch_bounds__.
//  * Wave model / block order: the grid is persistent (one CTA per SM) and
//    walks tiles in groups of `group_m` tile rows for L2 reuse.
//  * Column-major B ("PMPP Chapter 06: Performance considerations", section
//    1, corner turning): TMA reads B along its contiguous K direction
//    (coalesced), and the transposed access happens in shared memory.
//
// Out-of-range elements of A and B are zero-filled by TMA; stores of C are
// guarded, so any M, N, K works.
#include <cstdint>

#include "gemm_internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = kSimtBK;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 4;  // 16 KiB
constexpr int B_BYTES = BK * BN * 4;  // 16 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
constexpr int BAR_BYTES = 2 * STAGES * 8 + 16;
constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + BAR_BYTES;

static_assert(BM == 128 && BN == 128 && BK == 32, "thread mapping assumes 128x128x32 tiles");
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");

struct SimtParams {
    int M, N, K;
    int tiles_m, tiles_n, group_m;
    float *C;
    long long ldc;
    int *status;
    unsigned long long timeout_ns;
    int c_vec4;
};

// Tile t of the grouped order: groups of `group_m` tile rows, column-major
// inside a group, so CTAs running at the same time share A and B panels.
__device__ __forceinline__ void tile_coords(int t, const SimtParams &p, int &mb, int &nb)
{
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

template <int LAYOUT_B>
__global__ void __launch_bounds__(THREADS, 1)
    sgemm_simt_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const SimtParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t full_bar = sbase + STAGES * STAGE_BYTES;  // STAGES x 8 bytes
    const uint32_t empty_bar = full_bar + STAGES * 8;         // STAGES x 8 bytes
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + STAGES * STAGE_BYTES + 2 * STAGES * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int k_tiles = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CONSUMER_WARPS) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, p, mb, nb);
            for (int kt = 0; kt < k_tiles; ++kt, ++it) {
                const uint32_t s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait(empty_bar + 8 * s, ph ^ 1u, abort_flag, p.status,
                               kWaitProducerEmpty, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar + 8 * s;
                const uint32_t st = sbase + s * STAGE_BYTES;
                mbar_arrive_expect_tx(fb, STAGE_BYTES);
                tma_load_2d(st, &tmA, fb, kt * BK, mb * BM);
                if (LAYOUT_B == 0) {
#pragma unroll
                    for (int j = 0; j < BN / 32; ++j)
                        tma_load_2d(st + A_BYTES + j * 4096, &tmB, fb, nb * BN + 32 * j, kt * BK);
                } else {
                    tma_load_2d(st + A_BYTES, &tmB, fb, kt * BK, nb * BN);
                }
            }
        }
        if (!ok) {
            // Leave no copy in flight: wait (bounded) for the stages issued last.
            const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
            for (uint32_t i = it - n; i < it; ++i) {
                int dummy = 0;
                mbar_wait(full_bar + 8 * (i % STAGES), (i / STAGES) & 1u, &dummy, nullptr,
                          kWaitDrain, p.timeout_ns);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int wm = warp >> 1;  // 0..3
    const int wn = warp & 1;   // 0..1
    const int lr = lane >> 3;  // 0..3
    const int lc = lane & 7;   // 0..7
    // Rows row0 + 8*i (i < 8): the two warps of a 64-row band interleave by
    // four rows, so row & 7 is fixed per thread and distinct across the four
    // row groups of a warp (conflict-free swizzled A loads).
    const int row0 = (wm >> 1) * 64 + (wm & 1) * 4 + lr;
    uint32_t a_off[8], b_off[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) a_off[g] = row0 * 128 + ((g ^ (row0 & 7)) << 4);
    if (LAYOUT_B == 0) {
        // Columns wn*64 + 4*lc + {0..3} and +32: chunk lc of boxes 2wn and
        // 2wn+1; b_off[c] serves every k with k & 7 == c.
#pragma unroll
        for (int c = 0; c < 8; ++c) b_off[c] = A_BYTES + (2 * wn) * 4096 + ((lc ^ c) << 4);
    } else {
        // Columns col0 + 8*j: col0 & 7 == lc, distinct across the warp.
        const int col0 = wn * 64 + lc;
#pragma unroll
        for (int g = 0; g < 8; ++g) b_off[g] = A_BYTES + col0 * 128 + ((g ^ lc) << 4);
    }

    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, p, mb, nb);
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

        for (int kt = 0; kt < k_tiles; ++kt, ++it) {
            const uint32_t s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!mbar_wait(full_bar + 8 * s, ph, abort_flag, p.status, kWaitConsumerFull,
                           p.timeout_ns))
                return;
            const uint8_t *st = smem + s * STAGE_BYTES;
#pragma unroll
            for (int g = 0; g < BK / 4; ++g) {
                float4 a[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    a[i] = *reinterpret_cast<const float4 *>(st + a_off[g] + i * 1024);
                if (LAYOUT_B == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int k = 4 * g + kk;
                        const uint8_t *bp = st + b_off[k & 7] + k * 128;
                        const float4 b0 = *reinterpret_cast<const float4 *>(bp);
                        const float4 b1 = *reinterpret_cast<const float4 *>(bp + 4096);
                        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
                        }
                    }
                } else {
                    float4 b[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        b[j] = *reinterpret_cast<const float4 *>(st + b_off[g] + j * 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float bv = kk == 0 ? b[j].x : kk == 1 ? b[j].y : kk == 2 ? b[j].z : b[j].w;
                                acc[i][j] = fmaf(av, bv, acc[i][j]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * s);
        }

        // ------------------------------------------------------ epilogue
        const long long m_base = (long long)mb * BM + row0;
        if (LAYOUT_B == 0) {
            const int n_base = nb * BN + wn * 64 + 4 * lc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const long long m = m_base + 8 * i;
                if (m >= p.M) continue;
                float *crow = p.C + m * p.ldc;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = n_base + 32 * h;
                    if (p.c_vec4 && n + 3 < p.N) {
                        *reinterpret_cast<float4 *>(crow + n) =
                            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (n + q < p.N) crow[n + q] = acc[i][4 * h + q];
                    }
                }
            }
        } else {
            const int n_base = nb * BN + wn * 64 + lc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const long long m = m_base + 8 * i;
                if (m >= p.M) continue;
                float *crow = p.C + m * p.ldc;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int n = n_base + 8 * j;
                    if (n < p.N) crow[n] = acc[i][j];
                }
            }
        }
    }
}

template <int L>
cudaError_t set_attrs()
{
    return cudaFuncSetAttribute(sgemm_simt_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SMEM_BYTES);
}

}  // namespace

cudaError_t prepare_simt()
{
    cudaError_t e = set_attrs<0>();
    if (e == cudaSuccess) e = set_attrs<1>();
    return e;
}

int simt_grid(int tiles, int sm_count) { return tiles < sm_count ? tiles : sm_count; }

cudaError_t launch_simt_f32(const CUtensorMap &tmA, const CUtensorMap &tmB, int layout_b, int M,
                            int N, int K, float *C, int64_t ldc, bool c_vec4,
                            const LaunchCommon &lc)
{
    SimtParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.group_m = lc.group_m > 0 ? lc.group_m : 8;
    p.C = C;
    p.ldc = ldc;
    p.status = lc.status;
    p.timeout_ns = lc.timeout_ns;
    p.c_vec4 = c_vec4 ? 1 : 0;
    const dim3 grid(lc.grid), block(THREADS);
    if (layout_b == 0)
        sgemm_simt_kernel<0><<<grid, block, SMEM_BYTES, lc.stream>>>(tmA, tmB, p);
    else
        sgemm_simt_kernel<1><<<grid, block, SMEM_BYTES, lc.stream>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace dg
