// Tensor-core GEMM for sm_103a: C = A·B with tcgen05.mma, BF16 or TF32
// operands, FP32 accumulation in tensor memory (TMEM), FP32 C.
//
// The pages stop at Hopper ("GEMM 性能优化", 台阶 7: TMA moves tiles and the
// tensor cores read operands straight from shared memory).  This kernel is
// the Blackwell form of that step:
//  * warp 0, one thread: TMA producer filling a 4-stage shared-memory ring
//    (128-byte swizzled rows of A and B) guarded by full/empty mbarriers;
//  * warp 1: allocates 512 TMEM columns (two 128x256 FP32 accumulators) and,
//    from one thread, issues tcgen05.mma (M=128, N=256, K=32 bytes per
//    instruction); tcgen05.commit releases ring stages and announces a
//    finished accumulator;
//  * warps 2-5: epilogue, tcgen05.ld of their 32 TMEM lanes, guarded stores
//    of C.  With two accumulators the epilogue of one tile overlaps the
//    main loop of the next.
//  * persistent grid (one CTA per SM) walking tiles in groups of `group_m`
//    tile rows for L2 reuse ("GEMM 性能优化", Wave 模型与 L2 命中率).
// A is K-major.  B is K-major when stored column-major (the corner-turning
// case of "PMPP Chapter 06: Performance considerations", section 1) and
// MN-major when stored row-major; the shared-memory descriptor says which,
// so no transpose pass is needed.  MN-major TF32 tiles are staged with the
// 32-byte-atom variant of the 128-byte swizzle.  Out-of-range elements are zero-filled by
// TMA and stores are guarded, so any M, N, K works.
#include <cstdint>

#include "../../include/gemm.h"
#include "gemm_internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int BM = kTcBM, BN = kTcBN;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * 128;  // 16 KiB: 128 rows x 128 bytes of K
constexpr int B_BYTES = BN * 128;  // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;  // two accumulators of BN columns
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
static_assert(SMEM_BYTES > 116 * 1024, "one CTA per SM: TMEM allocation assumes it");

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, group_m;
    float *C;
    long long ldc;
    int *status;
    unsigned long long timeout_ns;
    int c_vec4;
};

__device__ __forceinline__ void tile_coords(int t, const TcParams &p, int &mb, int &nb)
{
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

// Instruction descriptor (kind::f16 / kind::tf32): FP32 accumulator, operand
// format, A K-major, B K- or MN-major, N/8 and M/16.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmt, uint32_t b_mn_major)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn_major << 16) |
           (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
}

// DT: 0 = BF16 (2-byte elements), 1 = TF32 (4-byte elements).
template <int DT, int LAYOUT_B>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int BK = 128 / ES;        // K elements per stage
    constexpr int UMMA_K = 32 / ES;     // K elements per MMA instruction
    constexpr int K_STEPS = BK / UMMA_K;  // 4
    constexpr int BOX_N = 128 / ES;     // row-major B: N elements per TMA box
    constexpr int B_BOXES = BN / BOX_N;
    constexpr int BOX_BYTES = BK * 128;  // one row-major B box
    constexpr uint32_t IDESC = make_idesc(DT == 0 ? 1u : 2u, LAYOUT_B == 0 ? 1u : 0u);
    // An MN-major operand of 32-bit elements uses the 128-byte swizzle with
    // 32-byte atoms (the row-major B tensor map is encoded to match); its
    // swizzle pattern repeats every 4 rows of K, so the K-direction stride of
    // the descriptor is 4 x 128 bytes instead of 8 x 128 bytes.
    constexpr uint32_t B_MN_LAYOUT = DT == 0 ? kLayoutSw128 : kLayoutSw128Atom32;
    constexpr uint32_t B_MN_SBO = DT == 0 ? 1024u : 512u;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t bars = sbase + STAGES * STAGE_BYTES;
    const uint32_t full_bar = bars;                      // [STAGES]
    const uint32_t empty_bar = bars + 8 * STAGES;        // [STAGES]
    const uint32_t tfull_bar = bars + 16 * STAGES;       // [2]
    const uint32_t tempty_bar = tfull_bar + 16;          // [2]
    const uint32_t drain_bar = tempty_bar + 16;          // [1]
    uint8_t *tail = smem + STAGES * STAGE_BYTES + NUM_BARS * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(tail);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int k_tiles = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar + 8 * b, 1);
            mbar_init(tempty_bar + 8 * b, 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(const_cast<uint32_t *>(tmem_slot)), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
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
                    const uint32_t a_st = sbase + s * STAGE_BYTES;
                    const uint32_t b_st = a_st + A_BYTES;
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(a_st, &tmA, fb, kt * BK, mb * BM);
                    if (LAYOUT_B == 0) {
#pragma unroll
                        for (int j = 0; j < B_BOXES; ++j)
                            tma_load_2d(b_st + j * BOX_BYTES, &tmB, fb, nb * BN + j * BOX_N, kt * BK);
                    } else {
                        tma_load_2d(b_st, &tmB, fb, kt * BK, nb * BN);
                    }
                }
            }
            if (!ok) {
                const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
                for (uint32_t i = it - n; i < it; ++i) {
                    int dummy = 0;
                    mbar_wait(full_bar + 8 * (i % STAGES), (i / STAGES) & 1u, &dummy, nullptr,
                              kWaitDrain, p.timeout_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, acc_it = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++acc_it) {
                const uint32_t abuf = acc_it & 1u;
                const uint32_t aph = (acc_it >> 1) & 1u;
                if (!mbar_wait(tempty_bar + 8 * abuf, aph ^ 1u, abort_flag, p.status,
                               kWaitMmaTmemEmpty, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + abuf * BN;
                for (int kt = 0; kt < k_tiles; ++kt, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait(full_bar + 8 * s, ph, abort_flag, p.status, kWaitMmaFull,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_st = sbase + s * STAGE_BYTES;
                    const uint32_t b_st = a_st + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < K_STEPS; ++kk) {
                        const uint64_t adesc = smem_desc(a_st + kk * 32, 16, 1024, kLayoutSw128);
                        const uint64_t bdesc =
                            LAYOUT_B == 0
                                ? smem_desc(b_st + kk * UMMA_K * 128, BOX_BYTES, B_MN_SBO, B_MN_LAYOUT)
                                : smem_desc(b_st + kk * 32, 16, 1024, kLayoutSw128);
                        const uint32_t accumulate = (kt > 0 || kk > 0) ? 1u : 0u;
                        if (DT == 0)
                            tc_mma_f16(d_tmem, adesc, bdesc, IDESC, accumulate);
                        else
                            tc_mma_tf32(d_tmem, adesc, bdesc, IDESC, accumulate);
                    }
                    issued = true;
                    tc_commit(empty_bar + 8 * s);
                }
                if (!ok) break;
                tc_commit(tfull_bar + 8 * abuf);
            }
            if (!ok && issued) {
                // Let every MMA already issued finish before TMEM is freed.
                tc_commit(drain_bar);
                int dummy = 0;
                mbar_wait(drain_bar, 0, &dummy, nullptr, kWaitDrain, p.timeout_ns);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        uint32_t acc_it = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++acc_it) {
            int mb, nb;
            tile_coords(tile, p, mb, nb);
            const uint32_t abuf = acc_it & 1u;
            const uint32_t aph = (acc_it >> 1) & 1u;
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait(tfull_bar + 8 * abuf, aph, abort_flag, p.status, kWaitEpiTmemFull,
                               p.timeout_ns);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            tc_fence_after_sync();
            const long long m = (long long)mb * BM + row;
            float *crow = p.C + m * p.ldc;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_load_32cols(t_row + c * 32, v);
                tmem_wait_ld();
                if (m < p.M) {
                    const int n0 = nb * BN + c * 32;
                    if (p.c_vec4 && n0 + 31 < p.N) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4 *>(crow + n0 + 4 * j) =
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (n0 + j < p.N) crow[n0 + j] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar + 8 * abuf);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int DT, int L>
cudaError_t set_attrs()
{
    return cudaFuncSetAttribute(gemm_tc_kernel<DT, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SMEM_BYTES);
}

}  // namespace

cudaError_t prepare_tc()
{
    cudaError_t e = set_attrs<0, 0>();
    if (e == cudaSuccess) e = set_attrs<0, 1>();
    if (e == cudaSuccess) e = set_attrs<1, 0>();
    if (e == cudaSuccess) e = set_attrs<1, 1>();
    return e;
}

int tc_grid(int tiles, int sm_count) { return tiles < sm_count ? tiles : sm_count; }

cudaError_t launch_tc(int dtype, int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                      const LaunchCommon &lc)
{
    TcParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.group_m = lc.group_m > 0 ? lc.group_m : 16;
    p.C = C;
    p.ldc = ldc;
    p.status = lc.status;
    p.timeout_ns = lc.timeout_ns;
    p.c_vec4 = c_vec4 ? 1 : 0;
    const dim3 grid(lc.grid), block(THREADS);
    if (dtype == GEMM_BF16) {
        if (layout_b == 0)
            gemm_tc_kernel<0, 0><<<grid, block, SMEM_BYTES, lc.stream>>>(tmA, tmB, p);
        else
            gemm_tc_kernel<0, 1><<<grid, block, SMEM_BYTES, lc.stream>>>(tmA, tmB, p);
    } else {
        if (layout_b == 0)
            gemm_tc_kernel<1, 0><<<grid, block, SMEM_BYTES, lc.stream>>>(tmA, tmB, p);
        else
            gemm_tc_kernel<1, 1><<<grid, block, SMEM_BYTES, lc.stream>>>(tmA, tmB, p);
    }
    return cudaGetLastError();
}

}  // namespace dg
