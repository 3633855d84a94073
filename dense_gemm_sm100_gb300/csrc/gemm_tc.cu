// Tensor-core GEMM for sm_103a: C = A·B with tcgen05.mma, BF16 or TF32
// operands, FP32 accumulation in tensor memory (TMEM), FP32 C.
//
// The pages stop at Hopper ("GEMM 性能优化", 台阶 7: TMA moves tiles and the
// tensor cores read operands straight from shared memory).  This kernel is
// the Blackwell form of that step:
//  * warp 0, one thread: TMA producer filling a 4-stage shared-memory ring
//    (128-byte swizzled rows of A and B) guarded by full/empty mbarriers;
//  * warp 1: allocates 512 TMEM columns (two 128x256 FP32 accumulators) and
//    runs the MMA loop as a whole warp (warp-uniform stage indices and
//    descriptors); one elected lane issues tcgen05.mma (M=128, N=256, K=32
//    bytes per instruction) and tcgen05.commit, which releases ring stages
//    and announces a finished accumulator;
//  * warps 2-5: epilogue, tcgen05.ld of their 32 TMEM lanes; each 32x32 FP32
//    chunk is staged in 128-byte-swizzled shared memory and written by one
//    TMA store (whole 128-byte lines; TMA clips the M and N edges).  With two
//    accumulators the epilogue of one tile overlaps the main loop of the
//    next.  A C that TMA cannot address (pitch or base not 16-byte aligned)
//    takes guarded per-thread stores instead.
//  * persistent grid walking tiles in groups of `group_m` tile rows for L2
//    reuse ("GEMM 性能优化", Wave 模型与 L2 命中率).
// A is K-major.  B is K-major when stored column-major (the corner-turning
// case of "PMPP Chapter 06: Performance considerations", section 1) and
// MN-major when stored row-major; the shared-memory descriptor says which,
// so no transpose pass is needed.  MN-major TF32 tiles are staged with the
// 32-byte-atom variant of the 128-byte swizzle.  Out-of-range elements are
// zero-filled by TMA and stores are guarded, so any M, N, K works.
#include <algorithm>
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
// Epilogue staging: per epilogue warp two 32x32 FP32 chunks (4 KB each,
// 128-byte swizzled) that TMA stores to C.
constexpr int EPI_CHUNK_BYTES = 32 * 32 * 4;
constexpr int EPI_BYTES = 4 * 2 * EPI_CHUNK_BYTES;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16;
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
static_assert(SMEM_BYTES > 116 * 1024, "one CTA per SM: TMEM allocation assumes it");
static_assert(kTcBoxBCol == BN / 2, "column-major B is loaded in two halves");

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, group_m;
    float *C;
    long long ldc;
    int *status;
    unsigned long long timeout_ns;
    int c_vec4;
    int c_tma;       // 1: C is written by TMA stores through tmC
    int b_chunks;    // 1 (row-major B, one-CTA or pair kernel): tmB is the 3-D chunk view, one box per stage
    int debug_drop;  // test hook: CTA 0 never loads its first stage
    // Pair kernel: the epilogue pauses this long between its 32-column C
    // chunks, spreading a tile's 256 KB of C writes instead of bursting them
    // against the operand loads (0: no pause; set only for tiles of at least
    // 32 ring stages, whose TMEM buffer has ample slack before reuse).
    unsigned epi_pace_ns;
    // K split: units are (tile unit, slice) slice-major; slice s covers
    // stages [s*kt_per_split, min(k_tiles, (s+1)*kt_per_split)) and its
    // accumulator goes to partials[s][tile row][tile column] (BM x BN floats)
    int splits, kt_per_split;
    float *partials;
};

// K range of work unit u; `base` = tile units per slice.
struct KRange {
    int ub, kt0, kt1, slice;
};

__device__ __forceinline__ KRange unit_krange(int u, const TcParams &p, int base, int k_tiles)
{
    KRange r;
    r.slice = u / base;
    r.ub = u - r.slice * base;
    r.kt0 = r.slice * p.kt_per_split;
    r.kt1 = min(k_tiles, r.kt0 + p.kt_per_split);
    return r;
}

// Unit u of the grouped order over (tile-row groups of CL tiles) x tiles_n:
// groups of `group_m` units along M, column-major inside a group, so CTAs
// running at the same time share A and B panels.  The CTA of cluster rank r
// takes tile row CL*um + r.
template <int CL>
__device__ __forceinline__ void unit_coords(int u, const TcParams &p, uint32_t rank, int &mb, int &nb)
{
    const int units_m = (p.tiles_m + CL - 1) / CL;
    const int per_group = p.group_m * p.tiles_n;
    const int g = u / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(units_m - first_m, p.group_m);
    const int r = u - g * per_group;
    mb = CL * (first_m + r % gm) + static_cast<int>(rank);
    nb = r / gm;
}

// Instruction descriptor (kind::f16 / kind::tf32): FP32 accumulator, operand
// format, A K-major, B K- or MN-major, N/8 and M/16.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmt, uint32_t b_mn_major)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn_major << 16) |
           (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
}

// DT: 0 = BF16 (2-byte elements), 1 = TF32 (4-byte elements).  One CTA per
// 128 x 256 tile.
template <int DT, int LAYOUT_B>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int BK = 128 / ES;          // K elements per stage
    constexpr int UMMA_K = 32 / ES;       // K elements per MMA instruction
    constexpr int K_STEPS = BK / UMMA_K;  // 4
    constexpr int BOX_N = 128 / ES;       // row-major B: N elements per TMA box
    constexpr int B_BOXES = BN / BOX_N;
    constexpr int BOX_BYTES = BK * 128;   // one row-major B box
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
    const uint32_t epi_base = sbase + STAGES * STAGE_BYTES;  // EPI_BYTES, 1024-aligned
    const uint32_t bars = epi_base + EPI_BYTES;
    const uint32_t full_bar = bars;                      // [STAGES]
    const uint32_t empty_bar = bars + 8 * STAGES;        // [STAGES]
    const uint32_t tfull_bar = bars + 16 * STAGES;       // [2]
    const uint32_t tempty_bar = tfull_bar + 16;          // [2]
    const uint32_t drain_bar = tempty_bar + 16;          // [1]
    uint8_t *tail = smem + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(tail);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = 0u;
    const int cluster = blockIdx.x;
    const int clusters = gridDim.x;
    const int base_units = p.tiles_m * p.tiles_n;
    const int num_units = base_units * p.splits;
    const int k_tiles = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, 1);  // released by the MMA issuer's commit
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
            for (int u = cluster; ok && u < num_units; u += clusters) {
                const KRange kr = unit_krange(u, p, base_units, k_tiles);
                int mb, nb;
                unit_coords<1>(kr.ub, p, rank, mb, nb);
                for (int kt = kr.kt0; kt < kr.kt1; ++kt, ++it) {
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
                    if (p.debug_drop && blockIdx.x == 0 && it == 0) continue;  // bytes that never come
                    tma_load_2d(a_st, &tmA, fb, kt * BK, mb * BM);
                    if (LAYOUT_B == 0) {
                        if (p.b_chunks) {
                            tma_load_3d(b_st, &tmB, fb, 0, kt * BK, nb * BN / BOX_N);  // all B_BOXES chunks
                        } else {
#pragma unroll
                            for (int j = 0; j < B_BOXES; ++j)
                                tma_load_2d(b_st + j * BOX_BYTES, &tmB, fb, nb * BN + j * BOX_N, kt * BK);
                        }
                    } else {
                        tma_load_2d(b_st, &tmB, fb, kt * BK, nb * BN);
                        tma_load_2d(b_st + B_BYTES / 2, &tmB, fb, kt * BK, nb * BN + BN / 2);
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
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // Whole warp, warp-uniform stage indices and descriptors; one elected
        // lane issues (as in the pair kernel below).
        {
            uint32_t it = 0, acc_it = 0;
            bool ok = true, issued = false;
            for (int u = cluster; ok && u < num_units; u += clusters, ++acc_it) {
                const uint32_t abuf = acc_it & 1u;
                const uint32_t aph = (acc_it >> 1) & 1u;
                if (!mbar_wait_warp(tempty_bar + 8 * abuf, aph ^ 1u, abort_flag, p.status, kWaitMmaTmemEmpty,
                                    p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + abuf * BN;
                const KRange kr = unit_krange(u, p, base_units, k_tiles);
                for (int kt = kr.kt0; kt < kr.kt1; ++kt, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait_warp(full_bar + 8 * s, ph, abort_flag, p.status, kWaitMmaFull, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_st = sbase + s * STAGE_BYTES;
                    const uint32_t b_st = a_st + A_BYTES;
                    uint64_t ad[K_STEPS], bd[K_STEPS];
#pragma unroll
                    for (int kk = 0; kk < K_STEPS; ++kk) {
                        ad[kk] = smem_desc(a_st + kk * 32, 16, 1024, kLayoutSw128);
                        bd[kk] = LAYOUT_B == 0 ? smem_desc(b_st + kk * UMMA_K * 128, BOX_BYTES, B_MN_SBO, B_MN_LAYOUT)
                                               : smem_desc(b_st + kk * 32, 16, 1024, kLayoutSw128);
                    }
                    const uint32_t acc0 = kt > kr.kt0 ? 1u : 0u;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < K_STEPS; ++kk) {
                            if (DT == 0)
                                tc_mma_f16(d_tmem, ad[kk], bd[kk], IDESC, kk > 0 ? 1u : acc0);
                            else
                                tc_mma_tf32(d_tmem, ad[kk], bd[kk], IDESC, kk > 0 ? 1u : acc0);
                        }
                        tc_commit(empty_bar + 8 * s);
                    }
                    __syncwarp();
                    issued = true;
                }
                if (!ok) break;
                if (elect_one()) tc_commit(tfull_bar + 8 * abuf);
                __syncwarp();
            }
            if (!ok && issued && lane == 0) {
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
        const uint32_t stage_buf = epi_base + static_cast<uint32_t>((warp - 2) * 2 * EPI_CHUNK_BYTES);
        if (p.c_tma && lane == 0) tma_prefetch_desc(&tmC);
        uint32_t acc_it = 0;
        for (int u = cluster; u < num_units; u += clusters, ++acc_it) {
            const KRange kr = unit_krange(u, p, base_units, k_tiles);
            int mb, nb;
            unit_coords<1>(kr.ub, p, rank, mb, nb);
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
                if (c == BN / 32 - 1) {
                    // The accumulator is in registers: hand TMEM back to the MMA warp.
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar + 8 * abuf);
                }
                const int n0 = nb * BN + c * 32;
                if (p.splits > 1) {
                    // a K slice: the whole partial tile (rows and columns past
                    // M and N hold zeros), added into C by the reduction kernel
                    if (mb < p.tiles_m) {
                        float *prow = p.partials +
                                      (((long long)kr.slice * p.tiles_m + mb) * p.tiles_n + nb) * (BM * BN) +
                                      row * BN + c * 32;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4 *>(prow + 4 * j) =
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    }
                } else if (p.c_tma) {
                    // Row `lane` of a 32x32 chunk, 128-byte swizzled (chunk j
                    // of row r at 16*(j ^ (r & 7))), then one TMA store of the
                    // chunk; TMA drops the rows and columns outside C.
                    const uint32_t buf = stage_buf + static_cast<uint32_t>(c & 1) * EPI_CHUNK_BYTES;
                    if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t addr = buf + lane * 128 + ((j ^ (lane & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[4 * j]),
                                     "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                                     : "memory");
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, buf, n0, mb * BM + q * 32);
                        bulk_commit_group();
                    }
                } else if (m < p.M) {
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
        }
        if (p.c_tma && lane == 0) bulk_wait_group_all();  // stores done before shared memory goes away
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Pair kernel: one 256 x 256 tile per cluster of two CTAs, computed by
// tcgen05.mma.cta_group::2 issued from the even CTA.  Each CTA stages only
// its 128 rows of A and its 128 columns of B (32 KB per 128-byte slice of K
// instead of 48 KB), so 192 KB of operands are in flight per SM.  D rows of
// CTA r live in CTA r's TMEM.
//
// SUB = K slices of 128 bytes per ring stage.  SUB = 1: six stages of one
// slice (4 MMA instructions between a full-barrier wait and a release).
// SUB = 2: three stages of two slices (8 MMAs per wait and release), the
// same bytes in flight with half the barrier round trips per MMA; the MMA
// issuer is a single thread whose per-stage wait and commit cost shows up
// directly as idle tensor-pipe cycles, so fewer, larger stages keep the
// pipe busier.
constexpr int P_A_BYTES = BM * 128;        // 16 KiB per slice
constexpr int P_B_BYTES = (BN / 2) * 128;  // 16 KiB per slice: this CTA's half of B
constexpr int P_RING_BYTES = 6 * (P_A_BYTES + P_B_BYTES);

template <int SUB>
struct PairCfg {
    static constexpr int STAGE_BYTES = SUB * (P_A_BYTES + P_B_BYTES);
    static constexpr int STAGES = P_RING_BYTES / STAGE_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
    static_assert(SMEM_BYTES > 116 * 1024 && SMEM_BYTES <= 227 * 1024, "one CTA per SM");
};

template <int DT, int LAYOUT_B, int SUB>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const TcParams p)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int BK_SLICE = 128 / ES;           // K elements per 128-byte slice
    constexpr int BK = SUB * BK_SLICE;           // K elements per stage
    constexpr int UMMA_K = 32 / ES;
    constexpr int K_STEPS = BK_SLICE / UMMA_K;   // MMA instructions per slice
    constexpr int P_STAGES = PairCfg<SUB>::STAGES;
    constexpr int P_STAGE_BYTES = PairCfg<SUB>::STAGE_BYTES;
    constexpr int P_NUM_BARS = PairCfg<SUB>::NUM_BARS;
    constexpr int BOX_N = 128 / ES;              // row-major B: N elements per TMA box
    constexpr int B_HALF_BOXES = (BN / 2) / BOX_N;
    constexpr int BOX_BYTES = BK_SLICE * 128;
    // M = 256 across the pair, N = 256.
    constexpr uint32_t IDESC = (1u << 4) | ((DT == 0 ? 1u : 2u) << 7) | ((DT == 0 ? 1u : 2u) << 10) |
                               ((LAYOUT_B == 0 ? 1u : 0u) << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
                               (static_cast<uint32_t>((2 * BM) >> 4) << 24);
    constexpr uint32_t B_MN_LAYOUT = DT == 0 ? kLayoutSw128 : kLayoutSw128Atom32;
    constexpr uint32_t B_MN_SBO = DT == 0 ? 1024u : 512u;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t epi_base = sbase + P_STAGES * P_STAGE_BYTES;
    const uint32_t bars = epi_base + EPI_BYTES;
    const uint32_t full_bar = bars;                    // [P_STAGES], used in the even CTA
    const uint32_t empty_bar = bars + 8 * P_STAGES;    // [P_STAGES], both CTAs
    const uint32_t tfull_bar = bars + 16 * P_STAGES;   // [2], both CTAs
    const uint32_t tempty_bar = tfull_bar + 16;        // [2], used in the even CTA
    const uint32_t drain_bar = tempty_bar + 16;        // [1]
    uint8_t *tail = smem + P_STAGES * P_STAGE_BYTES + EPI_BYTES + P_NUM_BARS * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(tail);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x / 2;
    const int clusters = gridDim.x / 2;
    const int base_units = ((p.tiles_m + 1) / 2) * p.tiles_n;
    const int num_units = base_units * p.splits;
    const int k_tiles = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);   // the even CTA's producer; bytes from both CTAs
            mbar_init(empty_bar + 8 * s, 1);  // the pair commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar + 8 * b, 1);   // the pair commit
            mbar_init(tempty_bar + 8 * b, 8);  // 4 epilogue warps in each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(const_cast<uint32_t *>(tmem_slot)), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t it = 0;
            bool ok = true;
            for (int u = cluster; ok && u < num_units; u += clusters) {
                const KRange kr = unit_krange(u, p, base_units, k_tiles);
                int mb, nb;
                unit_coords<2>(kr.ub, p, rank, mb, nb);
                for (int kt = kr.kt0; kt < kr.kt1; ++kt, ++it) {
                    const uint32_t s = it % P_STAGES;
                    const uint32_t ph = (it / P_STAGES) & 1u;
                    if (!mbar_wait(empty_bar + 8 * s, ph ^ 1u, abort_flag, p.status,
                                   kWaitProducerEmpty, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = full_bar + 8 * s;
                    const uint32_t fb = mapa_shared(fb_local, 0);  // the even CTA's barrier
                    const uint32_t a_st = sbase + s * P_STAGE_BYTES;
                    const uint32_t b_st = a_st + SUB * P_A_BYTES;
                    if (leader) mbar_arrive_expect_tx(fb_local, 2 * P_STAGE_BYTES);
                    if (p.debug_drop && blockIdx.x == 0 && it == 0) continue;  // bytes that never come
                    const int n_half = nb * BN + static_cast<int>(rank) * (BN / 2);
#pragma unroll
                    for (int sl = 0; sl < SUB; ++sl) {
                        // slice sl of the stage: K elements [kx, kx + BK_SLICE)
                        const int kx = kt * BK + sl * BK_SLICE;
                        const uint32_t a_sl = a_st + sl * P_A_BYTES;
                        const uint32_t b_sl = b_st + sl * P_B_BYTES;
                        tma_load_2d_pair(a_sl, &tmA, fb, kx, mb * BM);
                        if (LAYOUT_B == 0) {
                            if (p.b_chunks) {
                                // {column in chunk, k, chunk}: the B_HALF_BOXES chunks of
                                // this CTA's half land one after another, as the 2-D
                                // boxes would (the swizzle follows the address)
                                tma_load_3d_pair(b_sl, &tmB, fb, 0, kx, n_half / BOX_N);
                            } else {
#pragma unroll
                                for (int j = 0; j < B_HALF_BOXES; ++j)
                                    tma_load_2d_pair(b_sl + j * BOX_BYTES, &tmB, fb, n_half + j * BOX_N, kx);
                            }
                        } else {
                            tma_load_2d_pair(b_sl, &tmB, fb, kx, n_half);
                        }
                    }
                }
            }
            const uint32_t n = it < (uint32_t)P_STAGES ? it : (uint32_t)P_STAGES;
            if (ok) {
                // Every release of the last stages must have landed here
                // before shared memory goes away.
                for (uint32_t i = it - n; i < it; ++i)
                    mbar_wait(empty_bar + 8 * (i % P_STAGES), (i / P_STAGES) & 1u, abort_flag, p.status,
                              kWaitDrain, p.timeout_ns);
            } else if (leader) {
                // After an abort: the even CTA's full barriers count the copies
                // of both CTAs; wait (bounded) for those issued last.  The odd
                // CTA cannot pass the final cluster barrier before this ends.
                for (uint32_t i = it - n; i < it; ++i) {
                    int dummy = 0;
                    mbar_wait(full_bar + 8 * (i % P_STAGES), (i / P_STAGES) & 1u, &dummy, nullptr,
                              kWaitDrain, p.timeout_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (even CTA)
        // The whole warp runs the loop, so stage indices and descriptors are
        // warp-uniform values; one elected lane issues a stage's MMAs and its
        // commit.  The issue rate of this one warp bounds the tensor pipe
        // (four MMAs of 128 cycles per stage), and the warp-uniform form
        // issues them in about half the time of a single-lane loop.
        if (leader) {
            uint32_t it = 0, acc_it = 0;
            bool ok = true, issued = false;
            for (int u = cluster; ok && u < num_units; u += clusters, ++acc_it) {
                const uint32_t abuf = acc_it & 1u;
                const uint32_t aph = (acc_it >> 1) & 1u;
                if (!mbar_wait_warp(tempty_bar + 8 * abuf, aph ^ 1u, abort_flag, p.status, kWaitMmaTmemEmpty,
                                    p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + abuf * BN;
                const KRange kr = unit_krange(u, p, base_units, k_tiles);
                for (int kt = kr.kt0; kt < kr.kt1; ++kt, ++it) {
                    const uint32_t s = it % P_STAGES;
                    const uint32_t ph = (it / P_STAGES) & 1u;
                    if (!mbar_wait_warp(full_bar + 8 * s, ph, abort_flag, p.status, kWaitMmaFull, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_st = sbase + s * P_STAGE_BYTES;
                    const uint32_t b_st = a_st + SUB * P_A_BYTES;
                    uint64_t ad[SUB * K_STEPS], bd[SUB * K_STEPS];
#pragma unroll
                    for (int q = 0; q < SUB * K_STEPS; ++q) {
                        const int sl = q / K_STEPS, kk = q % K_STEPS;
                        ad[q] = smem_desc(a_st + sl * P_A_BYTES + kk * 32, 16, 1024, kLayoutSw128);
                        bd[q] = LAYOUT_B == 0 ? smem_desc(b_st + sl * P_B_BYTES + kk * UMMA_K * 128, BOX_BYTES,
                                                          B_MN_SBO, B_MN_LAYOUT)
                                              : smem_desc(b_st + sl * P_B_BYTES + kk * 32, 16, 1024, kLayoutSw128);
                    }
                    const uint32_t acc0 = kt > kr.kt0 ? 1u : 0u;
                    if (elect_one()) {
#pragma unroll
                        for (int q = 0; q < SUB * K_STEPS; ++q) {
                            if (DT == 0)
                                tc_mma_f16_pair(d_tmem, ad[q], bd[q], IDESC, q > 0 ? 1u : acc0);
                            else
                                tc_mma_tf32_pair(d_tmem, ad[q], bd[q], IDESC, q > 0 ? 1u : acc0);
                        }
                        tc_commit_pair_multicast(empty_bar + 8 * s, 0x3);
                    }
                    __syncwarp();
                    issued = true;
                }
                if (!ok) break;
                if (elect_one()) tc_commit_pair_multicast(tfull_bar + 8 * abuf, 0x3);
                __syncwarp();
            }
            if (!ok && issued && lane == 0) {
                tc_commit_pair_multicast(drain_bar, 0x1);
                int dummy = 0;
                mbar_wait(drain_bar, 0, &dummy, nullptr, kWaitDrain, p.timeout_ns);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t stage_buf = epi_base + static_cast<uint32_t>((warp - 2) * 2 * EPI_CHUNK_BYTES);
        if (p.c_tma && lane == 0) tma_prefetch_desc(&tmC);
        uint32_t acc_it = 0;
        for (int u = cluster; u < num_units; u += clusters, ++acc_it) {
            const KRange kr = unit_krange(u, p, base_units, k_tiles);
            int mb, nb;
            unit_coords<2>(kr.ub, p, rank, mb, nb);
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
                if (c == BN / 32 - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            mbar_arrive(tempty_bar + 8 * abuf);
                        else
                            mbar_arrive_cluster(mapa_shared(tempty_bar + 8 * abuf, 0));
                    }
                }
                const int n0 = nb * BN + c * 32;
                if (p.splits > 1) {
                    // a K slice: this CTA's 128 rows of the partial tile (the
                    // odd CTA of a last pair past M writes nothing)
                    if (mb < p.tiles_m) {
                        float *prow = p.partials +
                                      (((long long)kr.slice * p.tiles_m + mb) * p.tiles_n + nb) * (BM * BN) +
                                      row * BN + c * 32;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4 *>(prow + 4 * j) =
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    }
                } else if (p.c_tma) {
                    const uint32_t buf = stage_buf + static_cast<uint32_t>(c & 1) * EPI_CHUNK_BYTES;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t addr = buf + lane * 128 + ((j ^ (lane & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[4 * j]),
                                     "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                                     : "memory");
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, buf, n0, mb * BM + q * 32);
                        bulk_commit_group();
                    }
                    if (p.epi_pace_ns && c + 1 < BN / 32) __nanosleep(p.epi_pace_ns);
                } else if (m < p.M) {
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
        }
        if (p.c_tma && lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncwarp();
    cluster_sync();  // no CTA leaves while its peer may still target its shared memory
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int DT, int L, int SUB>
cudaError_t set_pair_attrs()
{
    return cudaFuncSetAttribute(gemm_tc_pair_kernel<DT, L, SUB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PairCfg<SUB>::SMEM_BYTES);
}

template <int DT, int L, int SUB>
cudaError_t launch_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TcParams &p, int grid, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = PairCfg<SUB>::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<DT, L, SUB>, tmA, tmB, tmC, p);
}

template <int DT, int L>
cudaError_t set_attrs()
{
    return cudaFuncSetAttribute(gemm_tc_kernel<DT, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

template <int DT, int L>
cudaError_t launch_one(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                       const TcParams &p, int grid, cudaStream_t stream)
{
    gemm_tc_kernel<DT, L><<<grid, THREADS, SMEM_BYTES, stream>>>(tmA, tmB, tmC, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_tc()
{
    cudaError_t e = cudaSuccess;
    cudaError_t (*fns[])() = {set_attrs<0, 0>, set_attrs<0, 1>, set_attrs<1, 0>, set_attrs<1, 1>,
                              set_pair_attrs<0, 0, 1>, set_pair_attrs<0, 1, 1>, set_pair_attrs<1, 0, 1>,
                              set_pair_attrs<1, 1, 1>, set_pair_attrs<0, 0, 2>, set_pair_attrs<0, 1, 2>,
                              set_pair_attrs<1, 0, 2>, set_pair_attrs<1, 1, 2>};
    for (auto f : fns)
        if (e == cudaSuccess) e = f();
    return e;
}

int64_t tc_units(int64_t M, int64_t N, int cluster)
{
    const int64_t tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int cl = cluster == 3 ? 2 : 1;
    return ((tiles_m + cl - 1) / cl) * tiles_n;
}

int tc_grid(int64_t M, int64_t N, int sm_count, int cluster, int splits)
{
    const int cl = cluster == 3 ? 2 : 1;
    const int64_t units = tc_units(M, N, cluster) * (splits > 1 ? splits : 1);
    const int64_t clusters = sm_count >= cl ? sm_count / cl : 1;
    return static_cast<int>(cl * (units < clusters ? units : clusters));
}

TcSplit tc_pick_splits(int64_t units, int64_t slots, int64_t K, int elem_bytes, int want)
{
    // Wave model ("GEMM 性能优化", Wave 模型): tile units that fill less than
    // one wave are cut along K so that units x slices fills it.
    TcSplit sp;
    const int64_t k_tiles = (K + (128 / elem_bytes) - 1) / (128 / elem_bytes);
    int64_t s;
    if (want > 1) {
        s = want < k_tiles ? want : k_tiles;
    } else {
        if (want == 1 || units <= 0 || units >= slots) return sp;
        s = slots / units;
        s = s < k_tiles / 4 ? s : k_tiles / 4;
        s = s < 16 ? s : 16;
        // Two slices do not pay for the second launch and the partial tiles
        // (BF16 128 x 14336 x 4096: 35.0 us whole, 38.9 us in two slices).
        if (s < 3) return sp;
    }
    if (s <= 1) return sp;
    const int64_t kt_per = (k_tiles + s - 1) / s;
    sp.splits = static_cast<int>((k_tiles + kt_per - 1) / kt_per);  // no empty slice
    sp.kt_per_split = static_cast<int>(kt_per);
    if (sp.splits <= 1) return TcSplit();
    return sp;
}

size_t tc_partial_bytes(int64_t M, int64_t N, const TcSplit &sp)
{
    if (sp.splits <= 1) return 0;
    const int64_t tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    return static_cast<size_t>(sp.splits) * tiles_m * tiles_n * BM * BN * sizeof(float);
}

cudaError_t launch_tc(int dtype, int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap *tmC, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                      const LaunchCommon &lc, int cluster, bool b_chunks, const TcSplit &sp, bool wide)
{
    TcParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    const int cl = cluster == 3 ? 3 : 1;
    // group_m counts units (tile rows, or tile-row pairs for CTA pairs) along M.
    // Pair MMA: the largest group whose A panel (group x 256 rows x K) stays
    // within 32 MB, a quarter of L2, so it is read from DRAM once while the
    // group sweeps the columns of B ("GEMM 性能优化", Wave 模型与 L2 命中率);
    // 16 for BF16 and 8 for TF32 at K = 4096 (measured best, FFN shape).
    int dflt = 16;
    if (cl == 3) {
        const int64_t panel = int64_t{2 * BM} * K * (dtype == GEMM_BF16 ? 2 : 4);
        const int64_t fit = panel > 0 ? (int64_t{32} << 20) / panel : 16;
        dflt = static_cast<int>(fit < 4 ? 4 : fit > 16 ? 16 : fit);
    }
    p.group_m = lc.group_m > 0 ? lc.group_m : dflt;
    p.C = C;
    p.ldc = ldc;
    p.status = lc.status;
    p.timeout_ns = lc.timeout_ns;
    p.c_vec4 = c_vec4 ? 1 : 0;
    p.c_tma = tmC != nullptr ? 1 : 0;
    p.b_chunks = b_chunks && layout_b == 0 ? 1 : 0;
    p.debug_drop = lc.debug_drop;
    const bool split = sp.splits > 1;
    wide = wide && !split;
    p.splits = split ? sp.splits : 1;
    p.kt_per_split = split ? sp.kt_per_split : (K + (128 / (dtype == GEMM_BF16 ? 2 : 4)) - 1) / (128 / (dtype == GEMM_BF16 ? 2 : 4));
    if (p.kt_per_split < 1) p.kt_per_split = 1;
    p.partials = split ? sp.partials : nullptr;
    // The epilogue spaces a tile's 8 C chunks 25 ns per ring stage of the
    // tile apart, at most 1 us (FFN shape: 1 us), which delays the TMEM
    // release by 7 spacings: at most 5.6 us for the shortest paced tile (32
    // stages, about 9 us of MMAs), so the MMA warp never waits for it.  C
    // writes cost the FFN shape 8 % (BF16) against a copy that skips them;
    // spread over the tile they cost less: interleaved on one box, BF16 /
    // TF32 TFLOP/s 1915 / 995 unpaced, 1925 / 989 at 500 ns, 1941 / 1000 at
    // 1 us, 1917 / 994 at 2 us; at 4 us the release came too late (1342).
    p.epi_pace_ns = cl == 3 && !split && p.kt_per_split >= 32
                        ? static_cast<unsigned>(std::min(1000, 25 * p.kt_per_split))
                        : 0u;
    const CUtensorMap &tc = tmC != nullptr ? *tmC : tmA;  // unused when c_tma == 0
    const bool bf16 = dtype == GEMM_BF16;
    if (cl == 3 && wide) {
        if (bf16) return layout_b == 0 ? launch_pair<0, 0, 2>(tmA, tmB, tc, p, lc.grid, lc.stream)
                                       : launch_pair<0, 1, 2>(tmA, tmB, tc, p, lc.grid, lc.stream);
        return layout_b == 0 ? launch_pair<1, 0, 2>(tmA, tmB, tc, p, lc.grid, lc.stream)
                             : launch_pair<1, 1, 2>(tmA, tmB, tc, p, lc.grid, lc.stream);
    }
    if (cl == 3) {
        if (bf16) return layout_b == 0 ? launch_pair<0, 0, 1>(tmA, tmB, tc, p, lc.grid, lc.stream)
                                       : launch_pair<0, 1, 1>(tmA, tmB, tc, p, lc.grid, lc.stream);
        return layout_b == 0 ? launch_pair<1, 0, 1>(tmA, tmB, tc, p, lc.grid, lc.stream)
                             : launch_pair<1, 1, 1>(tmA, tmB, tc, p, lc.grid, lc.stream);
    }
    if (bf16) return layout_b == 0 ? launch_one<0, 0>(tmA, tmB, tc, p, lc.grid, lc.stream)
                                   : launch_one<0, 1>(tmA, tmB, tc, p, lc.grid, lc.stream);
    return layout_b == 0 ? launch_one<1, 0>(tmA, tmB, tc, p, lc.grid, lc.stream)
                         : launch_one<1, 1>(tmA, tmB, tc, p, lc.grid, lc.stream);
}

}  // namespace dg
