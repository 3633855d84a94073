// FP32 SIMT GEMM for sm_103a: C = A·B with FP32 fused multiply-adds on the
// CUDA cores.
//
// Design, restating the optimisation steps of "GEMM 性能优化" (八个台阶) for
// Blackwell:
//  * 台阶 1 (shared-memory tiling along K): each CTA owns a BM x BN tile of C
//    and walks K in 32-element slices staged in shared memory.
//  * 台阶 2 (thread tiling): every consumer thread keeps an 8 x TN block of C
//    in registers and does 8*TN FMAs per k from 8 A and TN B values.
//  * 台阶 3/4 (vector loads, bank conflicts): the Tensor Memory Accelerator
//    writes each stage with a 128-byte XOR swizzle; every shared load is a
//    16-byte vector and the thread-to-data mapping below makes each warp-wide
//    load hit 32 distinct banks (or broadcast).
//  * 台阶 5 (warp tiling): a warp is 4 x 8 lanes covering 32 rows x 8*TN
//    columns; lanes that share a row group share A loads.
//  * 台阶 6/7 (double buffering, asynchronous copies): a dedicated producer
//    warp issues TMA copies into a multi-stage ring guarded by mbarriers, so
//    global loads overlap the math; fragments of the next k group are loaded
//    while the current one is multiplied.
//  * 台阶 8 (SASS tuning) is replaced by source-level structure: compile-time
//    power-of-two tiles, swizzled offsets computed once per thread, and
//    __launch_bounds__.
//  * Wave model / block order: the grid is persistent and walks tiles in
//    groups of `group_m` tile rows for L2 reuse.
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

constexpr int BK = kSimtBK;  // 32 FP32 = one 128-byte swizzle row

struct SimtParams {
    int M, N, K;
    int tiles_m, tiles_n, group_m;
    int splits;          // K slices per tile (1 = no split)
    int k_per_split;     // elements of K per slice, a multiple of BK
    float *C;
    long long ldc;
    long long split_stride;  // elements between the partial-C slices
    int *status;
    unsigned long long timeout_ns;
    int c_vec4;
    int debug_drop;  // test hook: CTA 0 never loads its first stage
};

// Work unit u (persistent loop index) -> output tile and K slice.
struct Unit {
    int mb, nb, kt_begin, kt_end, split;
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

// Units run slice-major: unit u is tile u % tiles of K slice u / tiles.  The
// K range of slice s is [s*k_per_split, min(K, (s+1)*k_per_split)) ("GEMM
// 性能优化", 台阶 1: partial sums over K slices add up to the product).
__device__ __forceinline__ Unit unit_coords(int u, const SimtParams &p)
{
    const int tiles = p.tiles_m * p.tiles_n;
    Unit w;
    w.split = u / tiles;
    tile_coords(u - w.split * tiles, p, w.mb, w.nb);
    const int k0 = w.split * p.k_per_split;
    const int k1 = min(p.K, k0 + p.k_per_split);
    w.kt_begin = k0 / kSimtBK;
    w.kt_end = (k1 + kSimtBK - 1) / kSimtBK;
    return w;
}

// WM x WN consumer warps; a thread owns 8 rows x TN columns of C; STAGES ring
// slots; GU k-groups (4 k each) per unrolled inner iteration (8 = a whole
// stage); F2 = 1 issues the multiply-adds of row-major B as packed pairs
// (fma.rn.f32x2: two independent FP32 FMAs per instruction, same rounding, so
// the same bits), halving the FMA instructions the scheduler has to issue.
// Column-major B keeps scalar FMAs: its B pairs would have to be assembled
// from two fragments, which costs more issue slots than the packing saves.
//
// LAYOUT_B: 0 = row-major B; 1 = column-major B, read transposed from shared
// memory by the consumers; 2 = column-major B turned in shared memory by the
// producer warp ("PMPP Chapter 06", section 1, corner turning): TMA lands the
// K-contiguous tile, the warp rewrites it in the row-major staging layout,
// and the consumers run the row-major (packed) inner loop.
template <int LAYOUT_B, int WM, int WN, int TN, int STAGES, int GU, int F2>
struct Simt {
    static_assert(WM % 2 == 0, "row interleave pairs warps along M");
    static_assert(TN % 4 == 0 && TN <= 16, "thread tile width");
    static_assert(LAYOUT_B != 1 || TN <= 8, "column-major B uses at most 8 columns per thread");
    static_assert(8 % GU == 0, "k groups per iteration");
    static constexpr int BM = WM * 32;
    static constexpr int BN = WN * 8 * TN;
    static_assert(LAYOUT_B != 2 || BN == 128, "the corner-turn lane mapping covers 128 columns");
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int LAND_BYTES = LAYOUT_B == 2 ? BN * 128 : 0;  // K-major landing zone
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + LAND_BYTES;
    static constexpr int NBAR = LAYOUT_B == 2 ? 3 : 2;  // full, empty (, ready)
    static constexpr int CONSUMER_WARPS = WM * WN;
    static constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NBAR * STAGES * 8 + 16;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
    static_assert(BM <= 256 && BN <= 256, "TMA box limit");
};

template <int LAYOUT_B, int WM, int WN, int TN, int STAGES, int GU, int F2>
__global__ void __launch_bounds__(Simt<LAYOUT_B, WM, WN, TN, STAGES, GU, F2>::THREADS, 1)
    sgemm_simt_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const SimtParams p)
{
    using S = Simt<LAYOUT_B, WM, WN, TN, STAGES, GU, F2>;
    constexpr int BM = S::BM, BN = S::BN, A_BYTES = S::A_BYTES, STAGE_BYTES = S::STAGE_BYTES;
    constexpr int CONSUMER_WARPS = S::CONSUMER_WARPS;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    constexpr int RL = LAYOUT_B == 2 ? 0 : LAYOUT_B;  // layout the consumers read
    constexpr int LAND = A_BYTES + S::B_BYTES;        // landing zone offset (LAYOUT_B == 2)
    const uint32_t full_bar = sbase + STAGES * STAGE_BYTES;  // STAGES x 8 bytes
    const uint32_t empty_bar = full_bar + STAGES * 8;         // STAGES x 8 bytes
    const uint32_t ready_bar = empty_bar + STAGES * 8;        // STAGES x 8 bytes (LAYOUT_B == 2)
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(smem + STAGES * STAGE_BYTES + S::NBAR * STAGES * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_units = p.tiles_m * p.tiles_n * p.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, CONSUMER_WARPS);
            if (LAYOUT_B == 2) mbar_init(ready_bar + 8 * s, 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (LAYOUT_B == 2 && warp == CONSUMER_WARPS) {
        // ------------------------------------------- producer + corner turn
        // Lane 0 keeps the ring STAGES-1 k-tiles ahead; all lanes turn each
        // landed K-major B tile (rows n, 128 bytes of k) into the row-major
        // staging layout (4 boxes of 32 k-rows x 32 columns, 128-byte
        // swizzle) that the consumers read.  Lane (g, t) = (lane/8, lane%8)
        // moves 4x4 blocks of rows 4*(8g+t)..+3 and k-chunk t ^ r (r < 8):
        // inside each group of 8 lanes both the 16-byte reads and the 16-byte
        // writes land on 8 distinct bank groups.
        uint32_t issued = 0;
        int iss_unit = blockIdx.x, iss_kt = 0, iss_kt_end = 0, iss_mb = 0, iss_nb = 0;
        auto iss_load_unit = [&]() {
            if (iss_unit < num_units) {
                const Unit w = unit_coords(iss_unit, p);
                iss_mb = w.mb;
                iss_nb = w.nb;
                iss_kt = w.kt_begin;
                iss_kt_end = w.kt_end;
            }
        };
        // lane 0: issue the next k-tile into its ring slot (bounded wait for the slot)
        auto issue_next = [&]() -> bool {
            const uint32_t slot = issued % STAGES;
            const uint32_t ph = (issued / STAGES) & 1u;
            if (!mbar_wait(empty_bar + 8 * slot, ph ^ 1u, abort_flag, p.status, kWaitProducerEmpty,
                           p.timeout_ns))
                return false;
            const uint32_t fb = full_bar + 8 * slot;
            const uint32_t st = sbase + slot * STAGE_BYTES;
            mbar_arrive_expect_tx(fb, A_BYTES + S::LAND_BYTES);
            if (!(p.debug_drop && blockIdx.x == 0 && issued == 0)) {
                tma_load_2d(st, &tmA, fb, iss_kt * BK, iss_mb * BM);
                tma_load_2d(st + LAND, &tmB, fb, iss_kt * BK, iss_nb * BN);
            }
            ++issued;
            if (++iss_kt >= iss_kt_end) {
                iss_unit += gridDim.x;
                iss_load_unit();
            }
            return true;
        };
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            iss_load_unit();
            for (int i = 0; ok && i < STAGES - 1 && iss_unit < num_units; ++i) ok = issue_next();
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        const int tg = lane >> 3, tt = lane & 7;
        const int nq = 8 * tg + tt;  // rows 4*nq .. 4*nq + 3 of the B tile
        uint32_t it = 0;
        for (int unit = blockIdx.x; ok && unit < num_units; unit += gridDim.x) {
            const Unit w = unit_coords(unit, p);
            for (int kt = w.kt_begin; ok && kt < w.kt_end; ++kt, ++it) {
                const uint32_t s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(full_bar + 8 * s, ph, abort_flag, p.status, kWaitConsumerFull,
                                    p.timeout_ns);
                if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) {
                    ok = false;
                    break;
                }
                const uint8_t *land = smem + s * STAGE_BYTES + LAND;
                uint8_t *brow = smem + s * STAGE_BYTES + A_BYTES + tg * 4096;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int c = tt ^ r;  // k chunk: k = 4c .. 4c + 3
                    float4 v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int n = 4 * nq + q;
                        v[q] = *reinterpret_cast<const float4 *>(land + n * 128 + ((c ^ (n & 7)) << 4));
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = 4 * c + e;
                        const float4 o = e == 0 ? make_float4(v[0].x, v[1].x, v[2].x, v[3].x)
                                       : e == 1 ? make_float4(v[0].y, v[1].y, v[2].y, v[3].y)
                                       : e == 2 ? make_float4(v[0].z, v[1].z, v[2].z, v[3].z)
                                                : make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
                        *reinterpret_cast<float4 *>(brow + k * 128 + ((tt ^ (k & 7)) << 4)) = o;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(ready_bar + 8 * s);
                    if (iss_unit < num_units) ok = issue_next();
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
        }
        if (!ok && lane == 0) {
            // Leave no copy in flight: wait (bounded) for every stage issued
            // but not yet turned.
            for (uint32_t i = it; i < issued; ++i) {
                int dummy = 0;
                mbar_wait(full_bar + 8 * (i % STAGES), (i / STAGES) & 1u, &dummy, nullptr, kWaitDrain,
                          p.timeout_ns);
            }
        }
        return;
    }

    if (warp == CONSUMER_WARPS) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        uint32_t it = 0;
        bool ok = true;
        for (int unit = blockIdx.x; ok && unit < num_units; unit += gridDim.x) {
            const Unit w = unit_coords(unit, p);
            const int mb = w.mb, nb = w.nb;
            for (int kt = w.kt_begin; kt < w.kt_end; ++kt, ++it) {
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
                if (p.debug_drop && blockIdx.x == 0 && it == 0) continue;  // bytes that never come
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
    const int wm = warp % WM;
    const int wn = warp / WM;
    const int lr = lane >> 3;  // 0..3
    const int lc = lane & 7;   // 0..7
    // Rows row0 + 8*i (i < 8): the two warps of a 64-row band interleave by
    // four rows, so row & 7 is fixed per thread and distinct across the four
    // row groups of a warp (conflict-free swizzled A loads).
    const int row0 = (wm >> 1) * 64 + (wm & 1) * 4 + lr;
    const uint32_t xa = row0 & 7;
    const uint32_t a_base = row0 * 128;
    // Row-major B: columns wn*8*TN + 32*c + 4*lc + {0..3} (c < TN/4), i.e.
    // chunk lc of box wn*TN/4 + c; the chunk's place in row k is lc ^ (k & 7).
    // Column-major B: columns col0 + 8*j with col0 & 7 == lc.
    const int col0 = RL == 0 ? wn * 8 * TN + 4 * lc : wn * 8 * TN + lc;
    const uint32_t b_base = RL == 0 ? A_BYTES + wn * (TN / 4) * 4096 : A_BYTES + col0 * 128;

    uint32_t it = 0;
    for (int unit = blockIdx.x; unit < num_units; unit += gridDim.x) {
        const Unit w = unit_coords(unit, p);
        const int mb = w.mb, nb = w.nb;
        // acc2[i][jp] holds columns 2*jp and 2*jp + 1 of row i.
        float2 acc2[8][TN / 2];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) acc2[i][j] = make_float2(0.0f, 0.0f);

        for (int kt = w.kt_begin; kt < w.kt_end; ++kt, ++it) {
            const uint32_t s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!mbar_wait(full_bar + 8 * s, ph, abort_flag, p.status, kWaitConsumerFull,
                           p.timeout_ns))
                return;
            if (LAYOUT_B == 2 && !mbar_wait(ready_bar + 8 * s, ph, abort_flag, p.status,
                                            kWaitConsumerFull, p.timeout_ns))
                return;
            const uint8_t *st = smem + s * STAGE_BYTES;
#pragma unroll 1
            for (int g0 = 0; g0 < 8; g0 += GU) {
#pragma unroll
                for (int h = 0; h < GU; ++h) {
                    const int g = g0 + h;
                    const uint8_t *ap = st + a_base + ((g ^ xa) << 4);
                    float4 a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = *reinterpret_cast<const float4 *>(ap + i * 1024);
                    float4 bcol[RL == 0 ? 1 : TN];
                    if (RL != 0) {
                        const uint8_t *bp = st + b_base + ((g ^ lc) << 4);
#pragma unroll
                        for (int j = 0; j < TN; ++j) bcol[j] = *reinterpret_cast<const float4 *>(bp + j * 1024);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // b2[jp] = columns (2*jp, 2*jp + 1) of B row k = 4*g + kk.
                        float2 b2[TN / 2];
                        if (RL == 0) {
                            const int k = 4 * g + kk;
                            const uint8_t *bp = st + b_base + k * 128 + ((lc ^ (k & 7)) << 4);
#pragma unroll
                            for (int c = 0; c < TN / 4; ++c) {
                                const float4 b4 = *reinterpret_cast<const float4 *>(bp + c * 4096);
                                b2[2 * c] = make_float2(b4.x, b4.y);
                                b2[2 * c + 1] = make_float2(b4.z, b4.w);
                            }
                        } else {
#pragma unroll
                            for (int jp = 0; jp < TN / 2; ++jp) {
                                const float4 u = bcol[2 * jp], v = bcol[2 * jp + 1];
                                b2[jp] = make_float2(kk == 0 ? u.x : kk == 1 ? u.y : kk == 2 ? u.z : u.w,
                                                     kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                            if (F2 && RL == 0) {
                                const float2 aa = make_float2(av, av);
#pragma unroll
                                for (int jp = 0; jp < TN / 2; ++jp) acc2[i][jp] = __ffma2_rn(aa, b2[jp], acc2[i][jp]);
                            } else {
#pragma unroll
                                for (int jp = 0; jp < TN / 2; ++jp) {
                                    acc2[i][jp].x = fmaf(av, b2[jp].x, acc2[i][jp].x);
                                    acc2[i][jp].y = fmaf(av, b2[jp].y, acc2[i][jp].y);
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * s);
        }

        // ------------------------------------------------------ epilogue
        // C itself, or the partial-sum slice of this unit's K range.
        float *cbase = p.C + (long long)w.split * p.split_stride;
        const long long m_base = (long long)mb * BM + row0;
        const int n_base = nb * BN + col0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const long long m = m_base + 8 * i;
            if (m >= p.M) continue;
            float *crow = cbase + m * p.ldc;
            if (RL == 0) {
                // columns 32*c + {0..3}: pairs 2c and 2c + 1
#pragma unroll
                for (int c = 0; c < TN / 4; ++c) {
                    const int n = n_base + 32 * c;
                    const float2 lo = acc2[i][2 * c], hi = acc2[i][2 * c + 1];
                    if (p.c_vec4 && n + 3 < p.N) {
                        *reinterpret_cast<float4 *>(crow + n) = make_float4(lo.x, lo.y, hi.x, hi.y);
                    } else {
                        if (n < p.N) crow[n] = lo.x;
                        if (n + 1 < p.N) crow[n + 1] = lo.y;
                        if (n + 2 < p.N) crow[n + 2] = hi.x;
                        if (n + 3 < p.N) crow[n + 3] = hi.y;
                    }
                }
            } else {
                // column col0 + 8*j is element j & 1 of pair j / 2
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const int n = n_base + 8 * j;
                    if (n < p.N) crow[n] = (j & 1) ? acc2[i][j / 2].y : acc2[i][j / 2].x;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ configs

struct ConfigEntry {
    int bm, bn_row, bn_col, ctas_per_sm;
    const char *name;
    cudaError_t (*prepare)(int *ctas_per_sm);
    void (*launch)(int layout_b, const CUtensorMap &, const CUtensorMap &, const SimtParams &,
                   int grid, cudaStream_t);
};

template <int L, int WM, int WN, int TN, int ST, int GU, int F2>
cudaError_t prepare_one(int *ctas)
{
    using S = Simt<L, WM, WN, TN, ST, GU, F2>;
    auto k = sgemm_simt_kernel<L, WM, WN, TN, ST, GU, F2>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, k, S::THREADS, S::SMEM_BYTES);
    return e;
}

// Row-major B runs the table's TN; column-major B runs min(TN, 8).  A packed
// configuration whose column-major tile is 128 wide turns B in shared memory
// (layout 2, at most 4 stages of 48 KB); the others read it transposed
// (layout 1).
constexpr int col_tn(int tn) { return tn < 8 ? tn : 8; }
constexpr int col_layout(int wn, int tn, int f2) { return (f2 && wn * 8 * col_tn(tn) == 128) ? 2 : 1; }
constexpr int col_stages(int wn, int tn, int f2, int st)
{
    return col_layout(wn, tn, f2) == 2 && st > 4 ? 4 : st;
}

template <int WM, int WN, int TN, int ST, int GU, int F2>
cudaError_t prepare_cfg(int *ctas)
{
    int c0 = 0, c1 = 0;
    cudaError_t e = prepare_one<0, WM, WN, TN, ST, GU, F2>(&c0);
    if (e == cudaSuccess)
        e = prepare_one<col_layout(WN, TN, F2), WM, WN, col_tn(TN), col_stages(WN, TN, F2, ST), GU, F2>(&c1);
    *ctas = c0 < c1 ? c0 : c1;
    return e;
}

template <int WM, int WN, int TN, int ST, int GU, int F2>
void launch_cfg(int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB, const SimtParams &p,
                int grid, cudaStream_t stream)
{
    if (layout_b == 0) {
        using S = Simt<0, WM, WN, TN, ST, GU, F2>;
        sgemm_simt_kernel<0, WM, WN, TN, ST, GU, F2><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    } else {
        constexpr int L = col_layout(WN, TN, F2), CST = col_stages(WN, TN, F2, ST);
        using S = Simt<L, WM, WN, col_tn(TN), CST, GU, F2>;
        sgemm_simt_kernel<L, WM, WN, col_tn(TN), CST, GU, F2><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    }
}

#define DG_SIMT_CFG(WM, WN, TN, ST, GU, F2, NAME)                                              \
    {WM * 32, WN * 8 * TN, WN * 8 * col_tn(TN), 0, NAME, prepare_cfg<WM, WN, TN, ST, GU, F2>,  \
     launch_cfg<WM, WN, TN, ST, GU, F2>}

// Config table; GEMM_OPT_SIMT_CONFIG selects entry (value - 1).
// Measured at 8192^3 on GB300 (row-major B): 128x128 64.6 TFLOP/s, the same
// tile with scalar FMAs 56.4, 64x128 59.2, 64x64 31.5; 8x16 per thread
// (128x256) and 16 warps of 8x4 spill under the 168-register cap that the
// producer warp's sub-partition sets, and run slower.
ConfigEntry g_configs[] = {
    DG_SIMT_CFG(4, 2, 8, 6, 8, 1, "128x128"),
    DG_SIMT_CFG(4, 2, 8, 6, 8, 0, "128x128s"),
    DG_SIMT_CFG(2, 2, 8, 4, 8, 1, "64x128"),
    DG_SIMT_CFG(2, 1, 8, 4, 8, 1, "64x64"),
};
constexpr int kNumConfigs = sizeof(g_configs) / sizeof(g_configs[0]);

}  // namespace

cudaError_t prepare_simt()
{
    for (int i = 0; i < kNumConfigs; ++i) {
        int ctas = 0;
        cudaError_t e = g_configs[i].prepare(&ctas);
        if (e != cudaSuccess) return e;
        g_configs[i].ctas_per_sm = ctas > 0 ? ctas : 1;
    }
    return cudaSuccess;
}

int simt_num_configs() { return kNumConfigs; }

SimtTile simt_tile(int config, int layout_b)
{
    const ConfigEntry &c = g_configs[config];
    return SimtTile{c.bm, layout_b == 0 ? c.bn_row : c.bn_col, c.ctas_per_sm, c.name};
}

int simt_pick_config(int64_t M, int64_t N, int sm_count)
{
    // The 128x128 tile everywhere: a smaller tile does not shorten a
    // thread's serial chain of 64*K multiply-adds, which is what bounds an
    // under-filled launch; split-K does (simt_pick_splits).
    (void)M;
    (void)N;
    (void)sm_count;
    return 0;
}

SplitK simt_pick_splits(int config, int layout_b, int64_t M, int64_t N, int64_t K, int sm_count)
{
    // Wave model ("GEMM 性能优化", Wave 模型): when the tiles fill less than one
    // wave, cut K into slices so tiles x slices fill it, keeping at least
    // four 32-element k-tiles per slice.
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    const int64_t slots = int64_t{sm_count} * t.ctas_per_sm;
    const int64_t k_tiles = (K + kSimtBK - 1) / kSimtBK;
    int64_t s = tiles > 0 ? slots / tiles : 1;
    s = s < k_tiles / 4 ? s : k_tiles / 4;
    s = s < 16 ? s : 16;
    SplitK sk;
    sk.splits = s > 1 ? static_cast<int>(s) : 1;
    if (sk.splits > 1) {
        const int64_t kt_per = (k_tiles + sk.splits - 1) / sk.splits;
        sk.k_per_split = static_cast<int>(kt_per * kSimtBK);
        sk.splits = static_cast<int>((k_tiles + kt_per - 1) / kt_per);  // no empty slice
    }
    return sk;
}

cudaError_t launch_simt_f32(int config, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            int layout_b, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                            const LaunchCommon &lc, const SplitK &sk)
{
    const SimtTile t = simt_tile(config, layout_b);
    SimtParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + t.bm - 1) / t.bm;
    p.tiles_n = (N + t.bn - 1) / t.bn;
    p.group_m = lc.group_m > 0 ? lc.group_m : 8;
    p.splits = sk.splits > 1 ? sk.splits : 1;
    p.k_per_split = p.splits > 1 ? sk.k_per_split : K;
    p.C = p.splits > 1 ? sk.partials : C;
    p.ldc = p.splits > 1 ? N : ldc;
    p.split_stride = static_cast<long long>(M) * N;
    p.status = lc.status;
    p.timeout_ns = lc.timeout_ns;
    p.c_vec4 = p.splits > 1 ? (N % 4 == 0) : (c_vec4 ? 1 : 0);
    p.debug_drop = lc.debug_drop;
    g_configs[config].launch(layout_b, tmA, tmB, p, lc.grid, lc.stream);
    return cudaGetLastError();
}

}  // namespace dg
