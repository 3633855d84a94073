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
#include <cstring>

#include "gemm_internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int BK = kSimtBK;  // 32 FP32 = one 128-byte swizzle row

struct SimtParams {
    int M, N, K;
    int tiles_m, tiles_n, group_m;
    // Units [0, full_units) are whole tiles (tile order position = unit);
    // then the last tail_tiles tiles of the order, each cut into `splits` K
    // slices of k_per_split elements (a multiple of BK), whose partial tiles
    // go to `partials` (slice-major, BM x BN floats each).
    int full_units, tail_tiles, splits, k_per_split;
    float *partials;
    // operands for the element-wise producer (LAYOUT_B == 3)
    const float *A, *B;
    long long lda, ldb;
    float *C;
    long long ldc;
    int *status;
    unsigned long long timeout_ns;
    int c_vec4;
    int debug_drop;  // test hook: CTA 0 never loads its first stage
};

// Work unit u (persistent loop index) -> output tile and K range; split < 0
// means the whole K range, written to C.
struct Unit {
    int mb, nb, kt_begin, kt_end, split, slot;
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

// Whole tiles first; the tail tiles run slice-major, so the slices of one
// tile go to different CTAs of the last wave.  The K range of slice s is
// [s*k_per_split, min(K, (s+1)*k_per_split)) ("GEMM 性能优化", 台阶 1:
// partial sums over K slices add up to the product; Wave 模型: the last,
// partial wave is spread over all CTAs).
__device__ __forceinline__ Unit unit_coords(int u, const SimtParams &p)
{
    Unit w;
    if (u < p.full_units) {
        tile_coords(u, p, w.mb, w.nb);
        w.kt_begin = 0;
        w.kt_end = (p.K + kSimtBK - 1) / kSimtBK;
        w.split = -1;
        w.slot = 0;
        return w;
    }
    const int v = u - p.full_units;
    const int r = v % p.tail_tiles;
    w.split = v / p.tail_tiles;
    w.slot = v;  // = split * tail_tiles + r
    tile_coords(p.full_units + r, p, w.mb, w.nb);
    const int k0 = w.split * p.k_per_split;
    const int k1 = min(p.K, k0 + p.k_per_split);
    w.kt_begin = k0 / kSimtBK;
    w.kt_end = (k1 + kSimtBK - 1) / kSimtBK;
    return w;
}

// Number of K stages (k-tiles) of work unit u, as unit_coords would give
// (kt_end - kt_begin) without the tile coordinates.
__device__ __forceinline__ int unit_stages(int u, const SimtParams &p)
{
    const int k_tiles = (p.K + kSimtBK - 1) / kSimtBK;
    if (u < p.full_units) return k_tiles;
    const int split = (u - p.full_units) / p.tail_tiles;
    const int k0 = split * p.k_per_split;
    const int k1 = min(p.K, k0 + p.k_per_split);
    return (k1 + kSimtBK - 1) / kSimtBK - k0 / kSimtBK;
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
// and the consumers run the row-major (packed) inner loop; 3 = row-major B
// with A or B at a pitch or address TMA cannot use (not a multiple of 16
// bytes): the producer warps copy every element with a 4-byte cp.async
// straight into the swizzled staging layout, zero-filling outside the
// matrices ("GEMM 性能优化", 台阶 7, asynchronous copies).
template <int LAYOUT_B, int WM, int WN, int TN, int STAGES, int GU, int F2, int PWG>
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
    // PWG = 0: one producer warp, registers capped for all warps alike.
    // PWG = 1: a producer warpgroup that gives up registers to the consumer
    // warpgroups (setmaxnreg), so a thread can hold a wider tile of C.
    static constexpr int PRODUCER_WARPS = PWG ? 4 : 1;
    // Column-major B turned in shared memory: with a producer warpgroup, its
    // first warp only issues the TMA copies and the other three turn the
    // tiles (so neither role needs the other's registers); a single producer
    // warp does both.
    static constexpr int TURN_WARPS = PWG ? 3 : 1;
    static constexpr int THREADS = (CONSUMER_WARPS + PRODUCER_WARPS) * 32;
    static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8;  // what __launch_bounds__ allows
    // the corner turn (column-major B) and the element-wise copies need more
    // registers than issuing TMA copies alone
    static constexpr int PRODUCER_REGS =
        CONSUMER_WARPS > 8 ? (LAYOUT_B == 3 ? 40 : LAYOUT_B == 2 ? 32 : 24) : 40;
    static constexpr int CONSUMER_REGS =
        ((LAUNCH_REGS * THREADS - PRODUCER_REGS * PRODUCER_WARPS * 32) / (CONSUMER_WARPS * 32)) / 8 * 8 > 240
            ? 240
            : ((LAUNCH_REGS * THREADS - PRODUCER_REGS * PRODUCER_WARPS * 32) / (CONSUMER_WARPS * 32)) / 8 * 8;
    static_assert(!PWG || (CONSUMER_WARPS % 4 == 0 && LAYOUT_B != 1), "warpgroups; B read as row-major");
    static_assert(LAYOUT_B != 3 || BN % 32 == 0, "element-wise B copies fill 32-column boxes");
    // 16 consumer warps leave 112 registers a thread: A fragments are then
    // loaded 2 k at a time (8-byte loads) instead of 4, to fit.
    static constexpr bool A_PAIRS = CONSUMER_WARPS >= 16;
    // Explicitly double-buffered fragments with the column-pair-major,
    // serpentine multiply-add order (packed FMAs on row-major staging, 8 x 8
    // thread tiles, 8 or 12 consumer warps).
    static constexpr bool PINGPONG = F2 && LAYOUT_B != 1 && !A_PAIRS && GU == 8 && TN == 8 && CONSUMER_WARPS >= 8;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NBAR * STAGES * 8 + 16;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
    static_assert(BM <= 256 && BN <= 256, "TMA box limit");
};

template <int LAYOUT_B, int WM, int WN, int TN, int STAGES, int GU, int F2, int PWG>
__global__ void __launch_bounds__(Simt<LAYOUT_B, WM, WN, TN, STAGES, GU, F2, PWG>::THREADS, 1)
    sgemm_simt_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const SimtParams p)
{
    using S = Simt<LAYOUT_B, WM, WN, TN, STAGES, GU, F2, PWG>;
    constexpr int BM = S::BM, BN = S::BN, A_BYTES = S::A_BYTES, STAGE_BYTES = S::STAGE_BYTES;
    constexpr int CONSUMER_WARPS = S::CONSUMER_WARPS;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    constexpr int RL = LAYOUT_B == 1 ? 1 : 0;  // layout the consumers read
    constexpr int LAND = A_BYTES + S::B_BYTES;        // landing zone offset (LAYOUT_B == 2)
    const uint32_t full_bar = sbase + STAGES * STAGE_BYTES;  // STAGES x 8 bytes
    const uint32_t empty_bar = full_bar + STAGES * 8;         // STAGES x 8 bytes
    const uint32_t ready_bar = empty_bar + STAGES * 8;        // STAGES x 8 bytes (LAYOUT_B == 2)
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(smem + STAGES * STAGE_BYTES + S::NBAR * STAGES * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_units = p.full_units + p.tail_tiles * p.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // TMA: one arrival plus the bytes; element-wise copies: one
            // arrival per producer thread when its copies have landed
            mbar_init(full_bar + 8 * s, LAYOUT_B == 3 ? S::PRODUCER_WARPS * 32 : 1);
            mbar_init(empty_bar + 8 * s, CONSUMER_WARPS);
            if (LAYOUT_B == 2) mbar_init(ready_bar + 8 * s, S::TURN_WARPS);  // every turning warp
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // Every producer role sits inside this one branch, after the register
    // release: ptxas then budgets the consumer code below with the consumers'
    // raised register count alone (producer code reachable after the branch
    // would be compiled under the producers' small count, and spill).
    if (warp >= CONSUMER_WARPS) {
        if (PWG) {
            setmaxnreg_dec<S::PRODUCER_REGS>();
            // one warp of the group issues the copies; with column-major B the
            // others turn the tiles, with element-wise copies all four copy
            if (warp != CONSUMER_WARPS && LAYOUT_B != 2 && LAYOUT_B != 3) return;
        }

        if (LAYOUT_B == 3) {
            // ------------------------------------------- element-wise producer
            // Thread pt of the PT producer threads copies elements pt, pt + PT,
            // ... of the stage: consecutive threads take consecutive k of an A
            // row and consecutive columns of a B row (coalesced reads; each warp
            // writes one 128-byte swizzled row, 32 distinct banks).
            constexpr int PT = S::PRODUCER_WARPS * 32;
            const int pt = threadIdx.x - CONSUMER_WARPS * 32;
            uint32_t it = 0;
            bool ok = true;
            for (int unit = blockIdx.x; ok && unit < num_units; unit += gridDim.x) {
                const Unit w = unit_coords(unit, p);
                for (int kt = w.kt_begin; kt < w.kt_end; ++kt, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    bool got = true;
                    if (lane == 0)
                        got = mbar_wait(empty_bar + 8 * s, ph ^ 1u, abort_flag, p.status, kWaitProducerEmpty,
                                        p.timeout_ns);
                    if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    const int k0 = kt * BK;
                    for (int e = pt; e < BM * BK; e += PT) {
                        const int r = e / BK, kk = e - (e / BK) * BK;
                        const long long m = (long long)w.mb * BM + r;
                        const bool in = m < p.M && k0 + kk < p.K;
                        const uint32_t dst = st + r * 128 + ((((kk >> 2) ^ (r & 7)) << 4) | ((kk & 3) << 2));
                        cp_async_4(dst, in ? p.A + m * p.lda + k0 + kk : p.A, in ? 4u : 0u);
                    }
                    for (int e = pt; e < BK * BN; e += PT) {
                        const int kk = e / BN, n = e - (e / BN) * BN;
                        const long long col = (long long)w.nb * BN + n;
                        const bool in = col < p.N && k0 + kk < p.K;
                        const uint32_t dst = st + A_BYTES + (n >> 5) * 4096 + kk * 128 +
                                             (((((n & 31) >> 2) ^ (kk & 7)) << 4) | ((n & 3) << 2));
                        cp_async_4(dst, in ? p.B + (long long)(k0 + kk) * p.ldb + col : p.B, in ? 4u : 0u);
                    }
                    cp_async_mbar_arrive_noinc(full_bar + 8 * s);
                }
            }
            cp_async_wait_all();  // no copy lands after the CTA has gone
            return;
        }

        if (LAYOUT_B == 2 && PWG && warp == CONSUMER_WARPS) {
            // ------------------------------------- TMA issuer (column-major B)
            // Lane 0 keeps every free ring slot loaded: A and the K-major B tile
            // (into the landing zone).  A slot is free again once the consumers
            // have released it, which they do only after the turn of its tile.
            if (lane != 0) return;
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t it = 0;
            bool ok = true;
            for (int unit = blockIdx.x; ok && unit < num_units; unit += gridDim.x) {
                const Unit w = unit_coords(unit, p);
                for (int kt = w.kt_begin; kt < w.kt_end; ++kt, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait(empty_bar + 8 * s, ph ^ 1u, abort_flag, p.status, kWaitProducerEmpty,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar + 8 * s;
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(fb, A_BYTES + S::LAND_BYTES);
                    if (p.debug_drop && blockIdx.x == 0 && it == 0) continue;  // bytes that never come
                    tma_load_2d(st, &tmA, fb, kt * BK, w.mb * BM);
                    tma_load_2d(st + LAND, &tmB, fb, kt * BK, w.nb * BN);
                }
            }
            if (!ok) {
                // Leave no copy in flight: wait (bounded) for the stages issued last.
                const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
                for (uint32_t i = it - n; i < it; ++i) {
                    int dummy = 0;
                    mbar_wait(full_bar + 8 * (i % STAGES), (i / STAGES) & 1u, &dummy, nullptr, kWaitDrain,
                              p.timeout_ns);
                }
            }
            return;
        }

        if (LAYOUT_B == 2 && PWG) {
            // ------------------------------------------ corner turn (3 warps)
            // Each landed K-major B tile (rows n, 128 bytes of k) is rewritten
            // in the row-major staging layout (4 boxes of 32 k-rows x 32
            // columns, 128-byte swizzle) that the consumers read.  Lane (g, t) =
            // (lane/8, lane%8) moves 4x4 blocks of rows 4*(8g+t)..+3 and k-chunk
            // t ^ r: inside each group of 8 lanes both the 16-byte reads and the
            // 16-byte writes land on 8 distinct bank groups.  Turning warp q
            // (0..2) moves k-chunks r = q, q + 3, q + 6 of every stage and then
            // arrives on the stage's ready barrier (count 3).
            const int q = warp - CONSUMER_WARPS - 1;
            const int tg = lane >> 3, tt = lane & 7;
            const int nq = 8 * tg + tt;  // rows 4*nq .. 4*nq + 3 of the B tile
            uint32_t it = 0;
            for (int unit = blockIdx.x; unit < num_units; unit += gridDim.x) {
                const int stages = unit_stages(unit, p);
                for (int j = 0; j < stages; ++j, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    bool got = true;
                    if (lane == 0)
                        got = mbar_wait(full_bar + 8 * s, ph, abort_flag, p.status, kWaitConsumerFull,
                                        p.timeout_ns);
                    if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) return;
                    // 32-bit shared-memory addresses keep the turn within the
                    // producers' register budget
                    const uint32_t land = sbase + s * STAGE_BYTES + LAND + nq * 512;
                    const uint32_t brow = sbase + s * STAGE_BYTES + A_BYTES + tg * 4096;
#pragma unroll 1
                    for (int r = q; r < 8; r += 3) {
                        const int c = tt ^ r;  // k chunk: k = 4c .. 4c + 3
                        // two rows at a time: rows 4*nq + 2h, +1 become the
                        // 8-byte half h of the four k rows' 16-byte chunks.
                        // The lane groups of odd tg take the halves in the
                        // other order, so each 8-byte store instruction puts
                        // two groups on different banks (2 wavefronts, not 4).
#pragma unroll 1
                        for (int hs = 0; hs < 2; ++hs) {
                            const int h = hs ^ (tg & 1);
                            // row n = 4*nq + e, so n & 7 = 4*(tt & 1) + e
                            const float4 v0 = lds_f4(land + (2 * h) * 128 + ((c ^ (4 * (tt & 1) + 2 * h)) << 4));
                            const float4 v1 = lds_f4(land + (2 * h + 1) * 128 + ((c ^ (4 * (tt & 1) + 2 * h + 1)) << 4));
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int k = 4 * c + e;
                                const float2 o = e == 0 ? make_float2(v0.x, v1.x)
                                               : e == 1 ? make_float2(v0.y, v1.y)
                                               : e == 2 ? make_float2(v0.z, v1.z)
                                                        : make_float2(v0.w, v1.w);
                                sts_f2(brow + k * 128 + ((tt ^ (k & 7)) << 4) + 8 * h, o);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ready_bar + 8 * s);
                }
            }
            return;
        }

        if (LAYOUT_B == 2) {
            // -------------------- single producer warp: issue + corner turn
            // Lane 0 keeps the ring STAGES-1 k-tiles ahead; the warp turns each
            // landed K-major B tile into the row-major staging layout with the
            // lane mapping of the three-warp form above (all 8 k-chunks), then
            // arrives on the stage's ready barrier (count 1).
            constexpr int R_PER = 8 / S::PRODUCER_WARPS;
            const int pw = warp - CONSUMER_WARPS;
            const bool issuer = pw == 0;
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
            if (issuer && lane == 0) {
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
                    for (int rr = 0; rr < R_PER; ++rr) {
                        const int r = pw * R_PER + rr;
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
                        if (issuer && iss_unit < num_units) ok = issue_next();
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                }
            }
            if (!ok && issuer && lane == 0) {
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

        {
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

    }  // producer roles

    if (PWG) setmaxnreg_inc<S::CONSUMER_REGS>();

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

        // A warp whose rows (or columns) of this tile all lie outside C has
        // no multiply-adds to do (the last tile row of 8192 rows in 192-row
        // tiles holds 128 real rows; the last tile column of N = 3073 in
        // 128-column tiles one): it only releases each stage, and the other
        // warps of its scheduler get the FMA pipe.
        const bool idle = (long long)mb * BM + (wm >> 1) * 64 + (wm & 1) * 4 >= p.M ||
                          (long long)nb * BN + wn * 8 * TN >= p.N;

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
            if (idle) {
            } else if (S::PINGPONG) {
                // Fragment double buffering ("GEMM 性能优化", 台阶 6, p-Loop
                // level): the A fragments of k group g+1 and the B fragment of
                // row k+1 are loaded while row k is multiplied.  The packed
                // multiply-adds run column pair by column pair (each B pair
                // serves 8 consecutive instructions) with the row order
                // reversed on every other pair, so the A value at the turn is
                // also reused: 67.2 -> 70.6 TFLOP/s at whole waves on GB300,
                // same bits (each accumulator still sums k in order).
                constexpr int NC = TN / 4;  // 16-byte B chunks per k row
                float4 a[2][8];
                float4 b[2][NC];
                {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        a[0][i] = *reinterpret_cast<const float4 *>(st + a_base + (xa << 4) + i * 1024);
                    const uint8_t *bp = st + b_base + (lc << 4);
#pragma unroll
                    for (int c = 0; c < NC; ++c) b[0][c] = *reinterpret_cast<const float4 *>(bp + c * 4096);
                }
#pragma unroll
                for (int g = 0; g < 8; ++g) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int k = 4 * g + kk;
                        if (k + 1 < BK) {
                            const int kn = k + 1;
                            const uint8_t *bp = st + b_base + kn * 128 + ((lc ^ (kn & 7)) << 4);
#pragma unroll
                            for (int c = 0; c < NC; ++c) b[kn & 1][c] = *reinterpret_cast<const float4 *>(bp + c * 4096);
                        }
                        if (kk == 0 && g + 1 < 8) {
                            const uint8_t *ap = st + a_base + (((g + 1) ^ xa) << 4);
#pragma unroll
                            for (int i = 0; i < 8; ++i) a[(g + 1) & 1][i] = *reinterpret_cast<const float4 *>(ap + i * 1024);
                        }
                        float2 b2[TN / 2];
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            const float4 b4 = b[k & 1][c];
                            b2[2 * c] = make_float2(b4.x, b4.y);
                            b2[2 * c + 1] = make_float2(b4.z, b4.w);
                        }
#pragma unroll
                        for (int jp = 0; jp < TN / 2; ++jp)
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                const int i = (jp & 1) ? 7 - r : r;
                                const float4 ai = a[g & 1][i];
                                const float av = kk == 0 ? ai.x : kk == 1 ? ai.y : kk == 2 ? ai.z : ai.w;
                                acc2[i][jp] = __ffma2_rn(make_float2(av, av), b2[jp], acc2[i][jp]);
                            }
                    }
                }
            } else
#pragma unroll 1
            for (int g0 = 0; g0 < 8; g0 += GU) {
#pragma unroll
                for (int h = 0; h < GU; ++h) {
                    const int g = g0 + h;
                    const uint8_t *ap = st + a_base + ((g ^ xa) << 4);
                    float4 a[S::A_PAIRS ? 1 : 8];
                    float2 a2[S::A_PAIRS ? 8 : 1];
                    if (!S::A_PAIRS) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) a[i] = *reinterpret_cast<const float4 *>(ap + i * 1024);
                    }
                    float4 bcol[RL == 0 ? 1 : TN];
                    if (RL != 0) {
                        const uint8_t *bp = st + b_base + ((g ^ lc) << 4);
#pragma unroll
                        for (int j = 0; j < TN; ++j) bcol[j] = *reinterpret_cast<const float4 *>(bp + j * 1024);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (S::A_PAIRS && (kk & 1) == 0) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                a2[i] = *reinterpret_cast<const float2 *>(ap + i * 1024 + (kk >> 1) * 8);
                        }
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
                            const float av = S::A_PAIRS ? ((kk & 1) ? a2[i].y : a2[i].x)
                                             : kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
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
        if (w.split >= 0) {
            // A partial tile of a K slice: the whole BM x BN tile, rows and
            // columns past M and N included (they hold zeros).
            float *tile = p.partials + (long long)w.slot * (BM * BN);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float *trow = tile + (row0 + 8 * i) * BN;
                if (RL == 0) {
#pragma unroll
                    for (int c = 0; c < TN / 4; ++c) {
                        const float2 lo = acc2[i][2 * c], hi = acc2[i][2 * c + 1];
                        *reinterpret_cast<float4 *>(trow + col0 + 32 * c) = make_float4(lo.x, lo.y, hi.x, hi.y);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < TN; ++j) trow[col0 + 8 * j] = (j & 1) ? acc2[i][j / 2].y : acc2[i][j / 2].x;
                }
            }
            continue;
        }
        const long long m_base = (long long)mb * BM + row0;
        const int n_base = nb * BN + col0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const long long m = m_base + 8 * i;
            if (m >= p.M) continue;
            float *crow = p.C + m * p.ldc;
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

// C for the tail tiles: the sum of their K-slice partial tiles, added in
// slice order s = 0, 1, ... (deterministic; exact for integer data).  One
// thread per 4 consecutive columns of a tile row.
__global__ void __launch_bounds__(256) simt_tail_reduce_kernel(const SimtParams p, int bm, int bn)
{
    const int quads = bm * bn / 4;
    const long long total = (long long)p.tail_tiles * quads;
    const long long tile_elems = (long long)bm * bn;
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int r = static_cast<int>(q / quads);
        const int e = static_cast<int>(q - (long long)r * quads) * 4;
        const int row = e / bn, col = e - (e / bn) * bn;
        int mb, nb;
        tile_coords(p.full_units + r, p, mb, nb);
        const long long m = (long long)mb * bm + row;
        const int n = nb * bn + col;
        if (m >= p.M || n >= p.N) continue;
        const float *src = p.partials + (long long)r * tile_elems + e;
        float4 acc = *reinterpret_cast<const float4 *>(src);
        for (int s = 1; s < p.splits; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(src + (long long)s * p.tail_tiles * tile_elems);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        float *c = p.C + m * p.ldc + n;
        if (p.c_vec4 && n + 3 < p.N) {
            *reinterpret_cast<float4 *>(c) = acc;
        } else {
            c[0] = acc.x;
            if (n + 1 < p.N) c[1] = acc.y;
            if (n + 2 < p.N) c[2] = acc.z;
            if (n + 3 < p.N) c[3] = acc.w;
        }
    }
}

// ------------------------------------------------------------------ configs

struct ConfigEntry {
    int bm, bn_row, bn_col, ctas_per_sm;  // ctas_per_sm 0: not usable on this device
    float rate_row, rate_col;             // measured TFLOP/s in whole waves; 0: not picked automatically
    const char *name;
    cudaError_t (*prepare)(int *ctas_per_sm);
    void (*launch)(int layout_b, const CUtensorMap &, const CUtensorMap &, const SimtParams &,
                   int grid, cudaStream_t);
};

template <int L, int WM, int WN, int TN, int ST, int GU, int F2, int PWG>
cudaError_t prepare_one(int *ctas)
{
    using S = Simt<L, WM, WN, TN, ST, GU, F2, PWG>;
    auto k = sgemm_simt_kernel<L, WM, WN, TN, ST, GU, F2, PWG>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, k, S::THREADS, S::SMEM_BYTES);
    if (e == cudaSuccess && PWG) {
        // setmaxnreg.inc waits until the CTA's launch registers can cover the
        // new counts; refuse the configuration unless they can.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, k);
        const int need = S::CONSUMER_REGS * S::CONSUMER_WARPS * 32 + S::PRODUCER_REGS * S::PRODUCER_WARPS * 32;
        if (e == cudaSuccess && fa.numRegs * S::THREADS < need) *ctas = 0;
    }
    return e;
}

// Row-major B runs the table's TN; column-major B runs min(TN, 8).  A packed
// configuration whose column-major tile is 128 wide turns B in shared memory
// (layout 2, at most 4 stages of 48 KB); the others read it transposed
// (layout 1).
constexpr int col_tn(int tn) { return tn < 8 ? tn : 8; }
constexpr int col_layout(int wn, int tn, int f2) { return (f2 && wn * 8 * col_tn(tn) == 128) ? 2 : 1; }
constexpr int col_stages(int wm, int wn, int tn, int f2, int st)
{
    // at most 4 stages, and as many of A + B + landing zone as fit in 227 KB
    return col_layout(wn, tn, f2) != 2 ? st
           : (st < 4 ? st : 4) < (232448 - 2048) / (wm * 32 * 128 + 2 * wn * 8 * col_tn(tn) * 128)
               ? (st < 4 ? st : 4)
               : (232448 - 2048) / (wm * 32 * 128 + 2 * wn * 8 * col_tn(tn) * 128);
}

// Column-major B uses the producer warpgroup only when it is turned in
// shared memory (layout 2); the transposed-read kernel (layout 1) keeps one
// producer warp.
constexpr int col_pwg(int wn, int tn, int f2, int pwg) { return pwg && col_layout(wn, tn, f2) == 2 ? 1 : 0; }

template <int WM, int WN, int TN, int ST, int GU, int F2, int PWG>
cudaError_t prepare_cfg(int *ctas)
{
    int c0 = 0, c1 = 0, c3 = 0;
    cudaError_t e = prepare_one<0, WM, WN, TN, ST, GU, F2, PWG>(&c0);
    if (e == cudaSuccess)
        e = prepare_one<col_layout(WN, TN, F2), WM, WN, col_tn(TN), col_stages(WM, WN, TN, F2, ST), GU, F2,
                        col_pwg(WN, TN, F2, PWG)>(&c1);
    if (e == cudaSuccess) e = prepare_one<3, WM, WN, TN, ST, GU, F2, PWG>(&c3);
    *ctas = c0 < c1 ? c0 : c1;
    *ctas = *ctas < c3 ? *ctas : c3;
    return e;
}

template <int WM, int WN, int TN, int ST, int GU, int F2, int PWG>
void launch_cfg(int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB, const SimtParams &p,
                int grid, cudaStream_t stream)
{
    if (layout_b == 0) {
        using S = Simt<0, WM, WN, TN, ST, GU, F2, PWG>;
        sgemm_simt_kernel<0, WM, WN, TN, ST, GU, F2, PWG><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    } else if (layout_b == 3) {
        using S = Simt<3, WM, WN, TN, ST, GU, F2, PWG>;
        sgemm_simt_kernel<3, WM, WN, TN, ST, GU, F2, PWG><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    } else {
        constexpr int L = col_layout(WN, TN, F2), CST = col_stages(WM, WN, TN, F2, ST);
        constexpr int CP = col_pwg(WN, TN, F2, PWG);
        using S = Simt<L, WM, WN, col_tn(TN), CST, GU, F2, CP>;
        sgemm_simt_kernel<L, WM, WN, col_tn(TN), CST, GU, F2, CP><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    }
}

#define DG_SIMT_CFG(WM, WN, TN, ST, GU, F2, PWG, RATE_ROW, RATE_COL, NAME)                           \
    {WM * 32,  WN * 8 * TN, WN * 8 * col_tn(TN), 0, RATE_ROW, RATE_COL, NAME,                          \
     prepare_cfg<WM, WN, TN, ST, GU, F2, PWG>, launch_cfg<WM, WN, TN, ST, GU, F2, PWG>}

// Config table; GEMM_OPT_SIMT_CONFIG selects entry (value - 1).  Rates are
// TFLOP/s measured on GB300 at sizes that fill whole waves (M = 7296,
// N = K = 8192); simt_pick_config weighs them against each shape's waves.
// With the double-buffered, column-pair-major inner loop (8 x 8 thread
// tiles): 192x128 with 12 consumer warps 70.3 row-major / 67.1 column-major
// B, 128x128 with 8 consumer warps 69.0 / 63.5.  16 consumer warps of 8 x 4
// (128x128w16, A loaded in pairs, row-pair-major order) 66.6 row-major.
// 64x128 (4 consumer warps) 58.9 / 51.4 and 64x64 (2) 31.5 / 29.3: they win
// only where a problem is a few tiles (128^3: 64x64 11.9 us per call against
// 14.4 for one 128x128 tile), because a CTA's serial work shrinks with its
// tile.  The scalar-FMA tile (56.4 at 8192^3 before the new inner loop),
// 128x256 with register reallocation (8x16 per thread, 64.0) and 16 consumer
// warps of 8x8 with A loaded in pairs (256x128, 112 registers, spills: 59.3)
// never win; they stay selectable.  With scalar FMAs instead of packed pairs
// the 192x128 tile is issue-bound (57.7).
ConfigEntry g_configs[] = {
    DG_SIMT_CFG(4, 2, 8, 6, 8, 1, 0, 69.0f, 63.5f, "128x128"),
    DG_SIMT_CFG(4, 2, 8, 6, 8, 0, 0, 0.0f, 0.0f, "128x128s"),
    DG_SIMT_CFG(2, 2, 8, 4, 8, 1, 0, 58.9f, 51.4f, "64x128"),
    DG_SIMT_CFG(2, 1, 8, 4, 8, 1, 0, 31.5f, 29.3f, "64x64"),
    DG_SIMT_CFG(4, 2, 16, 4, 8, 1, 1, 0.0f, 0.0f, "128x256r"),
    DG_SIMT_CFG(6, 2, 8, 4, 8, 1, 1, 70.3f, 67.1f, "192x128r"),
    DG_SIMT_CFG(4, 4, 4, 6, 8, 1, 1, 66.6f, 0.0f, "128x128w16"),
    DG_SIMT_CFG(8, 2, 8, 4, 8, 1, 1, 0.0f, 0.0f, "256x128r"),
};
constexpr int kNumConfigs = sizeof(g_configs) / sizeof(g_configs[0]);

}  // namespace

cudaError_t prepare_simt()
{
    // A configuration the device cannot run is marked unusable (never picked,
    // refused by GEMM_OPT_SIMT_CONFIG); only the default one must work.
    for (int i = 0; i < kNumConfigs; ++i) {
        int ctas = 0;
        cudaError_t e = g_configs[i].prepare(&ctas);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            if (i == 0) return e;
            ctas = 0;
        }
        g_configs[i].ctas_per_sm = ctas;
    }
    return cudaSuccess;
}

int simt_num_configs() { return kNumConfigs; }

bool simt_config_usable(int config)
{
    return config >= 0 && config < kNumConfigs && g_configs[config].ctas_per_sm > 0;
}

SimtTile simt_tile(int config, int layout_b)
{
    const ConfigEntry &c = g_configs[config];
    return SimtTile{c.bm, layout_b == 0 ? c.bn_row : c.bn_col, c.ctas_per_sm > 0 ? c.ctas_per_sm : 1, c.name};
}

namespace {

// Persistent waves a shape takes on `slots` CTA slots, counting a split
// partial last wave as the fraction of a wave it lasts.
double effective_waves(int config, int layout_b, int64_t M, int64_t N, int64_t K, int64_t slots)
{
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    const SplitK sk = simt_pick_splits(config, layout_b, M, N, K, slots);
    const int64_t tail = sk.splits > 1 ? sk.tail_tiles : 0;
    const double last = tail > 0 ? 1.0 / sk.splits : 0.0;
    return static_cast<double>((tiles - tail + slots - 1) / slots) + last;
}

}  // namespace

int simt_pick_config(int64_t M, int64_t N, int64_t K, int layout_b, int sm_count, int max_ctas)
{
    // The configuration with the least estimated time: effective waves x
    // tile area / measured rate ("GEMM 性能优化", Wave 模型).  A smaller tile
    // does not shorten a thread's serial chain of multiply-adds, which is
    // what bounds an under-filled launch; the K split does.
    int best = 0;
    double best_cost = -1.0;
    for (int c = 0; c < kNumConfigs; ++c) {
        const ConfigEntry &e = g_configs[c];
        const float rate = layout_b == 0 ? e.rate_row : e.rate_col;
        if (rate <= 0.0f || e.ctas_per_sm <= 0) continue;
        const int64_t slots = max_ctas > 0 ? max_ctas : int64_t{sm_count} * e.ctas_per_sm;
        const SimtTile t = simt_tile(c, layout_b);
        const double cost = effective_waves(c, layout_b, M, N, K, slots) * t.bm * t.bn / rate;
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = c;
        }
    }
    return best;
}

SplitK simt_pick_splits(int config, int layout_b, int64_t M, int64_t N, int64_t K, int64_t slots)
{
    // Wave model ("GEMM 性能优化", Wave 模型): the tiles that do not fill a
    // whole wave (all of them when there are fewer tiles than slots) are cut
    // into K slices so that tail x slices fills one wave, each slice at least
    // four 32-element k-tiles long.
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    const int64_t k_tiles = (K + kSimtBK - 1) / kSimtBK;
    SplitK sk;
    if (tiles <= 0 || slots <= 0) return sk;
    const int64_t tail = tiles < slots ? tiles : tiles % slots;
    if (tail == 0) return sk;
    int64_t s = slots / tail;
    s = s < k_tiles / 4 ? s : k_tiles / 4;
    s = s < 16 ? s : 16;
    if (s <= 1) return sk;
    return simt_split_k(tiles, tail, s, K);
}

SplitK simt_split_k(int64_t tiles, int64_t tail, int64_t want, int64_t K)
{
    SplitK sk;
    const int64_t k_tiles = (K + kSimtBK - 1) / kSimtBK;
    if (want > k_tiles) want = k_tiles;
    if (want <= 1 || tail <= 0 || tail > tiles) return sk;
    const int64_t kt_per = (k_tiles + want - 1) / want;
    sk.splits = static_cast<int>((k_tiles + kt_per - 1) / kt_per);  // no empty slice
    if (sk.splits <= 1) return SplitK();
    sk.k_per_split = static_cast<int>(kt_per * kSimtBK);
    sk.tail_tiles = tail;
    return sk;
}

namespace {

SimtParams simt_params(int config, int layout_b, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
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
    const bool split = sk.splits > 1 && sk.tail_tiles > 0;
    p.tail_tiles = split ? static_cast<int>(sk.tail_tiles) : 0;
    p.splits = split ? sk.splits : 1;
    p.k_per_split = split ? sk.k_per_split : K;
    p.full_units = p.tiles_m * p.tiles_n - p.tail_tiles;
    p.partials = split ? sk.partials : nullptr;
    p.C = C;
    p.ldc = ldc;
    p.status = lc.status;
    p.timeout_ns = lc.timeout_ns;
    p.c_vec4 = c_vec4 ? 1 : 0;
    p.debug_drop = lc.debug_drop;
    p.A = nullptr;
    p.B = nullptr;
    p.lda = 0;
    p.ldb = 0;
    return p;
}

}  // namespace

int64_t simt_units(int config, int layout_b, int64_t M, int64_t N, const SplitK &sk)
{
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    return sk.splits > 1 && sk.tail_tiles > 0 ? tiles - sk.tail_tiles + sk.tail_tiles * sk.splits : tiles;
}

size_t simt_partial_bytes(int config, int layout_b, const SplitK &sk)
{
    const SimtTile t = simt_tile(config, layout_b);
    if (sk.splits <= 1 || sk.tail_tiles <= 0) return 0;
    return static_cast<size_t>(sk.splits) * static_cast<size_t>(sk.tail_tiles) * t.bm * t.bn * sizeof(float);
}

cudaError_t launch_simt_f32(int config, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            int layout_b, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                            const LaunchCommon &lc, const SplitK &sk)
{
    const SimtParams p = simt_params(config, layout_b, M, N, K, C, ldc, c_vec4, lc, sk);
    g_configs[config].launch(layout_b, tmA, tmB, p, lc.grid, lc.stream);
    return cudaGetLastError();
}

cudaError_t launch_simt_f32_elementwise(int config, const float *A, int64_t lda, const float *B, int64_t ldb, int M,
                                        int N, int K, float *C, int64_t ldc, bool c_vec4, const LaunchCommon &lc,
                                        const SplitK &sk)
{
    SimtParams p = simt_params(config, 0, M, N, K, C, ldc, c_vec4, lc, sk);
    p.A = A;
    p.B = B;
    p.lda = lda;
    p.ldb = ldb;
    CUtensorMap unused;
    memset(&unused, 0, sizeof unused);
    g_configs[config].launch(3, unused, unused, p, lc.grid, lc.stream);
    return cudaGetLastError();
}

cudaError_t launch_simt_tail_reduce(int config, int layout_b, int M, int N, int K, float *C, int64_t ldc,
                                    bool c_vec4, const LaunchCommon &lc, const SplitK &sk, int sm_count)
{
    const SimtParams p = simt_params(config, layout_b, M, N, K, C, ldc, c_vec4, lc, sk);
    if (p.tail_tiles == 0) return cudaSuccess;
    const SimtTile t = simt_tile(config, layout_b);
    const long long threads = (long long)p.tail_tiles * (t.bm * t.bn / 4);
    long long blocks = (threads + 255) / 256;
    const long long cap = 8LL * (sm_count > 0 ? sm_count : 1);
    if (blocks > cap) blocks = cap;
    simt_tail_reduce_kernel<<<static_cast<int>(blocks), 256, 0, lc.stream>>>(p, t.bm, t.bn);
    return cudaGetLastError();
}

}  // namespace dg
