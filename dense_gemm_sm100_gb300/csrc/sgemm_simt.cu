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
//    16-byte vector, and the thread-to-data mapping below puts the lanes of
//    each quarter-warp on distinct bank groups or one broadcast address, so
//    a load takes the wavefronts its pattern needs and no more (ncu counts
//    bank conflicts at a fraction of a percent of the shared wavefronts).
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
    // go to `partials` (slice-major, BM x BN floats each).  splits == 0:
    // stream-K (sk below) instead of slices.
    int full_units, tail_tiles, splits, k_per_split;
    float *partials;
    // The element-wise producer (LAYOUT_B == 3) has no stream-K form, so its
    // operands and the stream-K plan share the space: the parameter block
    // stays at its size without stream-K (with 40 more bytes the
    // column-major kernel ran 6 % slower, though it never read them).
    union {
        struct {
            const float *A, *B;
            long long lda, ldb;
        } ew;
        // Stream-K: units [base, base + kmax * ctas) are segment k = (u -
        // base) / ctas of CTA c = (u - base) % ctas (the grid is ctas CTAs and
        // base a multiple of it, so CTA c runs them); CTA c < parts owns the
        // tail's k-tile iterations [c * iters / parts, (c + 1) * iters /
        // parts), at least one each.  Units in [full_units, base), of CTAs
        // c >= parts and segments past a CTA's range are empty.  A tail tile
        // has k_tiles iterations and at most smax segments.
        struct {
            long long iters;
            int parts, smax, base, kmax, ctas, k_tiles;
        } sk;
    };
    float *C;
    long long ldc;
    int *status;
    unsigned long long timeout_ns;
    int c_vec4;
    int debug_drop;  // test hook: CTA 0 never loads its first stage
};
static_assert(sizeof(SimtParams) == 120, "keep the parameter block at its measured size");

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

// Stream-K: the CTA owning iteration x of the tail, the last c with
// floor(c * I / P) <= x (P = sk.parts <= I, so every range is non-empty
// and consecutive tiles' owners are consecutive CTAs).
__device__ __forceinline__ long long sk_owner(long long x, const SimtParams &p)
{
    return ((x + 1) * p.sk.parts - 1) / p.sk.iters;
}

// Stream-K range of one CTA, worked out once per CTA (into shared memory)
// so that a unit's coordinates take no 64-bit division: iterations
// [lo, hi), tail tiles r0..r1 (r1 < r0: none), and the segment index of
// its first piece within tile r0.  Every later piece starts its tile, so
// it is that tile's segment 0.
struct SkCta {
    long long lo, hi;
    int r0, r1, split0;
};

__device__ __forceinline__ SkCta sk_cta_range(int c, const SimtParams &p)
{
    SkCta r;
    r.lo = r.hi = 0;
    r.r0 = 0;
    r.r1 = -1;
    r.split0 = 0;
    if (p.splits != 0 || c >= p.sk.parts) return r;
    r.lo = (long long)c * p.sk.iters / p.sk.parts;
    r.hi = (long long)(c + 1) * p.sk.iters / p.sk.parts;
    r.r0 = static_cast<int>(r.lo / p.sk.k_tiles);
    r.r1 = static_cast<int>((r.hi - 1) / p.sk.k_tiles);
    r.split0 = static_cast<int>(c - sk_owner((long long)r.r0 * p.sk.k_tiles, p));
    return r;
}

// Whole tiles first; the tail tiles run slice-major, so the slices of one
// tile go to different CTAs of the last wave.  The K range of slice s is
// [s*k_per_split, min(K, (s+1)*k_per_split)) ("GEMM 性能优化", 台阶 1:
// partial sums over K slices add up to the product; Wave 模型: the last,
// partial wave is spread over all CTAs).  With stream-K every CTA gets an
// equal share of the tail's k-tile iterations instead, cut at tile
// boundaries into segments; a unit with kt_begin == kt_end is empty.
template <bool SK>
__device__ __forceinline__ Unit unit_coords(int u, const SimtParams &p, const SkCta &sc)
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
    if constexpr (SK) {
        // u is a unit of this CTA (u = blockIdx.x + j * gridDim.x), whose
        // range `sc` holds; its k-th segment unit covers tail tile r0 + k
        w.mb = w.nb = 0;
        w.kt_begin = w.kt_end = 0;
        w.split = w.slot = 0;
        if (u < p.sk.base) return w;
        const int k = (u - p.sk.base) / p.sk.ctas;
        const int r = sc.r0 + k;  // tail tile of this segment
        if (r > sc.r1) return w;
        const long long t0 = (long long)r * p.sk.k_tiles;
        w.kt_begin = static_cast<int>((sc.lo > t0 ? sc.lo : t0) - t0);
        w.kt_end = static_cast<int>((sc.hi < t0 + p.sk.k_tiles ? sc.hi : t0 + p.sk.k_tiles) - t0);
        w.split = k == 0 ? sc.split0 : 0;  // segment index within the tile
        w.slot = r * p.sk.smax + w.split;
        tile_coords(p.full_units + r, p, w.mb, w.nb);
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
template <bool SK>
__device__ __forceinline__ int unit_stages(int u, const SimtParams &p, const SkCta &sc)
{
    const int k_tiles = (p.K + kSimtBK - 1) / kSimtBK;
    if (u < p.full_units) return k_tiles;
    if constexpr (SK) {
        const Unit w = unit_coords<SK>(u, p, sc);
        return w.kt_end - w.kt_begin;
    }
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

// SK: the stream-K form (its own instantiation, so the main loop of the
// other form is compiled exactly as without it).
template <int LAYOUT_B, int WM, int WN, int TN, int STAGES, int GU, int F2, int PWG, bool SK>
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
    const int num_units = SK ? p.sk.base + p.sk.kmax * p.sk.ctas : p.full_units + p.tail_tiles * p.splits;
    __shared__ SkCta sk_cta;  // referenced only by the stream-K form

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // TMA: one arrival plus the bytes; element-wise copies: one
            // arrival per producer thread when its copies have landed
            mbar_init(full_bar + 8 * s, LAYOUT_B == 3 ? S::PRODUCER_WARPS * 32 : 1);
            mbar_init(empty_bar + 8 * s, CONSUMER_WARPS);
            if (LAYOUT_B == 2) mbar_init(ready_bar + 8 * s, S::TURN_WARPS);  // every turning warp
        }
        *abort_flag = 0;
        if constexpr (SK) sk_cta = sk_cta_range(blockIdx.x, p);
        fence_barrier_init();
    }
    __syncthreads();
    // the tail reduction, if one follows, may be scheduled now; it waits for
    // this grid to end before it reads anything
    griddep_launch_dependents();

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
                const Unit w = unit_coords<SK>(unit, p, sk_cta);
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
                        cp_async_4(dst, in ? p.ew.A + m * p.ew.lda + k0 + kk : p.ew.A, in ? 4u : 0u);
                    }
                    for (int e = pt; e < BK * BN; e += PT) {
                        const int kk = e / BN, n = e - (e / BN) * BN;
                        const long long col = (long long)w.nb * BN + n;
                        const bool in = col < p.N && k0 + kk < p.K;
                        const uint32_t dst = st + A_BYTES + (n >> 5) * 4096 + kk * 128 +
                                             (((((n & 31) >> 2) ^ (kk & 7)) << 4) | ((n & 3) << 2));
                        cp_async_4(dst, in ? p.ew.B + (long long)(k0 + kk) * p.ew.ldb + col : p.ew.B, in ? 4u : 0u);
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
                const Unit w = unit_coords<SK>(unit, p, sk_cta);
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
                const int stages = unit_stages<SK>(unit, p, sk_cta);
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
            // the next unit of this CTA that has stages (stream-K units can be empty)
            auto iss_load_unit = [&]() {
                for (; iss_unit < num_units; iss_unit += gridDim.x) {
                    const Unit w = unit_coords<SK>(iss_unit, p, sk_cta);
                    if (!SK || w.kt_end > w.kt_begin) {
                        iss_mb = w.mb;
                        iss_nb = w.nb;
                        iss_kt = w.kt_begin;
                        iss_kt_end = w.kt_end;
                        return;
                    }
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
                const Unit w = unit_coords<SK>(unit, p, sk_cta);
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
                const Unit w = unit_coords<SK>(unit, p, sk_cta);
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
        const Unit w = unit_coords<SK>(unit, p, sk_cta);
        if constexpr (SK) {
            if (w.kt_end <= w.kt_begin) continue;  // an empty stream-K unit: no stages, nothing to write
        }
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

// C for the tail tiles: the sum of their partial tiles, added in k order
// (slice s = 0, 1, ... or stream-K segment j = 0, 1, ...; deterministic,
// exact for integer data).  Block (r, c) covers tail tile r, chunk c of its
// groups of 4 columns, one group per thread where the grid allows; thread 0
// works out the tile's coordinates and pieces once for the block.  A
// thread issues the loads of up to 8 pieces before it adds them (in order),
// so they wait out one L2 round trip together, not one each.  Launched as
// a programmatic dependent of the GEMM kernel: it may start before the GEMM
// ends and waits for it in griddep_wait.
__global__ void __launch_bounds__(256) simt_tail_reduce_kernel(const SimtParams p, int bm, int bn)
{
    __shared__ long long s_m_tile, s_base, s_stride;
    __shared__ int s_n_tile, s_parts;
    const int r = blockIdx.x;
    if (threadIdx.x == 0) {
        int mb, nb;
        tile_coords(p.full_units + r, p, mb, nb);
        const long long tile_elems = (long long)bm * bn;
        if (p.splits == 0) {  // stream-K segments j at slot r * smax + j
            const long long t0 = (long long)r * p.sk.k_tiles;
            s_parts = static_cast<int>(sk_owner(t0 + p.sk.k_tiles - 1, p) - sk_owner(t0, p) + 1);
            s_stride = tile_elems;
            s_base = (long long)r * p.sk.smax * tile_elems;
        } else {  // slices s at slot s * tail + r
            s_parts = p.splits;
            s_stride = (long long)p.tail_tiles * tile_elems;
            s_base = (long long)r * tile_elems;
        }
        s_m_tile = (long long)mb * bm;
        s_n_tile = nb * bn;
    }
    __syncthreads();
    const long long m_tile = s_m_tile, stride = s_stride;
    const int n_tile = s_n_tile, parts = s_parts;
    griddep_wait();  // the partial tiles are complete and visible from here on
    const float *base = p.partials + s_base;
    const int quads = bm * bn / 4;
    for (int q = blockIdx.y * blockDim.x + threadIdx.x; q < quads; q += gridDim.y * blockDim.x) {
        const int e = q * 4;
        const int row = e / bn, col = e - row * bn;
        const long long m = m_tile + row;
        const int n = n_tile + col;
        if (m >= p.M || n >= p.N) continue;
        const float *src = base + e;
        float4 v[8];
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (s < parts) v[s] = *reinterpret_cast<const float4 *>(src + s * stride);
        float4 acc = v[0];
#pragma unroll
        for (int s = 1; s < 8; ++s) {
            if (s < parts) {
                acc.x += v[s].x;
                acc.y += v[s].y;
                acc.z += v[s].z;
                acc.w += v[s].w;
            }
        }
        for (int s = 8; s < parts; ++s) {
            const float4 w = *reinterpret_cast<const float4 *>(src + s * stride);
            acc.x += w.x;
            acc.y += w.y;
            acc.z += w.z;
            acc.w += w.w;
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
    bool stream_k;                        // has the stream-K kernels (TMA-loaded operands)
    float rate_row, rate_col;             // measured TFLOP/s in whole waves; 0: not picked automatically
    const char *name;
    cudaError_t (*prepare)(int *ctas_per_sm);
    void (*launch)(int layout_b, const CUtensorMap &, const CUtensorMap &, const SimtParams &,
                   int grid, cudaStream_t);
};

template <int L, int WM, int WN, int TN, int ST, int GU, int F2, int PWG, bool SK>
cudaError_t prepare_one(int *ctas)
{
    using S = Simt<L, WM, WN, TN, ST, GU, F2, PWG>;
    auto k = sgemm_simt_kernel<L, WM, WN, TN, ST, GU, F2, PWG, SK>;
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

// SKF: the configuration also has stream-K kernels for TMA-loaded operands
// (layouts 0, 1 and 2); the element-wise producer (layout 3) always cuts
// the tail into slices.
template <int WM, int WN, int TN, int ST, int GU, int F2, int PWG, bool SKF>
cudaError_t prepare_cfg(int *ctas)
{
    constexpr int CL = col_layout(WN, TN, F2), CST = col_stages(WM, WN, TN, F2, ST);
    constexpr int CT = col_tn(TN), CP = col_pwg(WN, TN, F2, PWG);
    int c0 = 0, c1 = 0, c3 = 0, s0 = 1, s1 = 1;
    cudaError_t e = prepare_one<0, WM, WN, TN, ST, GU, F2, PWG, false>(&c0);
    if (e == cudaSuccess) e = prepare_one<CL, WM, WN, CT, CST, GU, F2, CP, false>(&c1);
    if (e == cudaSuccess) e = prepare_one<3, WM, WN, TN, ST, GU, F2, PWG, false>(&c3);
    if constexpr (SKF) {
        if (e == cudaSuccess) e = prepare_one<0, WM, WN, TN, ST, GU, F2, PWG, true>(&s0);
        if (e == cudaSuccess) e = prepare_one<CL, WM, WN, CT, CST, GU, F2, CP, true>(&s1);
    }
    int c = c0 < c1 ? c0 : c1;
    c = c < c3 ? c : c3;
    c = c < s0 ? c : s0;
    *ctas = c < s1 ? c : s1;
    return e;
}

template <int WM, int WN, int TN, int ST, int GU, int F2, int PWG, bool SK>
void launch_form(int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB, const SimtParams &p,
                 int grid, cudaStream_t stream)
{
    if (layout_b == 0) {
        using S = Simt<0, WM, WN, TN, ST, GU, F2, PWG>;
        sgemm_simt_kernel<0, WM, WN, TN, ST, GU, F2, PWG, SK><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    } else if (layout_b == 3) {
        using S = Simt<3, WM, WN, TN, ST, GU, F2, PWG>;
        sgemm_simt_kernel<3, WM, WN, TN, ST, GU, F2, PWG, false><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    } else {
        constexpr int L = col_layout(WN, TN, F2), CST = col_stages(WM, WN, TN, F2, ST);
        constexpr int CP = col_pwg(WN, TN, F2, PWG);
        using S = Simt<L, WM, WN, col_tn(TN), CST, GU, F2, CP>;
        sgemm_simt_kernel<L, WM, WN, col_tn(TN), CST, GU, F2, CP, SK><<<grid, S::THREADS, S::SMEM_BYTES, stream>>>(tmA, tmB, p);
    }
}

template <int WM, int WN, int TN, int ST, int GU, int F2, int PWG, bool SKF>
void launch_cfg(int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB, const SimtParams &p,
                int grid, cudaStream_t stream)
{
    if constexpr (SKF) {
        if (p.splits == 0) {
            launch_form<WM, WN, TN, ST, GU, F2, PWG, true>(layout_b, tmA, tmB, p, grid, stream);
            return;
        }
    }
    launch_form<WM, WN, TN, ST, GU, F2, PWG, false>(layout_b, tmA, tmB, p, grid, stream);
}

#define DG_SIMT_CFG(WM, WN, TN, ST, GU, F2, PWG, SKF, RATE_ROW, RATE_COL, NAME)                      \
    {WM * 32,  WN * 8 * TN, WN * 8 * col_tn(TN), 0, SKF, RATE_ROW, RATE_COL, NAME,                     \
     prepare_cfg<WM, WN, TN, ST, GU, F2, PWG, SKF>, launch_cfg<WM, WN, TN, ST, GU, F2, PWG, SKF>}

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
ConfigEntry g_tile_table[] = {
    DG_SIMT_CFG(4, 2, 8, 6, 8, 1, 0, true, 69.0f, 63.5f, "128x128"),
    DG_SIMT_CFG(4, 2, 8, 6, 8, 0, 0, false, 0.0f, 0.0f, "128x128s"),
    DG_SIMT_CFG(2, 2, 8, 4, 8, 1, 0, true, 58.9f, 51.4f, "64x128"),
    DG_SIMT_CFG(2, 1, 8, 4, 8, 1, 0, true, 31.5f, 29.3f, "64x64"),
    DG_SIMT_CFG(4, 2, 16, 4, 8, 1, 1, false, 0.0f, 0.0f, "128x256r"),
    DG_SIMT_CFG(6, 2, 8, 4, 8, 1, 1, true, 70.3f, 67.1f, "192x128r"),
    DG_SIMT_CFG(4, 4, 4, 6, 8, 1, 1, false, 66.6f, 0.0f, "128x128w16"),
    DG_SIMT_CFG(8, 2, 8, 4, 8, 1, 1, false, 0.0f, 0.0f, "256x128r"),
};
constexpr int kNumConfigs = sizeof(g_tile_table) / sizeof(g_tile_table[0]);

}  // namespace

cudaError_t prepare_simt()
{
    // A configuration the device cannot run is marked unusable (never picked,
    // refused by GEMM_OPT_SIMT_CONFIG); only the default one must work.
    for (int i = 0; i < kNumConfigs; ++i) {
        int ctas = 0;
        cudaError_t e = g_tile_table[i].prepare(&ctas);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            if (i == 0) return e;
            ctas = 0;
        }
        g_tile_table[i].ctas_per_sm = ctas;
    }
    return cudaSuccess;
}

int simt_num_configs() { return kNumConfigs; }

bool simt_has_stream_k(int config)
{
    return config >= 0 && config < kNumConfigs && g_tile_table[config].stream_k;
}

bool simt_config_usable(int config)
{
    return config >= 0 && config < kNumConfigs && g_tile_table[config].ctas_per_sm > 0;
}

SimtTile simt_tile(int config, int layout_b)
{
    const ConfigEntry &c = g_tile_table[config];
    return SimtTile{c.bm, layout_b == 0 ? c.bn_row : c.bn_col, c.ctas_per_sm > 0 ? c.ctas_per_sm : 1, c.name};
}

namespace {

// Estimated time of an M x N x K product on `config` ("GEMM 性能优化",
// Wave 模型), in units of 2K / 1e12 seconds.  The measured whole-wave rate
// is with ctas_per_sm CTAs on every SM; a CTA that shares its SM with k - 1
// others is taken to run at 1/k of the SM's share of that rate, so its tile
// takes k x tile area x SMs / rate.  Whole rounds of `slots` tiles, then
// the partial last round: n CTAs, each running its share g of a tile's K
// (1 without a split; else the longest slice or stream-K range).
double simt_cost(int config, int layout_b, int64_t M, int64_t N, int64_t K, int sm_count, int64_t slots,
                 float rate)
{
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    const int64_t sms = sm_count > 0 ? sm_count : 1;
    const double tile = double(t.bm) * double(t.bn) * double(sms) / double(rate);
    auto sharing = [&](int64_t n) {  // CTAs per SM when n run at once
        int64_t k = (n + sms - 1) / sms;
        k = k < t.ctas_per_sm ? k : t.ctas_per_sm;
        return double(k > 1 ? k : 1);
    };
    const SplitK sk = simt_pick_splits(config, layout_b, M, N, K, slots);
    const int64_t tail = sk.active() ? sk.tail_tiles : 0;
    const int64_t whole = tiles - tail;
    double cost = double(whole / slots) * tile * sharing(slots);
    if (whole % slots) cost += tile * sharing(whole % slots);
    if (tail > 0) {
        const int64_t k_tiles = (K + kSimtBK - 1) / kSimtBK;
        const double g = double(sk.k_per_split / kSimtBK) / double(k_tiles);
        const int64_t n = sk.stream_k ? sk.sk_parts : tail * sk.splits;
        cost += g * tile * sharing(n);
    }
    return cost;
}

}  // namespace

int simt_pick_config(int64_t M, int64_t N, int64_t K, int layout_b, int sm_count, int max_ctas)
{
    // The configuration with the least estimated time (simt_cost).  A
    // smaller tile does not shorten a thread's serial chain of
    // multiply-adds, which is what bounds an under-filled launch; the K
    // split does.
    int best = 0;
    double best_cost = -1.0;
    for (int c = 0; c < kNumConfigs; ++c) {
        const ConfigEntry &e = g_tile_table[c];
        const float rate = layout_b == 0 ? e.rate_row : e.rate_col;
        if (rate <= 0.0f || e.ctas_per_sm <= 0) continue;
        const int64_t slots = max_ctas > 0 ? max_ctas : int64_t{sm_count} * e.ctas_per_sm;
        const double cost = simt_cost(c, layout_b, M, N, K, sm_count, slots, rate);
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = c;
        }
    }
    return best;
}

SplitK simt_pick_splits(int config, int layout_b, int64_t M, int64_t N, int64_t K, int64_t slots, int stream_k)
{
    // Wave model ("GEMM 性能优化", Wave 模型): the tiles that do not fill a
    // whole wave (all of them when there are fewer tiles than slots) are cut
    // along K.  Slices: tail x slices fills one wave, each slice at least
    // four 32-element k-tiles long, so the last wave lasts 1/slices of a
    // wave.  Stream-K: the tail's k-tiles, tile after tile, are shared out
    // in equal contiguous ranges (at least four k-tiles each) over up to
    // `slots` CTAs, crossing tile boundaries, so the last wave lasts the
    // longest range over k-tiles.  Stream-K is taken when that is shorter
    // (1024^3 as 128x128 tiles: 14/32 against 16/32 of a wave; 8192^3 as
    // 192x128 tiles: 27/256 against 29/256, measured 0.5 % faster); on a tie,
    // slices.
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    const int64_t k_tiles = (K + kSimtBK - 1) / kSimtBK;
    SplitK sk;
    if (tiles <= 0 || slots <= 0 || k_tiles <= 0) return sk;
    const int64_t tail = tiles < slots ? tiles : tiles % slots;
    if (tail == 0) return sk;
    int64_t s = slots / tail;
    s = s < k_tiles / 4 ? s : k_tiles / 4;
    s = s < 16 ? s : 16;
    const SplitK sliced = s > 1 ? simt_split_k(tiles, tail, s, K) : SplitK();
    if (stream_k == 1 || !simt_has_stream_k(config)) return sliced;
    const SplitK streamed = simt_stream_k(tiles, tail, slots, K);
    if (stream_k == 2) return streamed;
    const double f_slices = sliced.active() ? double(sliced.k_per_split / kSimtBK) / double(k_tiles) : 1.0;
    const double f_stream = streamed.active() ? double(streamed.k_per_split / kSimtBK) / double(k_tiles) : 1.0;
    return f_stream < f_slices ? streamed : sliced;
}

SplitK simt_stream_k(int64_t tiles, int64_t tail, int64_t ctas, int64_t K)
{
    SplitK sk;
    const int64_t k_tiles = (K + kSimtBK - 1) / kSimtBK;
    if (tail <= 0 || tail > tiles || ctas <= 0 || k_tiles <= 0) return sk;
    const int64_t iters = tail * k_tiles;
    // ranges of at least four k-tiles, as for slices (shorter ones cost more
    // in partial tiles and fills than they save)
    const int64_t most = iters / 4 > 1 ? iters / 4 : 1;
    const int64_t parts = ctas < most ? ctas : most;
    const int64_t per = (iters + parts - 1) / parts;  // longest range of one CTA
    sk.stream_k = 1;
    sk.tail_tiles = tail;
    sk.sk_ctas = ctas;
    sk.sk_parts = parts;
    // every range is at least floor(iters / parts) >= 1 iterations long, so
    // the ranges meeting one tile's k_tiles iterations number at most
    // ceil(k_tiles / floor(iters / parts)) + 1
    const int64_t min_len = iters / parts;
    sk.sk_smax = (k_tiles + min_len - 1) / min_len + 1;
    if (sk.sk_smax > parts) sk.sk_smax = parts;
    sk.splits = 1;
    sk.k_per_split = static_cast<int>(per * kSimtBK);
    return sk;
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
    memset(&p, 0, sizeof p);
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + t.bm - 1) / t.bm;
    p.tiles_n = (N + t.bn - 1) / t.bn;
    p.group_m = lc.group_m > 0 ? lc.group_m : 8;
    const bool split = sk.active();
    const bool streamed = split && sk.stream_k;
    p.tail_tiles = split ? static_cast<int>(sk.tail_tiles) : 0;
    p.splits = streamed ? 0 : split ? sk.splits : 1;
    p.k_per_split = split ? sk.k_per_split : K;
    p.full_units = p.tiles_m * p.tiles_n - p.tail_tiles;
    p.partials = split ? sk.partials : nullptr;
    if (streamed) {
        p.sk.k_tiles = (K + kSimtBK - 1) / kSimtBK;
        p.sk.ctas = static_cast<int>(sk.sk_ctas);
        p.sk.parts = static_cast<int>(sk.sk_parts);
        p.sk.smax = static_cast<int>(sk.sk_smax);
        p.sk.iters = (long long)p.tail_tiles * p.sk.k_tiles;
        // units of the whole tiles, rounded up to whole rounds of the grid,
        // then each CTA's segments: a range of at most ceil(I / P) iterations
        // spans at most ceil(ceil(I / P) / k_tiles) + 1 tiles
        p.sk.base = (p.full_units + p.sk.ctas - 1) / p.sk.ctas * p.sk.ctas;
        p.sk.kmax = static_cast<int>(((p.sk.iters + p.sk.parts - 1) / p.sk.parts + p.sk.k_tiles - 1) / p.sk.k_tiles + 1);
    }
    p.C = C;
    p.ldc = ldc;
    p.status = lc.status;
    p.timeout_ns = lc.timeout_ns;
    p.c_vec4 = c_vec4 ? 1 : 0;
    p.debug_drop = lc.debug_drop;
    return p;
}

}  // namespace

int64_t simt_units(int config, int layout_b, int64_t M, int64_t N, const SplitK &sk)
{
    const SimtTile t = simt_tile(config, layout_b);
    const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
    if (!sk.active()) return tiles;
    if (!sk.stream_k) return tiles - sk.tail_tiles + sk.tail_tiles * sk.splits;
    // The launch grid must be sk_ctas CTAs, each running its whole tiles and
    // then its segments (the kernel counts those itself); this is the grid.
    return sk.sk_ctas;
}

size_t simt_partial_bytes(int config, int layout_b, const SplitK &sk)
{
    const SimtTile t = simt_tile(config, layout_b);
    return static_cast<size_t>(sk.partial_tiles()) * t.bm * t.bn * sizeof(float);
}

cudaError_t launch_simt_f32(int config, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            int layout_b, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                            const LaunchCommon &lc, const SplitK &sk)
{
    const SimtParams p = simt_params(config, layout_b, M, N, K, C, ldc, c_vec4, lc, sk);
    g_tile_table[config].launch(layout_b, tmA, tmB, p, lc.grid, lc.stream);
    return cudaGetLastError();
}

cudaError_t launch_simt_f32_elementwise(int config, const float *A, int64_t lda, const float *B, int64_t ldb, int M,
                                        int N, int K, float *C, int64_t ldc, bool c_vec4, const LaunchCommon &lc,
                                        const SplitK &sk)
{
    if (sk.active() && sk.stream_k) return cudaErrorInvalidValue;  // the element-wise form has no stream-K
    SimtParams p = simt_params(config, 0, M, N, K, C, ldc, c_vec4, lc, sk);
    p.ew.A = A;
    p.ew.B = B;
    p.ew.lda = lda;
    p.ew.ldb = ldb;
    CUtensorMap unused;
    memset(&unused, 0, sizeof unused);
    g_tile_table[config].launch(3, unused, unused, p, lc.grid, lc.stream);
    return cudaGetLastError();
}

cudaError_t launch_simt_tail_reduce(int config, int layout_b, int M, int N, int K, float *C, int64_t ldc,
                                    bool c_vec4, const LaunchCommon &lc, const SplitK &sk, int sm_count)
{
    const SimtParams p = simt_params(config, layout_b, M, N, K, C, ldc, c_vec4, lc, sk);
    if (p.tail_tiles == 0) return cudaSuccess;
    const SimtTile t = simt_tile(config, layout_b);
    // one group of 4 columns of a tile per thread (blocks of 256 threads)
    const int quads = t.bm * t.bn / 4;
    const int chunks = quads / 256 > 0 ? quads / 256 : 1;
    (void)sm_count;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.tail_tiles), static_cast<unsigned>(chunks > 0 ? chunks : 1), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, simt_tail_reduce_kernel, p, t.bm, t.bn);
}

}  // namespace dg
