// Host-side interface between the C ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dg {

// The FP32 SIMT kernel (sgemm_simt.cu) comes in several tile configurations.
// K advances kSimtBK elements (128 bytes) per stage in all of them.  TMA boxes
// (innermost dimension first): A {kSimtBK, bm}; row-major B {32, kSimtBK}
// repeated bn/32 times; column-major B {kSimtBK, bn}.
constexpr int kSimtBK = 32;

struct SimtTile {
    int bm, bn;        // C tile of the configuration for the given B layout
    int ctas_per_sm;   // resident CTAs per SM (persistent grid = SMs x this)
    const char *name;
};

// Split of K for the tail of the tile order: the last tail_tiles tiles (all
// of them for a uniform split) are computed as partial tiles that a second
// kernel sums.  Two forms:
//  * slices (stream_k == 0): each tail tile is cut into `splits` K slices of
//    k_per_split elements; partial tile (slice, tail tile r) at slot
//    slice * tail_tiles + r;
//  * stream-K (stream_k == 1): the tail tiles' k-tile iterations, tile after
//    tile, are cut into sk_parts equal contiguous ranges, one for each of the
//    first sk_parts persistent CTAs (the launch grid must be sk_ctas; there
//    are fewer parts than CTAs only when there are fewer than four k-tiles
//    per CTA); a range that crosses a tile boundary yields one segment per
//    tile it touches.
//    Segment j (in k order) of tail tile r goes to slot r * sk_smax + j.
//    k_per_split holds the longest range, in elements.
struct SplitK {
    int splits = 1;             // slices: 1 = no split, every tile writes C directly
    int k_per_split = 0;        // slices: elements of K per slice (multiple of kSimtBK)
    int64_t tail_tiles = 0;     // tiles cut into slices / segments
    int stream_k = 0;           // 1: stream-K segments instead of equal slices
    int64_t sk_ctas = 0;        // stream-K: CTAs of the launch grid
    int64_t sk_parts = 0;       // stream-K: CTAs with a range, min(sk_ctas, iterations / 4), at least 1
    int64_t sk_smax = 0;        // stream-K: most segments of one tile (slots per tile)
    float *partials = nullptr;  // partial tiles of bm x bn floats
    bool active() const { return tail_tiles > 0 && (stream_k ? sk_parts > 0 : splits > 1); }
    int64_t partial_tiles() const { return !active() ? 0 : stream_k ? tail_tiles * sk_smax : splits * tail_tiles; }
};

int simt_num_configs();
SimtTile simt_tile(int config, int layout_b);
// Configuration for an M x N x K problem on a GPU with sm_count SMs (grid
// capped at max_ctas CTAs when max_ctas > 0).
int simt_pick_config(int64_t M, int64_t N, int64_t K, int layout_b, int sm_count, int max_ctas);
bool simt_config_usable(int config);  // false if the device cannot run it
bool simt_has_stream_k(int config);   // true if it has stream-K kernels (TMA-loaded operands)
// K slices for the tiles of a partial last wave, on `slots` CTA slots.
// stream_k: 0 = slices or stream-K, whichever the wave model rates faster;
// 1 = slices only; 2 = stream-K whenever there is a tail.  A configuration
// without stream-K kernels always takes slices; so must a caller whose
// operands go through the element-wise producer.
SplitK simt_pick_splits(int config, int layout_b, int64_t M, int64_t N, int64_t K, int64_t slots,
                        int stream_k = 0);
// `want` slices (fewer if K is short) of the last `tail` of `tiles` tiles.
SplitK simt_split_k(int64_t tiles, int64_t tail, int64_t want, int64_t K);
// Stream-K over the last `tail` of `tiles` tiles on `ctas` CTAs.
SplitK simt_stream_k(int64_t tiles, int64_t tail, int64_t ctas, int64_t K);
// Work units of the persistent FP32 kernel (the launch grid is at most
// that; with stream-K it is exactly the grid the plan was made for), and
// the workspace its partial tiles need.
int64_t simt_units(int config, int layout_b, int64_t M, int64_t N, const SplitK &sk);
size_t simt_partial_bytes(int config, int layout_b, const SplitK &sk);

// Geometry of the tensor-core kernel (gemm_tc.cu).  A tile of C is
// kTcBM x kTcBN; every stage holds 128 bytes of K per operand row, i.e.
// 64 BF16 or 32 TF32 elements.  TMA boxes (innermost first): A {bk, kTcBM};
// row-major B {128/es, bk}, kTcBN*es/128 boxes per stage; column-major B
// {bk, kTcBoxBCol}, two boxes per stage.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBoxBCol = 128;
constexpr int tc_bk(int elem_bytes) { return 128 / elem_bytes; }

struct LaunchCommon {
    int *status;          // device status word (0 = fine)
    uint64_t timeout_ns;  // limit of every in-kernel wait
    int grid;             // persistent CTAs to launch
    int group_m;          // tile-order group height (tiles)
    cudaStream_t stream;
    int debug_drop = 0;   // test hook: CTA 0 skips the copies of its first stage
};

// Each kernel family raises its dynamic shared-memory limit on the current
// device.  Returns the first CUDA error.
cudaError_t prepare_simt();
cudaError_t prepare_tc();

// FP32 GEMM for small problems (sgemm_small.cu): one 32 x 32 tile of C per
// CTA, A and B read at any pitch and alignment.  simt_small_fits: the
// library's choice of it (at most one tile per SM, K <= 384).
bool simt_small_fits(int64_t M, int64_t N, int64_t K, int sm_count);
cudaError_t launch_simt_small(int layout_b, const float *A, int64_t lda, const float *B, int64_t ldb, float *C,
                              int64_t ldc, int M, int N, int K, cudaStream_t stream);

// FP32 SIMT GEMM with configuration `config`.  tmA maps A (dims {K, M}),
// tmB maps the stored B (row-major: dims {N, K}; column-major: dims {K, N}),
// both FP32 with a 128-byte swizzle and the boxes of simt_tile(config).
// With a split (sk.splits > 1) the kernel writes the tail tiles' slices to
// sk.partials and launch_simt_tail_reduce, queued next with the same
// arguments, sums them into C.
cudaError_t launch_simt_f32(int config, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            int layout_b, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                            const LaunchCommon &lc, const SplitK &sk = SplitK());
// The same for row-major B without TMA: A (pitch lda) and B (pitch ldb) at
// any 4-byte-aligned address and pitch, copied element by element.
cudaError_t launch_simt_f32_elementwise(int config, const float *A, int64_t lda, const float *B, int64_t ldb, int M,
                                        int N, int K, float *C, int64_t ldc, bool c_vec4, const LaunchCommon &lc,
                                        const SplitK &sk = SplitK());
cudaError_t launch_simt_tail_reduce(int config, int layout_b, int M, int N, int K, float *C, int64_t ldc,
                                    bool c_vec4, const LaunchCommon &lc, const SplitK &sk, int sm_count);

// Tensor-core GEMM; dtype is GEMM_TF32 or GEMM_BF16.  tmA/tmB as above.
// tmC (may be null): C as FP32 dims {N, M}, box {32, 32}, 128-byte swizzle,
// used for TMA stores; null means per-thread stores.  cluster = 1 runs one
// CTA per 128x256 tile; cluster = 3 runs the pair MMA (cta_group::2, 256x256
// per pair of CTAs); lc.grid must then be even.
constexpr int kTcBoxC = 32;
// K split of the tensor-core kernels (modes 1 and 3): every tile unit is cut
// into `splits` slices of kt_per_split stages; slice s of tile (mb, nb) goes
// to partials + ((s*tiles_m + mb)*tiles_n + nb)*kTcBM*kTcBN (row-major
// 128 x 256 floats) and launch_tile_split_reduce adds the slices into C.
struct TcSplit {
    int splits = 1;
    int kt_per_split = 0;
    float *partials = nullptr;
};
// Slices for a launch of `units` tile units on `slots` unit slots (CTAs, or
// CTA pairs in mode 3) when they fill at most a third of a wave: 3 to 16
// slices of at least four stages each (want > 1 forces that many).
TcSplit tc_pick_splits(int64_t units, int64_t slots, int64_t K, int elem_bytes, int want);
size_t tc_partial_bytes(int64_t M, int64_t N, const TcSplit &sp);

// b_chunks (row-major B; one-CTA or pair MMA mode): tmB is the 3-D view
// {128-byte column chunk, K, chunk index} with a box of the columns one CTA
// stages (kTcBN, or kTcBN/2 in a pair), fetched by one TMA instruction per
// stage instead of one per chunk.
// wide (pair MMA mode without a K split): three ring stages of two 128-byte
// K slices each instead of six of one (same tensor maps and boxes).
cudaError_t launch_tc(int dtype, int layout_b, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap *tmC, int M, int N, int K, float *C, int64_t ldc, bool c_vec4,
                      const LaunchCommon &lc, int cluster, bool b_chunks, const TcSplit &sp = TcSplit(),
                      bool wide = false);

// Persistent grid of the tensor-core kernel: one CTA per SM, whole clusters.
int tc_grid(int64_t M, int64_t N, int sm_count, int cluster, int splits = 1);
// Tile units of a tensor-core launch (tiles, or tile pairs in mode 3).
int64_t tc_units(int64_t M, int64_t N, int cluster);

// C[m][n] = sum over s of partials[s][mb][nb][m % bm][n % bn], slices added in
// order s = 0, 1, ... (deterministic), for m < M, n < N.
cudaError_t launch_tile_split_reduce(const float *partials, int splits, int64_t tiles_m, int64_t tiles_n, int bm,
                                     int bn, float *C, int64_t ldc, int64_t M, int64_t N, bool c_vec4, int sm_count,
                                     cudaStream_t stream);

// dst[r*ldd + c] = src[r*lds + c] for r < rows, c < cols (elem_bytes 2 or 4).
cudaError_t launch_repack(const void *src, int64_t lds, void *dst, int64_t ldd, int64_t rows,
                          int64_t cols, int elem_bytes, int sm_count, cudaStream_t stream);

// Three-part TF32 split of an FP32 operand (rows x cols at pitch lds) for the
// FP32-accurate tensor-core mode: x = hi + lo, hi = x with its low 13
// mantissa bits cleared, lo = x - hi.  along_rows = false (A, or column-major
// B: K is the column index): dst row r = [p0 | p1 | p2], 3*cols wide;
// along_rows = true (row-major B: K is the row index): dst rows r, r + rows,
// r + 2*rows = p0, p1, p2.  (p0, p1, p2) = (hi, hi, lo) for A, (hi, lo, hi)
// for B (b_side), so A3 B3 = hi(A)hi(B) + hi(A)lo(B) + lo(A)hi(B).
cudaError_t launch_split3(const float *src, int64_t lds, float *dst, int64_t ldd, int64_t rows, int64_t cols,
                          bool along_rows, bool b_side, int sm_count, cudaStream_t stream);

// C[i*ldc + j] = 0 for i < M, j < N.
cudaError_t launch_zero_fill(float *C, int64_t ldc, int64_t M, int64_t N, int sm_count,
                             cudaStream_t stream);


}  // namespace dg
