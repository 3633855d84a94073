// The C ABI of include/gemm.h: argument checks, dispatch to the kernels,
// TMA tensor-map encoding, the handle's workspace, and the host-buffer entry.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <new>
#include <string>

#include "../../include/gemm.h"
#include "gemm_internal.h"

struct gemm_ctx {
    int device = 0;
    int sm_count = 0;
    int *d_status = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    // Recorded on the caller's stream after every call that used the
    // workspace; growth waits on it (stream-ordered) before the old buffer
    // is released.
    cudaEvent_t ws_event = nullptr;
    bool ws_event_recorded = false;
    std::string last_error;
    std::string last_path;
    int64_t launches = 0;
    int force_repack = 0;
    uint64_t timeout_ns = 4000000000ull;
    int simt_group_m = 0;
    int tc_group_m = 0;
    int max_ctas = 0;
    int simt_config = 0;  // 0: chosen per shape; else configuration index + 1
    int elementwise = 0;  // FP32 unaligned operands: element-wise producer (1) or re-pack (0)
    size_t ws_limit = 0;  // 0: none; else the workspace never grows beyond this many bytes
    int split_k = 0;      // 0: chosen per shape; 1: never; n > 1: n K slices (FP32 path)
    int stream_k = 0;     // FP32 tail: 0 chosen per shape, 1 slices, 2 stream-K
    int simt_small = 0;   // FP32 small-problem kernel: 0 chosen per shape, 1 never, 2 always
    int tc_cluster = 3;   // tensor-core mode: 1 one CTA per tile, 3 pair MMA
    int tc_tma_store = 1; // tensor-core epilogue writes C with TMA stores when C allows it
    int tc_slices = 0;    // pair MMA: K slices per ring stage (0: library's choice)
    int debug_drop = 0;   // test hook (GEMM_OPT_DEBUG_DROP_LOAD)
    // gemm_run_host pipeline: copy streams and events (created on first use)
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_a[16] = {}, ev_b[8] = {}, ev_c[16 * 8] = {};  // row panels, column panels, blocks
};

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1024;  // kernels index tiles with int
constexpr int64_t kMaxLd = int64_t{1} << 36;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode()
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

int elem_bytes(int dtype) { return dtype == GEMM_BF16 ? 2 : 4; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int fail(gemm_ctx *h, int code, const std::string &msg)
{
    if (h) h->last_error = msg;
    return code;
}

int cuda_fail(gemm_ctx *h, cudaError_t e, const char *what)
{
    cudaGetLastError();  // clear a non-sticky error so the next call starts clean
    return fail(h, GEMM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Shared by gemm_validate, gemm_run and gemm_run_host.
int check_args(int layout_b, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
               const void *B, int64_t ldb, const void *C, int64_t ldc, int dtype,
               std::string *why)
{
    auto bad = [&](int code, const char *msg) {
        if (why) *why = msg;
        return code;
    };
    if (layout_b != GEMM_B_ROW_MAJOR && layout_b != GEMM_B_COL_MAJOR)
        return bad(GEMM_ERR_INVALID, "layout_b must be GEMM_B_ROW_MAJOR or GEMM_B_COL_MAJOR");
    if (dtype != GEMM_F32 && dtype != GEMM_TF32 && dtype != GEMM_BF16 && dtype != GEMM_F32_3XTF32)
        return bad(GEMM_ERR_INVALID, "dtype must be GEMM_F32, GEMM_TF32, GEMM_BF16 or GEMM_F32_3XTF32");
    if (M < 0 || N < 0 || K < 0) return bad(GEMM_ERR_INVALID, "M, N and K must be >= 0");
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return bad(GEMM_ERR_INVALID, "M, N and K must be below 2^31 - 1024");
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return bad(GEMM_ERR_INVALID, "C is NULL");
    if (ldc < N || ldc > kMaxLd) return bad(GEMM_ERR_INVALID, "ldc must satisfy N <= ldc <= 2^36");
    if (reinterpret_cast<uintptr_t>(C) % 4) return bad(GEMM_ERR_ALIGNMENT, "C is not 4-byte aligned");
    if (K == 0) return GEMM_OK;
    if (!A || !B) return bad(GEMM_ERR_INVALID, "A or B is NULL");
    if (lda < K || lda > kMaxLd) return bad(GEMM_ERR_INVALID, "lda must satisfy K <= lda <= 2^36");
    if (layout_b == GEMM_B_ROW_MAJOR && (ldb < N || ldb > kMaxLd))
        return bad(GEMM_ERR_INVALID, "row-major B needs N <= ldb <= 2^36");
    if (layout_b == GEMM_B_COL_MAJOR && (ldb < K || ldb > kMaxLd))
        return bad(GEMM_ERR_INVALID, "column-major B needs K <= ldb <= 2^36");
    const uintptr_t es = static_cast<uintptr_t>(elem_bytes(dtype));
    if (reinterpret_cast<uintptr_t>(A) % es || reinterpret_cast<uintptr_t>(B) % es)
        return bad(GEMM_ERR_ALIGNMENT, "A or B is not aligned to its element size");
    return GEMM_OK;
}

bool tma_ready(const void *p, int64_t ld, int es)
{
    return reinterpret_cast<uintptr_t>(p) % 16 == 0 && (ld * es) % 16 == 0;
}

// Workspace a run needs: re-packed operands (when not TMA-ready) followed by
// the split-K partial products of the FP32 path.
struct PackPlan {
    bool small = false;        // FP32 small-problem kernel: reads A and B where they are
    bool a = false, b = false;
    bool elementwise = false;  // FP32, row-major B: copy unaligned operands element-wise instead
    int64_t lda = 0, ldb = 0;
    size_t a_bytes = 0, b_bytes = 0;
    int simt_config = 0;
    dg::SplitK split;     // partials pointer is filled in by run_device
    dg::TcSplit tc_split; // tensor-core K split (partials filled in by run_device)
    size_t split_bytes = 0;  // partial tiles of either split
    size_t total() const { return a_bytes + b_bytes + split_bytes; }
};

// Tensor-core mode for an M-row problem: the configured CTA-pair mode needs
// more than one 128-row tile row.
int tc_cluster_for(const gemm_ctx *h, int64_t M) { return h->tc_cluster == 3 && M > dg::kTcBM ? 3 : 1; }

PackPlan plan_pack(const gemm_ctx *h, int layout_b, int64_t M, int64_t N, int64_t K,
                   const void *A, int64_t lda, const void *B, int64_t ldb, int dtype)
{
    PackPlan pp;
    if (M == 0 || N == 0 || K == 0) return pp;
    if (dtype == GEMM_F32_3XTF32) {
        // The split operands always live in the workspace: A3 is M x 3K, B3
        // 3K x N (row-major) or N x 3K (column-major), 16-byte pitches; then
        // a TF32 product over 3K, planned as such.
        const int64_t K3 = 3 * K;
        const bool row = layout_b == GEMM_B_ROW_MAJOR;
        pp.a = pp.b = true;
        pp.lda = round_up(K3, 4);
        pp.a_bytes = static_cast<size_t>(round_up(M * pp.lda * 4, 256));
        pp.ldb = round_up(row ? N : K3, 4);
        pp.b_bytes = static_cast<size_t>(round_up((row ? K3 : N) * pp.ldb * 4, 256));
        const int cluster = tc_cluster_for(h, M);
        const int64_t ctas = h->max_ctas > 0 ? h->max_ctas : h->sm_count;
        const int64_t slots = cluster == 3 ? ctas / 2 : ctas;
        pp.tc_split = dg::tc_pick_splits(dg::tc_units(M, N, cluster), slots, K3, 4, h->split_k);
        pp.split_bytes = static_cast<size_t>(
            round_up(static_cast<int64_t>(dg::tc_partial_bytes(M, N, pp.tc_split)), 256));
        return pp;
    }
    if (dtype == GEMM_F32 && !h->force_repack &&
        (h->simt_small == 2 || (h->simt_small == 0 && h->simt_config == 0 && h->max_ctas == 0 &&
                                h->split_k == 0 && dg::simt_small_fits(M, N, K, h->sm_count)))) {
        pp.small = true;  // no workspace: any pitch and alignment
        return pp;
    }
    const int es = elem_bytes(dtype);
    const int64_t align_elems = 16 / es;
    pp.a = h->force_repack || !tma_ready(A, lda, es);
    pp.b = h->force_repack || !tma_ready(B, ldb, es);
    if (dtype == GEMM_F32 && layout_b == GEMM_B_ROW_MAJOR && !h->force_repack && h->elementwise &&
        (pp.a || pp.b)) {
        pp.elementwise = true;  // the producer reads A and B where they are
        pp.a = pp.b = false;
    }
    if (pp.a) {
        pp.lda = round_up(K, align_elems);
        pp.a_bytes = static_cast<size_t>(round_up(M * pp.lda * es, 256));
    }
    if (pp.b) {
        const int64_t rows = layout_b == GEMM_B_ROW_MAJOR ? K : N;
        const int64_t cols = layout_b == GEMM_B_ROW_MAJOR ? N : K;
        pp.ldb = round_up(cols, align_elems);
        pp.b_bytes = static_cast<size_t>(round_up(rows * pp.ldb * es, 256));
    }
    if (dtype == GEMM_F32) {
        pp.simt_config = h->simt_config > 0 ? h->simt_config - 1 : dg::simt_pick_config(M, N, K, layout_b, h->sm_count, h->max_ctas);
        const dg::SimtTile t = dg::simt_tile(pp.simt_config, layout_b);
        if (h->split_k == 0) {
            const int64_t slots = h->max_ctas > 0 ? h->max_ctas : int64_t{h->sm_count} * t.ctas_per_sm;
            // the element-wise producer has no stream-K form
            pp.split = dg::simt_pick_splits(pp.simt_config, layout_b, M, N, K, slots,
                                            pp.elementwise ? 1 : h->stream_k);
        } else if (h->split_k > 1) {  // every tile in split_k slices
            const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
            pp.split = dg::simt_split_k(tiles, tiles, h->split_k, K);
        }
        pp.split_bytes = static_cast<size_t>(
            round_up(static_cast<int64_t>(dg::simt_partial_bytes(pp.simt_config, layout_b, pp.split)), 256));
    } else {
        const int cluster = tc_cluster_for(h, M);
        const int64_t ctas = h->max_ctas > 0 ? h->max_ctas : h->sm_count;
        const int64_t slots = cluster == 3 ? ctas / 2 : ctas;
        pp.tc_split = dg::tc_pick_splits(dg::tc_units(M, N, cluster), slots, K, es, h->split_k);
        pp.split_bytes = static_cast<size_t>(
            round_up(static_cast<int64_t>(dg::tc_partial_bytes(M, N, pp.tc_split)), 256));
    }
    return pp;
}

// Grows the workspace in stream order on `stream`: the stream first waits
// for the last call that used the old buffer, then frees it and allocates
// the new one from the device's stream-ordered pool.  Nothing waits on the
// host, and work the caller queued on other streams is not held up.
int ensure_workspace(gemm_ctx *h, size_t need, cudaStream_t stream)
{
    if (need <= h->ws_bytes) return GEMM_OK;
    if (h->ws_limit > 0 && need > h->ws_limit) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "workspace of %zu bytes needed, limit %zu (GEMM_OPT_WORKSPACE_LIMIT)", need,
                      h->ws_limit);
        return fail(h, GEMM_ERR_NOMEM, msg);
    }
    size_t grow = h->ws_bytes + h->ws_bytes / 2;
    size_t bytes = need > grow ? need : grow;
    bytes = (bytes + (size_t{2} << 20) - 1) & ~((size_t{2} << 20) - 1);
    if (h->ws_limit > 0 && bytes > h->ws_limit) bytes = need;  // stay within the limit
    cudaError_t e = cudaSuccess;
    if (h->ws) {
        // Earlier calls (on this or another stream) may still read the old buffer.
        if (h->ws_event_recorded) e = cudaStreamWaitEvent(stream, h->ws_event, 0);
        if (e == cudaSuccess) e = cudaFreeAsync(h->ws, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "stream-ordered release of the old workspace");
    }
    h->ws = nullptr;
    h->ws_bytes = 0;
    h->ws_event_recorded = false;
    e = cudaMallocAsync(&h->ws, bytes, stream);
    if (e != cudaSuccess) {
        h->ws = nullptr;
        cudaGetLastError();
        return fail(h, GEMM_ERR_NOMEM, std::string("workspace cudaMallocAsync: ") + cudaGetErrorString(e));
    }
    h->ws_bytes = bytes;
    return GEMM_OK;
}

// After a call whose launches read or write the workspace: its end on
// `stream` is what the next growth waits for.
int note_workspace_use(gemm_ctx *h, cudaStream_t stream)
{
    cudaError_t e = cudaEventRecord(h->ws_event, stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "workspace-use event");
    h->ws_event_recorded = true;
    return GEMM_OK;
}

int encode_2d(gemm_ctx *h, CUtensorMap *map, int es, const void *base, int64_t inner,
              int64_t outer, int64_t ld, int box_inner, int box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld operand",
                      static_cast<int>(r), static_cast<long long>(outer), static_cast<long long>(inner));
        return fail(h, GEMM_ERR_CUDA, msg);
    }
    return GEMM_OK;
}

// Row-major B as a 3-D tensor of 128-byte column chunks: {column in chunk,
// k, chunk}, strides ld*es and chunk*es bytes.  Only for N a multiple of the
// chunk, so no box reaches past the last row of B.
int encode_b_chunks(gemm_ctx *h, CUtensorMap *map, int es, const void *base, int64_t N, int64_t K, int64_t ld,
                    int box_k, int box_chunks, CUtensorMapSwizzle swizzle)
{
    const int64_t chunk = 128 / es;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(chunk), static_cast<cuuint64_t>(K),
                                static_cast<cuuint64_t>(N / chunk)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * es, static_cast<cuuint64_t>(chunk) * es};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(chunk), static_cast<cuuint32_t>(box_k),
                               static_cast<cuuint32_t>(box_chunks)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUresult r = g_encode(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled (3-D B chunks) failed (%d)", static_cast<int>(r));
        return fail(h, GEMM_ERR_CUDA, msg);
    }
    return GEMM_OK;
}

class DeviceGuard {
  public:
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        if (prev_ != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
    }

  private:
    int prev_ = -1;
};

// Queue C = A·B on device buffers.  The workspace must already hold
// `ws_offset + plan.total()` bytes; packed operands go after ws_offset.
int run_device(gemm_ctx *h, int layout_b, int64_t M, int64_t N, int64_t K, const void *A,
               int64_t lda, const void *B, int64_t ldb, float *C, int64_t ldc, int dtype,
               cudaStream_t stream, const PackPlan &pp, size_t ws_offset)
{
    if (M == 0 || N == 0) {
        h->last_path = "noop";
        return GEMM_OK;
    }
    if (K == 0) {
        cudaError_t e = dg::launch_zero_fill(C, ldc, M, N, h->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "zero-fill launch");
        ++h->launches;
        h->last_path = "zero_fill";
        return GEMM_OK;
    }
    const int es = elem_bytes(dtype);
    std::string path;
    uint8_t *ws = static_cast<uint8_t *>(h->ws) + ws_offset;
    const int64_t rows_b = layout_b == GEMM_B_ROW_MAJOR ? K : N;
    const int64_t cols_b = layout_b == GEMM_B_ROW_MAJOR ? N : K;
    const bool split3 = dtype == GEMM_F32_3XTF32;
    if (split3) {
        // FP32-accurate tensor-core mode: split A and B into TF32 parts
        // (three along K) and run the TF32 path over 3K on them.
        float *A3 = reinterpret_cast<float *>(ws);
        float *B3 = reinterpret_cast<float *>(ws + pp.a_bytes);
        cudaError_t e = dg::launch_split3(static_cast<const float *>(A), lda, A3, pp.lda, M, K, false, false,
                                          h->sm_count, stream);
        if (e == cudaSuccess)
            e = dg::launch_split3(static_cast<const float *>(B), ldb, B3, pp.ldb, rows_b, cols_b,
                                  layout_b == GEMM_B_ROW_MAJOR, true, h->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "operand split launch");
        h->launches += 2;
        A = A3;
        lda = pp.lda;
        B = B3;
        ldb = pp.ldb;
        K *= 3;
        dtype = GEMM_TF32;
        path += "+split3";
    }
    if (pp.a && !split3) {
        cudaError_t e = dg::launch_repack(A, lda, ws, pp.lda, M, K, es, h->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "repack A launch");
        ++h->launches;
        A = ws;
        lda = pp.lda;
        path += "+repackA";
    }
    if (pp.b && !split3) {
        void *dst = ws + pp.a_bytes;
        cudaError_t e = dg::launch_repack(B, ldb, dst, pp.ldb, rows_b, cols_b, es, h->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "repack B launch");
        ++h->launches;
        B = dst;
        ldb = pp.ldb;
        path += "+repackB";
    }

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    const bool c_vec4 = reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 4 == 0;
    dg::LaunchCommon lc;
    lc.status = h->d_status;
    lc.timeout_ns = h->timeout_ns;
    lc.stream = stream;
    lc.debug_drop = h->debug_drop;
    const char *lay = layout_b == GEMM_B_ROW_MAJOR ? "rowB" : "colB";
    int rc;
    if (dtype == GEMM_F32 && pp.small) {
        cudaError_t e = dg::launch_simt_small(layout_b, static_cast<const float *>(A), lda,
                                              static_cast<const float *>(B), ldb, C, ldc, static_cast<int>(M),
                                              static_cast<int>(N), static_cast<int>(K), stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "FP32 small-problem kernel launch");
        path = std::string("simt_f32_small32x32_") + lay + path;
    } else if (dtype == GEMM_F32) {
        const int cfg = pp.simt_config;
        const dg::SimtTile t = dg::simt_tile(cfg, layout_b);
        if (!pp.elementwise) {
            rc = encode_2d(h, &tmA, 4, A, K, M, lda, dg::kSimtBK, t.bm);
            if (rc) return rc;
            if (layout_b == GEMM_B_ROW_MAJOR)
                rc = encode_2d(h, &tmB, 4, B, N, K, ldb, 32, dg::kSimtBK);
            else
                rc = encode_2d(h, &tmB, 4, B, K, N, ldb, dg::kSimtBK, t.bn);
            if (rc) return rc;
        }
        dg::SplitK sk = pp.split;
        if (sk.active()) sk.partials = reinterpret_cast<float *>(ws + pp.a_bytes + pp.b_bytes);
        const int64_t units = dg::simt_units(cfg, layout_b, M, N, sk);
        const int64_t cap = h->max_ctas > 0 ? h->max_ctas : int64_t{h->sm_count} * t.ctas_per_sm;
        lc.grid = static_cast<int>(units < cap ? units : cap);
        lc.group_m = h->simt_group_m;
        cudaError_t e =
            pp.elementwise
                ? dg::launch_simt_f32_elementwise(cfg, static_cast<const float *>(A), lda, static_cast<const float *>(B),
                                                  ldb, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), C,
                                                  ldc, c_vec4, lc, sk)
                : dg::launch_simt_f32(cfg, tmA, tmB, layout_b, static_cast<int>(M), static_cast<int>(N),
                                      static_cast<int>(K), C, ldc, c_vec4, lc, sk);
        if (e != cudaSuccess) return cuda_fail(h, e, "FP32 SIMT kernel launch");
        path = std::string("simt_f32_") + t.name + "_" + lay + (pp.elementwise ? "+cpasync" : "") + path;
        if (sk.active()) {
            ++h->launches;
            e = dg::launch_simt_tail_reduce(cfg, layout_b, static_cast<int>(M), static_cast<int>(N),
                                            static_cast<int>(K), C, ldc, c_vec4, lc, sk, h->sm_count);
            if (e != cudaSuccess) return cuda_fail(h, e, "split-K reduction launch");
            const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
            if (sk.stream_k)
                path += "+streamk" + std::to_string(sk.tail_tiles) + "on" + std::to_string(sk.sk_parts);
            else
                path += sk.tail_tiles == tiles ? "+splitk" + std::to_string(sk.splits)
                                               : "+tail" + std::to_string(sk.tail_tiles) + "x" + std::to_string(sk.splits);
        }
    } else {
        const int bk = dg::tc_bk(es);
        rc = encode_2d(h, &tmA, es, A, K, M, lda, bk, dg::kTcBM);
        if (rc) return rc;
        const int cluster = tc_cluster_for(h, M);
        // MN-major B; 32-bit elements need 32-byte swizzle atoms there.
        const CUtensorMapSwizzle b_swz = es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
        const bool b_chunks = layout_b == GEMM_B_ROW_MAJOR && N % (128 / es) == 0;
        if (b_chunks)
            rc = encode_b_chunks(h, &tmB, es, B, N, K, ldb, bk, (cluster == 3 ? dg::kTcBN / 2 : dg::kTcBN) / (128 / es),
                                 b_swz);
        else if (layout_b == GEMM_B_ROW_MAJOR)
            rc = encode_2d(h, &tmB, es, B, N, K, ldb, 128 / es, bk, b_swz);
        else
            rc = encode_2d(h, &tmB, es, B, K, N, ldb, bk, dg::kTcBoxBCol);
        if (rc) return rc;
        dg::TcSplit sp = pp.tc_split;
        if (sp.splits > 1) sp.partials = reinterpret_cast<float *>(ws + pp.a_bytes + pp.b_bytes);
        int grid = dg::tc_grid(M, N, h->max_ctas > 0 ? h->max_ctas : h->sm_count, cluster, sp.splits);
        lc.grid = grid;
        lc.group_m = h->tc_group_m;
        alignas(64) CUtensorMap tmC;
        const bool c_tma = c_vec4 && h->tc_tma_store && sp.splits == 1;
        if (c_tma) {
            rc = encode_2d(h, &tmC, 4, C, N, M, ldc, dg::kTcBoxC, dg::kTcBoxC);
            if (rc) return rc;
        }
        const bool wide = cluster == 3 && sp.splits == 1 && h->tc_slices == 2;
        cudaError_t e = dg::launch_tc(dtype, layout_b, tmA, tmB, c_tma ? &tmC : nullptr, static_cast<int>(M),
                                      static_cast<int>(N), static_cast<int>(K), C, ldc, c_vec4, lc, cluster,
                                      b_chunks, sp, wide);
        if (e != cudaSuccess) return cuda_fail(h, e, "tensor-core kernel launch");
        path = std::string(split3 ? "f32x3_tc_tf32" : dtype == GEMM_BF16 ? "tc_bf16" : "tc_tf32") +
               (cluster == 3 ? (wide ? "_pair256x256w_" : "_pair256x256_") : "_128x256_") + lay +
               (b_chunks ? "+b3d" : "") + path;
        if (sp.splits > 1) {
            ++h->launches;
            e = dg::launch_tile_split_reduce(sp.partials, sp.splits, (M + dg::kTcBM - 1) / dg::kTcBM,
                                             (N + dg::kTcBN - 1) / dg::kTcBN, dg::kTcBM, dg::kTcBN, C, ldc, M, N,
                                             c_vec4, h->sm_count, stream);
            if (e != cudaSuccess) return cuda_fail(h, e, "split-K reduction launch");
            path += "+splitk" + std::to_string(sp.splits);
        }
    }
    ++h->launches;
    h->last_path = path;
    return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_version(void) { return GEMM_VERSION; }

const char *gemm_status_string(int code)
{
    switch (code) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID: return "GEMM_ERR_INVALID";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_DEVICE: return "GEMM_ERR_DEVICE";
    case GEMM_ERR_NOMEM: return "GEMM_ERR_NOMEM";
    default: return "unknown gemm status";
    }
}

int gemm_create(gemm_handle_t *out, int device)
{
    if (!out) return GEMM_ERR_INVALID;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();
        return GEMM_ERR_DEVICE;
    }
    if (device < 0 || device >= count) return GEMM_ERR_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_DEVICE;
    }
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_DEVICE;  // built for sm_103a only
    gemm_ctx *h = new (std::nothrow) gemm_ctx;
    if (!h) return GEMM_ERR_NOMEM;
    h->device = device;
    h->sm_count = prop.multiProcessorCount;
    DeviceGuard guard(device);
    std::call_once(g_encode_once, load_encode);
    cudaError_t e = g_encode ? cudaSuccess : cudaErrorNotSupported;
    if (e == cudaSuccess) e = dg::prepare_simt();
    if (e == cudaSuccess) e = dg::prepare_tc();
    if (e == cudaSuccess) e = cudaMalloc(&h->d_status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ws_event, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (h->d_status) cudaFree(h->d_status);
        if (h->ws_event) cudaEventDestroy(h->ws_event);
        delete h;
        return GEMM_ERR_CUDA;
    }
    *out = h;
    return GEMM_OK;
}

int gemm_destroy(gemm_handle_t h)
{
    if (!h) return GEMM_OK;
    {
        DeviceGuard guard(h->device);
        cudaDeviceSynchronize();
        if (h->ws) {
            cudaFreeAsync(h->ws, nullptr);  // allocated from the stream-ordered pool
            cudaStreamSynchronize(nullptr);
        }
        if (h->d_status) cudaFree(h->d_status);
        if (h->ws_event) cudaEventDestroy(h->ws_event);
        if (h->copy_in) cudaStreamDestroy(h->copy_in);
        if (h->copy_out) cudaStreamDestroy(h->copy_out);
        for (cudaEvent_t ev : {h->ev_start, h->ev_done})
            if (ev) cudaEventDestroy(ev);
        for (cudaEvent_t ev : h->ev_a)
            if (ev) cudaEventDestroy(ev);
        for (cudaEvent_t ev : h->ev_b)
            if (ev) cudaEventDestroy(ev);
        for (cudaEvent_t ev : h->ev_c)
            if (ev) cudaEventDestroy(ev);
    }
    delete h;
    return GEMM_OK;
}

int gemm_validate(int layout_b, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                  const void *B, int64_t ldb, const float *C, int64_t ldc, int dtype)
{
    return check_args(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, nullptr);
}

int gemm_run(gemm_handle_t h, int layout_b, int64_t M, int64_t N, int64_t K, const void *A,
             int64_t lda, const void *B, int64_t ldb, float *C, int64_t ldc, int dtype,
             cudaStream_t stream)
{
    if (!h) return GEMM_ERR_INVALID;
    std::string why;
    int rc = check_args(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, &why);
    if (rc) return fail(h, rc, why);
    DeviceGuard guard(h->device);
    const PackPlan pp = plan_pack(h, layout_b, M, N, K, A, lda, B, ldb, dtype);
    if (pp.total()) {
        rc = ensure_workspace(h, pp.total(), stream);
        if (rc) return rc;
    }
    rc = run_device(h, layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream, pp, 0);
    if (rc == GEMM_OK && pp.total()) rc = note_workspace_use(h, stream);
    return rc;
}

namespace {

constexpr int kMaxRowPanels = 16, kMaxColPanels = 8;

int ensure_pipeline(gemm_ctx *h)
{
    if (h->copy_in) return GEMM_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking);
    for (cudaEvent_t *ev : {&h->ev_start, &h->ev_done})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    const auto create = [&](cudaEvent_t *evs, int n) {
        for (int i = 0; i < n && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&evs[i], cudaEventDisableTiming);
    };
    create(h->ev_a, kMaxRowPanels);
    create(h->ev_b, kMaxColPanels);
    create(h->ev_c, kMaxRowPanels * kMaxColPanels);
    return e == cudaSuccess ? GEMM_OK : cuda_fail(h, e, "creating the host-copy pipeline");
}

int64_t gcd64(int64_t a, int64_t b)
{
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// How gemm_run_host cuts C into blocks: the first pm-1 row panels of A
// (rows each) times pn column panels of B (cols each), one launch per block,
// then the last row panel times all of B in one launch.  With pm == 1 the
// only row panel is cut into the pn column blocks.
struct HostBlocks {
    int64_t rows = 0, cols = 0;
    int pm = 1, pn = 1;
};

// Output tile, tile slots of one persistent wave, for the kernel the
// problem will run on.
void tile_shape(const gemm_ctx *h, int layout_b, int64_t M, int64_t N, int64_t K, int dtype, int64_t *bm,
                int64_t *bn, int64_t *slots, int64_t *full_slots)
{
    if (dtype == GEMM_F32) {
        const int cfg = h->simt_config > 0 ? h->simt_config - 1
                                           : dg::simt_pick_config(M, N, K, layout_b, h->sm_count, h->max_ctas);
        const dg::SimtTile t = dg::simt_tile(cfg, layout_b);
        *bm = t.bm;
        *bn = t.bn;
        *full_slots = int64_t{h->sm_count} * t.ctas_per_sm;
        *slots = h->max_ctas > 0 ? h->max_ctas : *full_slots;
    } else {
        const bool pair = h->tc_cluster == 3;
        const int64_t ctas = h->max_ctas > 0 ? h->max_ctas : h->sm_count;
        *bm = pair ? 2 * dg::kTcBM : dg::kTcBM;  // a pair covers two tile rows
        *bn = dg::kTcBN;
        *slots = pair ? ctas / 2 : ctas;
        *full_slots = pair ? h->sm_count / 2 : h->sm_count;
    }
    if (*slots < 1) *slots = 1;
    if (*full_slots < *slots) *full_slots = *slots;
}

// Blocks for the host-buffer pipeline.  While one block runs, the copy of
// the operand panels of the next in and of the previous block's C out proceed
// on their own streams, so only the first block's operands and the last
// launch's C are not hidden.  Blocks of the first row panels are whole
// persistent waves, at least two ("GEMM 性能优化", Wave 模型); the last row
// panel spans all columns, so its partial wave is shared as in one call.
// Candidates: one block, and 1, 2, 4 or 8 column panels; the one with the
// least estimated time wins.
HostBlocks plan_host_blocks(const gemm_ctx *h, int layout_b, int64_t M, int64_t N, int64_t K, int dtype)
{
    HostBlocks best;
    best.rows = M;
    best.cols = N;
    if (K == 0) return best;
    const int es = elem_bytes(dtype);
    int64_t bm, bn, slots, full_slots;
    tile_shape(h, layout_b, M, N, K, dtype, &bm, &bn, &slots, &full_slots);
    const auto waves = [&](int64_t mp, int64_t np) {
        const int64_t tiles = ((mp + bm - 1) / bm) * ((np + bn - 1) / bn);
        return (tiles + slots - 1) / slots;
    };
    // Rough rates of these kernels on all SMs and of the host link; they only
    // rank plans.  A wave takes as long with fewer slots (GEMM_OPT_MAX_CTAS).
    const double rate = dtype == GEMM_F32           ? 64e12
                        : dtype == GEMM_TF32        ? 800e12
                        : dtype == GEMM_F32_3XTF32 ? 270e12
                                                    : 1650e12;  // FLOP/s
    const double link = 200e9;                                                             // bytes/s each way
    const double wave_s = 2.0 * bm * bn * K * full_slots / rate;
    const double h2d_all = (double(M) * K + double(K) * N) * es, d2h_all = double(M) * N * 4;
    const auto estimate = [&](int64_t w, int launches, double head, double tail) {
        const double body = std::max({w * wave_s, (h2d_all - head) / link, (d2h_all - tail) / link});
        return head / link + body + tail / link + launches * 10e-6;
    };
    double best_s = estimate(waves(M, N), 1, h2d_all, d2h_all);
    for (int pn_try = 1; pn_try <= kMaxColPanels; pn_try *= 2) {
        const int64_t cols = round_up((N + pn_try - 1) / pn_try, bn);
        const int pn = static_cast<int>((N + cols - 1) / cols);
        if (pn != pn_try) continue;
        const int64_t last_cols = N - (pn - 1) * cols;
        const int64_t tiles_n = cols / bn;
        int64_t unit = slots / gcd64(slots, tiles_n);  // fewest tile rows that fill whole waves
        if (unit > 64) {
            if (pn > 1) continue;  // column panels only where waves come out whole
            unit = 1;
        }
        int64_t bands = unit;
        while (bands * tiles_n < 2 * slots) bands += unit;
        int64_t rows = bands * bm;
        if ((M + rows - 1) / rows > kMaxRowPanels) rows = round_up((M + kMaxRowPanels - 1) / kMaxRowPanels, unit * bm);
        if (rows >= M) rows = M;
        const int pm = static_cast<int>((M + rows - 1) / rows);
        if (pm == 1 && pn == 1) continue;  // the one-block plan, estimated above
        const int64_t last_rows = M - (pm - 1) * rows;
        const int64_t panel_rows = pm > 1 ? rows : M;
        int64_t w = int64_t{pm > 1 ? pm - 1 : 1} * ((pn - 1) * waves(panel_rows, cols) + waves(panel_rows, last_cols));
        if (pm > 1) w += waves(last_rows, N);
        const int launches = (pm > 1 ? pm - 1 : 1) * pn + (pm > 1 ? 1 : 0);
        const double head = (double(panel_rows) + (pn > 1 ? cols : N)) * K * es;
        const double tail = pm > 1 ? double(last_rows) * N * 4 : double(M) * last_cols * 4;
        const double t = estimate(w, launches, head, tail);
        if (t < best_s) {
            best_s = t;
            best.rows = panel_rows;
            best.cols = cols;
            best.pm = pm;
            best.pn = pn;
        }
    }
    return best;
}

}  // namespace

int gemm_run_host(gemm_handle_t h, int layout_b, int64_t M, int64_t N, int64_t K, const void *A_host,
                  int64_t lda, const void *B_host, int64_t ldb, float *C_host, int64_t ldc,
                  int dtype, cudaStream_t stream)
{
    if (!h) return GEMM_ERR_INVALID;
    std::string why;
    int rc = check_args(layout_b, M, N, K, A_host, lda, B_host, ldb, C_host, ldc, dtype, &why);
    if (rc) return fail(h, rc, why);
    if (M == 0 || N == 0) {
        h->last_path = "noop";
        return GEMM_OK;
    }
    DeviceGuard guard(h->device);
    rc = ensure_pipeline(h);
    if (rc) return rc;
    const int es = elem_bytes(dtype);
    const bool b_row = layout_b == GEMM_B_ROW_MAJOR;
    const int64_t al = 16 / es;
    const int64_t rows_b = b_row ? K : N;
    const int64_t cols_b = b_row ? N : K;
    const int64_t lda_d = K ? round_up(K, al) : 0;
    const int64_t ldb_d = K ? round_up(cols_b, al) : 0;
    const int64_t ldc_d = round_up(N, 4);
    const size_t a_bytes = static_cast<size_t>(round_up(M * lda_d * es, 256));
    const size_t b_bytes = static_cast<size_t>(round_up(rows_b * ldb_d * es, 256));
    const size_t c_bytes = static_cast<size_t>(round_up(M * ldc_d * 4, 256));
    const size_t staged = a_bytes + b_bytes + c_bytes;

    const HostBlocks hb = plan_host_blocks(h, layout_b, M, N, K, dtype);
    const auto block_m = [&](int i) { return i == hb.pm - 1 ? M - i * hb.rows : hb.rows; };
    const auto block_n = [&](int j) { return j == hb.pn - 1 ? N - j * hb.cols : hb.cols; };
    // The staged buffers are 256-byte aligned with 16-byte-multiple rows and
    // block offsets, so no launch needs a re-pack; only split-K partial tiles
    // need room, as much as the largest of the launches' shapes.
    size_t extra = 0;
    for (int64_t mi : {block_m(0), block_m(hb.pm - 1)})
        for (int64_t nj : {block_n(0), block_n(hb.pn - 1), N})
            extra = std::max(extra, plan_pack(h, layout_b, mi, nj, K, nullptr, lda_d, nullptr, ldb_d, dtype).total());
    rc = ensure_workspace(h, staged + extra, stream);
    if (rc) return rc;
    uint8_t *ws = static_cast<uint8_t *>(h->ws);
    uint8_t *A_d = ws, *B_d = ws + a_bytes;
    float *C_d = reinterpret_cast<float *>(ws + a_bytes + b_bytes);
    const uint8_t *A_h = static_cast<const uint8_t *>(A_host);
    const uint8_t *B_h = static_cast<const uint8_t *>(B_host);

    // Column panel j of B: columns j*cols.. of a row-major K x N matrix, or
    // rows j*cols.. of the column-major (N x K) storage.
    const auto b_offset_d = [&](int j) { return b_row ? j * hb.cols * es : j * hb.cols * ldb_d * es; };
    const auto copy_b = [&](int j) {
        const int64_t nj = block_n(j);
        if (b_row)
            return cudaMemcpy2DAsync(B_d + b_offset_d(j), ldb_d * es, B_h + j * hb.cols * es, ldb * es, nj * es, K,
                                     cudaMemcpyHostToDevice, h->copy_in);
        return cudaMemcpy2DAsync(B_d + b_offset_d(j), ldb_d * es, B_h + j * hb.cols * ldb * es, ldb * es, K * es,
                                 nj, cudaMemcpyHostToDevice, h->copy_in);
    };
    const auto copy_a = [&](int i) {
        return cudaMemcpy2DAsync(A_d + i * hb.rows * lda_d * es, lda_d * es, A_h + i * hb.rows * lda * es, lda * es,
                                 K * es, block_m(i), cudaMemcpyHostToDevice, h->copy_in);
    };

    cudaError_t e = cudaEventRecord(h->ev_start, stream);  // after earlier work on the stream
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_in, h->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->copy_out, h->ev_start, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "host-copy pipeline set-up");
    // Copies in: B_0, A_0 .. A_{pm-1}, B_1 .. B_{pn-1}.  Launches: the blocks
    // of the first row panels column panel by column panel, each waiting only
    // for its own two panels, then the last row panel across all columns.
    std::string path;
    int block = 0;
    const auto launch = [&](int64_t m0, int64_t n0, int64_t mi, int64_t nj) {
        uint8_t *A_p = A_d + m0 * lda_d * es;
        uint8_t *B_p = B_d + (b_row ? n0 * es : n0 * ldb_d * es);
        float *C_p = C_d + m0 * ldc_d + n0;
        const PackPlan pp = plan_pack(h, layout_b, mi, nj, K, A_p, lda_d, B_p, ldb_d, dtype);
        int r = run_device(h, layout_b, mi, nj, K, A_p, lda_d, B_p, ldb_d, C_p, ldc_d, dtype, stream, pp, staged);
        if (r) return r;
        if (block == 0) path = h->last_path;
        cudaError_t err = cudaEventRecord(h->ev_c[block], stream);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(h->copy_out, h->ev_c[block], 0);
        if (err == cudaSuccess)
            err = cudaMemcpy2DAsync(C_host + m0 * ldc + n0, ldc * 4, C_p, ldc_d * 4, nj * 4, mi,
                                    cudaMemcpyDeviceToHost, h->copy_out);
        ++block;
        return err == cudaSuccess ? GEMM_OK : cuda_fail(h, err, "copy of C to the host");
    };
    const auto wait_copy = [&](cudaError_t err, cudaEvent_t ev, const char *what) {
        if (err == cudaSuccess) err = cudaEventRecord(ev, h->copy_in);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, ev, 0);
        return err == cudaSuccess ? GEMM_OK : cuda_fail(h, err, what);
    };
    const int blocked_panels = hb.pm > 1 ? hb.pm - 1 : 1;
    for (int j = 0; j < hb.pn; ++j) {
        if (K > 0 && (rc = wait_copy(copy_b(j), h->ev_b[j], "copy of B to the device"))) return rc;
        for (int i = 0; i < blocked_panels; ++i) {
            if (K > 0 && j == 0 && (rc = wait_copy(copy_a(i), h->ev_a[i], "copy of A to the device"))) return rc;
            if ((rc = launch(i * hb.rows, j * hb.cols, block_m(i), block_n(j)))) return rc;
        }
        if (K > 0 && j == 0 && hb.pm > 1) {  // A's last panel, before the rest of B
            e = copy_a(hb.pm - 1);
            if (e == cudaSuccess) e = cudaEventRecord(h->ev_a[hb.pm - 1], h->copy_in);
            if (e != cudaSuccess) return cuda_fail(h, e, "copy of A to the device");
        }
    }
    if (hb.pm > 1) {
        if (K > 0 && (e = cudaStreamWaitEvent(stream, h->ev_a[hb.pm - 1], 0)) != cudaSuccess)
            return cuda_fail(h, e, "copy of A to the device");
        if ((rc = launch((hb.pm - 1) * hb.rows, 0, block_m(hb.pm - 1), N))) return rc;
    }
    e = cudaEventRecord(h->ev_done, h->copy_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->ev_done, 0);  // the call ends on `stream`
    if (e != cudaSuccess) return cuda_fail(h, e, "host-copy pipeline completion");
    if ((rc = note_workspace_use(h, stream))) return rc;
    h->last_path = "host+" + path;
    if (block > 1) h->last_path += "+blocks" + std::to_string(hb.pm) + "x" + std::to_string(hb.pn);  // launches: (pm-1)*pn+1
    return GEMM_OK;
}

int gemm_sync_status(gemm_handle_t h, cudaStream_t stream)
{
    if (!h) return GEMM_ERR_INVALID;
    DeviceGuard guard(h->device);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
    int st = 0;
    e = cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(h, e, "read of the status word");
    if (st != 0) {
        cudaMemset(h->d_status, 0, sizeof(int));
        char msg[128];
        std::snprintf(msg, sizeof msg, "an in-kernel wait expired (code 0x%x); C is incomplete", st);
        return fail(h, GEMM_ERR_TIMEOUT, msg);
    }
    return GEMM_OK;
}

int gemm_set_option(gemm_handle_t h, int option, int64_t value)
{
    if (!h) return GEMM_ERR_INVALID;
    switch (option) {
    case GEMM_OPT_FORCE_REPACK:
        if (value != 0 && value != 1) break;
        h->force_repack = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_WAIT_TIMEOUT_NS:
        if (value < 1000000 || value > int64_t{60} * 1000000000) break;
        h->timeout_ns = static_cast<uint64_t>(value);
        return GEMM_OK;
    case GEMM_OPT_SIMT_GROUP_M:
        if (value < 0 || value > 1024) break;
        h->simt_group_m = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_TC_GROUP_M:
        if (value < 0 || value > 1024) break;
        h->tc_group_m = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_MAX_CTAS:
        if (value < 0 || value > 4 * int64_t{h->sm_count}) break;
        h->max_ctas = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_SIMT_CONFIG:
        if (value < 0 || value > dg::simt_num_configs()) break;
        if (value > 0 && !dg::simt_config_usable(static_cast<int>(value) - 1)) break;
        h->simt_config = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_WORKSPACE_LIMIT:
        if (value < 0) break;
        h->ws_limit = static_cast<size_t>(value);
        return GEMM_OK;
    case GEMM_OPT_ELEMENTWISE:
        if (value != 0 && value != 1) break;
        h->elementwise = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_DEBUG_DROP_LOAD:
        if (value != 0 && value != 1) break;
        h->debug_drop = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_TC_TMA_STORE:
        if (value != 0 && value != 1) break;
        h->tc_tma_store = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_TC_CLUSTER:
        if (value != 1 && value != 3) break;
        h->tc_cluster = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_TC_STAGE_SLICES:
        if (value < 0 || value > 2) break;
        h->tc_slices = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_SPLIT_K:
        if (value < 0 || value > 64) break;
        h->split_k = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_STREAM_K:
        if (value < 0 || value > 2) break;
        h->stream_k = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_SIMT_SMALL:
        if (value < 0 || value > 2) break;
        h->simt_small = static_cast<int>(value);
        return GEMM_OK;
    default:
        return fail(h, GEMM_ERR_INVALID, "unknown option");
    }
    return fail(h, GEMM_ERR_INVALID, "option value out of range");
}

const char *gemm_last_error_string(gemm_handle_t h) { return h ? h->last_error.c_str() : ""; }

const char *gemm_last_path(gemm_handle_t h) { return h ? h->last_path.c_str() : ""; }

int64_t gemm_launch_count(gemm_handle_t h) { return h ? h->launches : 0; }

}  // extern "C"
