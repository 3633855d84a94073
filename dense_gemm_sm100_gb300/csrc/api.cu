// The C ABI of include/gemm.h: argument checks, dispatch to the kernels,
// TMA tensor-map encoding, the handle's workspace, and the host-buffer entry.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

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
    std::string last_error;
    std::string last_path;
    int64_t launches = 0;
    int force_repack = 0;
    uint64_t timeout_ns = 4000000000ull;
    int simt_group_m = 0;
    int tc_group_m = 0;
    int max_ctas = 0;
    int simt_config = 0;  // 0: chosen per shape; else configuration index + 1
    int split_k = 0;      // 0: chosen per shape; 1: never; n > 1: n K slices (FP32 path)
    int tc_cluster = 3;   // tensor-core mode: 1 one CTA per tile, 2 multicast pairs, 3 pair MMA
    int tc_tma_store = 1; // tensor-core epilogue writes C with TMA stores when C allows it
    int debug_drop = 0;   // test hook (GEMM_OPT_DEBUG_DROP_LOAD)
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
    if (dtype != GEMM_F32 && dtype != GEMM_TF32 && dtype != GEMM_BF16)
        return bad(GEMM_ERR_INVALID, "dtype must be GEMM_F32, GEMM_TF32 or GEMM_BF16");
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
    bool a = false, b = false;
    int64_t lda = 0, ldb = 0;
    size_t a_bytes = 0, b_bytes = 0;
    int simt_config = 0;
    dg::SplitK split;     // partials pointer is filled in by run_device
    size_t split_bytes = 0;
    size_t total() const { return a_bytes + b_bytes + split_bytes; }
};

PackPlan plan_pack(const gemm_ctx *h, int layout_b, int64_t M, int64_t N, int64_t K,
                   const void *A, int64_t lda, const void *B, int64_t ldb, int dtype)
{
    PackPlan pp;
    if (M == 0 || N == 0 || K == 0) return pp;
    const int es = elem_bytes(dtype);
    const int64_t align_elems = 16 / es;
    pp.a = h->force_repack || !tma_ready(A, lda, es);
    pp.b = h->force_repack || !tma_ready(B, ldb, es);
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
        pp.simt_config = h->simt_config > 0 ? h->simt_config - 1 : dg::simt_pick_config(M, N, h->sm_count);
        if (h->split_k == 0) {
            pp.split = dg::simt_pick_splits(pp.simt_config, layout_b, M, N, K, h->sm_count);
        } else if (h->split_k > 1) {
            const int64_t k_tiles = (K + dg::kSimtBK - 1) / dg::kSimtBK;
            const int64_t want = h->split_k < k_tiles ? h->split_k : k_tiles;
            const int64_t kt_per = (k_tiles + want - 1) / want;
            pp.split.splits = static_cast<int>((k_tiles + kt_per - 1) / kt_per);
            pp.split.k_per_split = static_cast<int>(kt_per * dg::kSimtBK);
        }
        if (pp.split.splits > 1)
            pp.split_bytes = static_cast<size_t>(round_up(int64_t{pp.split.splits} * M * N * 4, 256));
    }
    return pp;
}

int ensure_workspace(gemm_ctx *h, size_t need)
{
    if (need <= h->ws_bytes) return GEMM_OK;
    size_t grow = h->ws_bytes + h->ws_bytes / 2;
    size_t bytes = need > grow ? need : grow;
    bytes = (bytes + (size_t{2} << 20) - 1) & ~((size_t{2} << 20) - 1);
    // Earlier queued work may still read the old buffer.
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaDeviceSynchronize before workspace growth");
    if (h->ws) cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_bytes = 0;
    e = cudaMalloc(&h->ws, bytes);
    if (e != cudaSuccess) {
        h->ws = nullptr;
        cudaGetLastError();
        return fail(h, GEMM_ERR_NOMEM, std::string("workspace cudaMalloc: ") + cudaGetErrorString(e));
    }
    h->ws_bytes = bytes;
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
    if (pp.a) {
        cudaError_t e = dg::launch_repack(A, lda, ws, pp.lda, M, K, es, h->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "repack A launch");
        ++h->launches;
        A = ws;
        lda = pp.lda;
        path += "+repackA";
    }
    if (pp.b) {
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
    if (dtype == GEMM_F32) {
        const int cfg = pp.simt_config;
        const dg::SimtTile t = dg::simt_tile(cfg, layout_b);
        rc = encode_2d(h, &tmA, 4, A, K, M, lda, dg::kSimtBK, t.bm);
        if (rc) return rc;
        if (layout_b == GEMM_B_ROW_MAJOR)
            rc = encode_2d(h, &tmB, 4, B, N, K, ldb, 32, dg::kSimtBK);
        else
            rc = encode_2d(h, &tmB, 4, B, K, N, ldb, dg::kSimtBK, t.bn);
        if (rc) return rc;
        dg::SplitK sk = pp.split;
        if (sk.splits > 1) sk.partials = reinterpret_cast<float *>(ws + pp.a_bytes + pp.b_bytes);
        const int64_t units = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn) * sk.splits;
        const int64_t cap = h->max_ctas > 0 ? h->max_ctas : int64_t{h->sm_count} * t.ctas_per_sm;
        lc.grid = static_cast<int>(units < cap ? units : cap);
        lc.group_m = h->simt_group_m;
        cudaError_t e = dg::launch_simt_f32(cfg, tmA, tmB, layout_b, static_cast<int>(M), static_cast<int>(N),
                                            static_cast<int>(K), C, ldc, c_vec4, lc, sk);
        if (e != cudaSuccess) return cuda_fail(h, e, "FP32 SIMT kernel launch");
        path = std::string("simt_f32_") + t.name + "_" + lay + path;
        if (sk.splits > 1) {
            ++h->launches;
            e = dg::launch_splitk_reduce(sk.partials, sk.splits, C, ldc, M, N, h->sm_count, stream);
            if (e != cudaSuccess) return cuda_fail(h, e, "split-K reduction launch");
            path += "+splitk" + std::to_string(sk.splits);
        }
    } else {
        const int bk = dg::tc_bk(es);
        rc = encode_2d(h, &tmA, es, A, K, M, lda, bk, dg::kTcBM);
        if (rc) return rc;
        if (layout_b == GEMM_B_ROW_MAJOR)
            // MN-major B; 32-bit elements need 32-byte swizzle atoms there.
            rc = encode_2d(h, &tmB, es, B, N, K, ldb, 128 / es, bk,
                           es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B);
        else
            rc = encode_2d(h, &tmB, es, B, K, N, ldb, bk, dg::kTcBoxBCol);
        if (rc) return rc;
        const int cluster = h->tc_cluster >= 2 && M > dg::kTcBM ? h->tc_cluster : 1;
        int grid = dg::tc_grid(M, N, h->max_ctas > 0 ? h->max_ctas : h->sm_count, cluster);
        lc.grid = grid;
        lc.group_m = h->tc_group_m;
        alignas(64) CUtensorMap tmC;
        const bool c_tma = c_vec4 && h->tc_tma_store;
        if (c_tma) {
            rc = encode_2d(h, &tmC, 4, C, N, M, ldc, dg::kTcBoxC, dg::kTcBoxC);
            if (rc) return rc;
        }
        cudaError_t e = dg::launch_tc(dtype, layout_b, tmA, tmB, c_tma ? &tmC : nullptr, static_cast<int>(M),
                                      static_cast<int>(N), static_cast<int>(K), C, ldc, c_vec4, lc, cluster);
        if (e != cudaSuccess) return cuda_fail(h, e, "tensor-core kernel launch");
        path = std::string(dtype == GEMM_BF16 ? "tc_bf16" : "tc_tf32") +
               (cluster == 3 ? "_pair256x256_" : "_128x256_") + lay + (cluster == 2 ? "_cluster2" : "") + path;
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
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (h->d_status) cudaFree(h->d_status);
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
        if (h->ws) cudaFree(h->ws);
        if (h->d_status) cudaFree(h->d_status);
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
        rc = ensure_workspace(h, pp.total());
        if (rc) return rc;
    }
    return run_device(h, layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream, pp, 0);
}

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
    const int es = elem_bytes(dtype);
    const int64_t al = 16 / es;
    const int64_t rows_b = layout_b == GEMM_B_ROW_MAJOR ? K : N;
    const int64_t cols_b = layout_b == GEMM_B_ROW_MAJOR ? N : K;
    const int64_t lda_d = K ? round_up(K, al) : 0;
    const int64_t ldb_d = K ? round_up(cols_b, al) : 0;
    const int64_t ldc_d = round_up(N, 4);
    const size_t a_bytes = static_cast<size_t>(round_up(M * lda_d * es, 256));
    const size_t b_bytes = static_cast<size_t>(round_up(rows_b * ldb_d * es, 256));
    const size_t c_bytes = static_cast<size_t>(round_up(M * ldc_d * 4, 256));
    const size_t staged = a_bytes + b_bytes + c_bytes;
    // Pointers are only needed for the alignment test of the pack plan; the
    // staged buffers below are 256-byte aligned with 16-byte-multiple rows.
    rc = ensure_workspace(h, staged);
    if (rc) return rc;
    uint8_t *ws = static_cast<uint8_t *>(h->ws);
    void *A_d = ws, *B_d = ws + a_bytes;
    float *C_d = reinterpret_cast<float *>(ws + a_bytes + b_bytes);
    const PackPlan pp = plan_pack(h, layout_b, M, N, K, A_d, lda_d, B_d, ldb_d, dtype);
    if (pp.total()) {
        rc = ensure_workspace(h, staged + pp.total());  // may move the buffer: recompute below
        if (rc) return rc;
        ws = static_cast<uint8_t *>(h->ws);
        A_d = ws;
        B_d = ws + a_bytes;
        C_d = reinterpret_cast<float *>(ws + a_bytes + b_bytes);
    }
    cudaError_t e;
    if (K > 0) {
        e = cudaMemcpy2DAsync(A_d, lda_d * es, A_host, lda * es, K * es, M, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "copy of A to the device");
        e = cudaMemcpy2DAsync(B_d, ldb_d * es, B_host, ldb * es, cols_b * es, rows_b,
                              cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "copy of B to the device");
    }
    rc = run_device(h, layout_b, M, N, K, A_d, lda_d, B_d, ldb_d, C_d, ldc_d, dtype, stream, pp, staged);
    if (rc) return rc;
    e = cudaMemcpy2DAsync(C_host, ldc * 4, C_d, ldc_d * 4, N * 4, M, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "copy of C to the host");
    h->last_path = "host+" + h->last_path;
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
        h->simt_config = static_cast<int>(value);
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
        if (value < 1 || value > 3) break;
        h->tc_cluster = static_cast<int>(value);
        return GEMM_OK;
    case GEMM_OPT_SPLIT_K:
        if (value < 0 || value > 64) break;
        h->split_k = static_cast<int>(value);
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
