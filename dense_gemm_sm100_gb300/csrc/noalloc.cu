// gemm_run_noalloc: the GEMM without any device allocation.
//
// Some callers cannot call cudaMalloc: code running under a framework whose
// memory manager owns all device memory (a caching allocator that must see
// every allocation, or a process whose memory budget is reserved up front),
// and latency-critical threads that must not take cudaMalloc's implicit
// device synchronisation.  gemm_create/gemm_run allocate a status word and a
// growable workspace, so they are not usable there.  This entry point needs
// no handle: operands whose address or pitch is not a multiple of 16 bytes
// are re-packed into a fixed scratch array that lives in this file as a
// static __device__ array, reserved on every GPU that loads this module until
// the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/gemm.h"
#include "gemm_internal.h"

namespace {

// The scratch for re-packed A and B (GEMM_NOALLOC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

// Status word of these calls on this device: a kernel whose in-kernel wait
// expires writes its code here, as a handle's kernels write the handle's
// status word; gemm_noalloc_sync_status reads and clears it.  Zero at load.
static __device__ int g_noalloc_status;

// Process-wide settings of these calls (gemm_noalloc_set_option).
std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<int> g_debug_drop{0};

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool done = false;
    int rc = GEMM_OK;
    int sm_count = 0;
    void *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int *status = nullptr;    // device address of g_noalloc_status on this device
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;

// Once per device, with that device current: check the device, raise the
// kernels' shared-memory limits, find the tensor-map encoder and look up the
// device addresses of the scratch array and the status word.
int setup_device(int dev, DeviceSetup **out)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup &s = g_setup[dev];
    if (!s.done) {
        s.done = true;
        s.rc = GEMM_OK;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess || prop.major != 10 || prop.minor != 3) {
            cudaGetLastError();
            s.rc = GEMM_ERR_DEVICE;
        } else {
            s.sm_count = prop.multiProcessorCount;
            if (!g_encode_fn) {
                void *fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q) == cudaSuccess &&
                    q == cudaDriverEntryPointSuccess)
                    g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
            cudaError_t e = g_encode_fn ? cudaSuccess : cudaErrorNotSupported;
            if (e == cudaSuccess) e = dg::prepare_simt();
            if (e == cudaSuccess) e = dg::prepare_tc();
            if (e == cudaSuccess) e = cudaGetSymbolAddress(&s.scratch, g_noalloc_scratch);
            if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void **>(&s.status), g_noalloc_status);
            if (e != cudaSuccess) {
                cudaGetLastError();
                s.scratch = nullptr;
                s.status = nullptr;
                s.rc = GEMM_ERR_CUDA;
            }
        }
    }
    *out = &s;
    return s.rc;
}

int64_t up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int current_device_setup(DeviceSetup **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_DEVICE;
    }
    return setup_device(dev, out);
}

bool tma_ok(const void *p, int64_t ld, int es)
{
    return reinterpret_cast<uintptr_t>(p) % 16 == 0 && (ld * es) % 16 == 0;
}

bool encode(CUtensorMap *map, int es, const void *base, int64_t inner, int64_t outer, int64_t ld,
            int box_inner, int box_outer, CUtensorMapSwizzle swizzle)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode_fn(map, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       2, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int gemm_run_noalloc(int layout_b, int64_t M, int64_t N, int64_t K, const void *A,
                                int64_t lda, const void *B, int64_t ldb, float *C, int64_t ldc,
                                int dtype, cudaStream_t stream)
{
    int rc = gemm_validate(layout_b, M, N, K, A, lda, B, ldb, C, ldc, dtype);
    if (rc != GEMM_OK) return rc;
    if (dtype == GEMM_F32_3XTF32) return GEMM_ERR_INVALID;  // its split operands need a workspace
    DeviceSetup *s = nullptr;
    rc = current_device_setup(&s);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    if (K == 0) {
        return dg::launch_zero_fill(C, ldc, M, N, s->sm_count, stream) == cudaSuccess ? GEMM_OK
                                                                                      : GEMM_ERR_CUDA;
    }

    // Re-pack plan: which operands need a 16-byte pitch, and where they go.
    const int es = dtype == GEMM_BF16 ? 2 : 4;
    const int64_t al = 16 / es;
    const int64_t rows_b = layout_b == GEMM_B_ROW_MAJOR ? K : N;
    const int64_t cols_b = layout_b == GEMM_B_ROW_MAJOR ? N : K;
    const bool pack_a = !tma_ok(A, lda, es);
    const bool pack_b = !tma_ok(B, ldb, es);
    const int64_t lda_p = pack_a ? up(K, al) : lda;
    const int64_t ldb_p = pack_b ? up(cols_b, al) : ldb;
    const int64_t a_bytes = pack_a ? up(M * lda_p * es, 256) : 0;
    const int64_t b_bytes = pack_b ? up(rows_b * ldb_p * es, 256) : 0;
    if (a_bytes + b_bytes > static_cast<int64_t>(GEMM_NOALLOC_SCRATCH_BYTES))
        return GEMM_ERR_INVALID;  // re-packed operands would not fit the static scratch

    unsigned char *scratch = static_cast<unsigned char *>(s->scratch);
    if (pack_a) {
        if (dg::launch_repack(A, lda, scratch, lda_p, M, K, es, s->sm_count, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        A = scratch;
    }
    if (pack_b) {
        if (dg::launch_repack(B, ldb, scratch + a_bytes, ldb_p, rows_b, cols_b, es, s->sm_count,
                              stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        B = scratch + a_bytes;
    }

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    dg::LaunchCommon lc;
    lc.status = s->status;  // read by gemm_noalloc_sync_status
    lc.timeout_ns = g_timeout_ns.load();
    lc.group_m = 0;
    lc.stream = stream;
    lc.debug_drop = g_debug_drop.load();
    const bool c_vec4 = reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 4 == 0;
    cudaError_t e;
    if (dtype == GEMM_F32) {
        const int cfg = dg::simt_pick_config(M, N, K, layout_b, s->sm_count, 0);
        const dg::SimtTile t = dg::simt_tile(cfg, layout_b);
        bool ok = encode(&tmA, 4, A, K, M, lda_p, dg::kSimtBK, t.bm, CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && (layout_b == GEMM_B_ROW_MAJOR
                        ? encode(&tmB, 4, B, N, K, ldb_p, 32, dg::kSimtBK, CU_TENSOR_MAP_SWIZZLE_128B)
                        : encode(&tmB, 4, B, K, N, ldb_p, dg::kSimtBK, t.bn, CU_TENSOR_MAP_SWIZZLE_128B));
        if (!ok) return GEMM_ERR_CUDA;
        const int64_t tiles = ((M + t.bm - 1) / t.bm) * ((N + t.bn - 1) / t.bn);
        const int64_t cap = int64_t{s->sm_count} * t.ctas_per_sm;
        lc.grid = static_cast<int>(tiles < cap ? tiles : cap);
        e = dg::launch_simt_f32(cfg, tmA, tmB, layout_b, static_cast<int>(M), static_cast<int>(N),
                                static_cast<int>(K), C, ldc, c_vec4, lc);
    } else {
        const int bk = dg::tc_bk(es);
        bool ok = encode(&tmA, es, A, K, M, lda_p, bk, dg::kTcBM, CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && (layout_b == GEMM_B_ROW_MAJOR
                        ? encode(&tmB, es, B, N, K, ldb_p, 128 / es, bk,
                                 es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B)
                        : encode(&tmB, es, B, K, N, ldb_p, bk, dg::kTcBoxBCol, CU_TENSOR_MAP_SWIZZLE_128B));
        if (!ok) return GEMM_ERR_CUDA;
        lc.grid = dg::tc_grid(M, N, s->sm_count, 1);
        e = dg::launch_tc(dtype, layout_b, tmA, tmB, nullptr, static_cast<int>(M), static_cast<int>(N),
                          static_cast<int>(K), C, ldc, c_vec4, lc, 1, false);
    }
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

extern "C" int gemm_noalloc_sync_status(cudaStream_t stream)
{
    DeviceSetup *s = nullptr;
    int rc = current_device_setup(&s);
    if (rc != GEMM_OK) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    int st = 0;
    if (cudaMemcpy(&st, s->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (st == 0) return GEMM_OK;
    if (cudaMemset(s->status, 0, sizeof st) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_ERR_TIMEOUT;
}

extern "C" int gemm_noalloc_set_option(int option, int64_t value)
{
    switch (option) {
    case GEMM_OPT_WAIT_TIMEOUT_NS:
        if (value < 1000000 || value > int64_t{60} * 1000000000) return GEMM_ERR_INVALID;
        g_timeout_ns.store(static_cast<uint64_t>(value));
        return GEMM_OK;
    case GEMM_OPT_DEBUG_DROP_LOAD:
        if (value != 0 && value != 1) return GEMM_ERR_INVALID;
        g_debug_drop.store(static_cast<int>(value));
        return GEMM_OK;
    default:
        return GEMM_ERR_INVALID;
    }
}
