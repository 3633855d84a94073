// Peak-rate microbenchmarks of the two arithmetic units the GEMM kernels are
// bound by ("GEMM 性能优化", Roofline 模型: the compute roof is the rate of
// the unit the kernel runs on; "PMPP Chapter 06: Performance
// considerations", the compute-bound side of the roofline):
//
//  * FP32 fused multiply-adds on the CUDA cores, scalar (fma.rn.f32) or packed
//    in pairs (fma.rn.f32x2), as the SIMT GEMM issues them.  Every thread runs
//    independent chains x <- x * a + b that stay near 1 (no overflow, no
//    subnormals); 32 warps per SM hide the FMA latency.  Each chain starts
//    from a value that depends on the thread, so the compiler can neither
//    merge chains nor evaluate one at compile time: a chain started exactly
//    at the fixed point x = 1 (1 * 0.999 + 0.001 rounds to 1 in FP32) was
//    once folded away, and the FLOP count then overstated the work by 16/15.
//  * tcgen05 MMAs from shared memory into tensor memory, BF16 or TF32 inputs
//    with FP32 accumulation, M = 128, N = 256 (one CTA per SM), as the
//    tensor-core GEMM issues them but with operands that stay in shared
//    memory: no copies, so the rate is the tensor pipe's alone.
//
// The host times a launch with CUDA events; the FLOP count of a launch is
// returned by the launch call.
#include <cstdint>

#include "../../include/gemm.h"
#include "../../include/gemm_peaks.h"
#include "gemm_internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int kFmaThreads = 256;
constexpr int kFmaBlocksPerSm = 4;  // 32 warps per SM
constexpr int kFmaChains = 8;       // independent accumulator pairs per thread
constexpr int kFmaUnroll = 16;

__global__ void __launch_bounds__(kFmaThreads) fma_peak_kernel(int packed, long long iters, float *sink)
{
    float2 acc[kFmaChains];
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c)
        acc[c] = make_float2(0.5f + 0.03125f * c + 0.0009765625f * (threadIdx.x & 31),
                             0.25f + 0.03125f * c + 0.0009765625f * (threadIdx.x & 31));
    const float2 a = make_float2(0.999f, 0.999f), b = make_float2(0.001f, 0.001f);
    if (packed) {
        for (long long i = 0; i < iters; i += kFmaUnroll)
#pragma unroll
            for (int u = 0; u < kFmaUnroll; ++u)
#pragma unroll
                for (int c = 0; c < kFmaChains; ++c) acc[c] = __ffma2_rn(acc[c], a, b);
    } else {
        for (long long i = 0; i < iters; i += kFmaUnroll)
#pragma unroll
            for (int u = 0; u < kFmaUnroll; ++u)
#pragma unroll
                for (int c = 0; c < kFmaChains; ++c) {
                    acc[c].x = fmaf(acc[c].x, a.x, b.x);
                    acc[c].y = fmaf(acc[c].y, a.y, b.y);
                }
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) s += acc[c].x + acc[c].y;
    if (s == -1.0f) sink[0] = s;  // never true; keeps the chains live
    if (blockIdx.x == 0 && threadIdx.x == 0) sink[1] = s;
}

constexpr int kMmaThreads = 128;
constexpr int kMmaA = 128 * 128;  // 128 rows x 128 bytes of K
constexpr int kMmaB = 256 * 128;  // 256 rows x 128 bytes of K
constexpr int kMmaSmem = 1024 + kMmaA + kMmaB + 64;
constexpr uint32_t kMmaCols = 256;

// DT: 0 = BF16, 1 = TF32.  Both operands K-major with the 128-byte swizzle,
// the layout the GEMM's TMA copies produce.
template <int DT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    mma_peak_kernel(long long iters, int *status, unsigned long long timeout_ns)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int UMMA_K = 32 / ES;        // K per instruction
    constexpr int K_STEPS = 128 / 32;      // instructions per 128-byte K slice
    constexpr uint32_t FMT = DT == 0 ? 1u : 2u;
    constexpr uint32_t IDESC = (1u << 4) | (FMT << 7) | (FMT << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
    (void)UMMA_K;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
    uint8_t *smem = smem_raw + pad;
    const uint32_t a_base = raw_addr + pad;
    const uint32_t b_base = a_base + kMmaA;
    const uint32_t bar = b_base + kMmaB;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + kMmaA + kMmaB + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMmaA + kMmaB + 16);

    // Operands: small values of both signs (the tensor pipe's power, and so
    // its clock, depends on the data).
    uint32_t *words = reinterpret_cast<uint32_t *>(smem);
    for (int i = threadIdx.x; i < (kMmaA + kMmaB) / 4; i += kMmaThreads) {
        const uint32_t h = (static_cast<uint32_t>(i) * 2654435761u) ^ (blockIdx.x * 40503u);
        if (DT == 0) {
            // two BF16 values in [-1, 1): sign, exponent 126..127, 7 mantissa bits
            const uint32_t lo = ((h & 1u) << 15) | ((126u + ((h >> 1) & 1u)) << 7) | ((h >> 2) & 0x7Fu);
            const uint32_t hi = (((h >> 9) & 1u) << 15) | ((126u + ((h >> 10) & 1u)) << 7) | ((h >> 11) & 0x7Fu);
            words[i] = lo | (hi << 16);
        } else {
            words[i] = ((h & 1u) << 31) | ((126u + ((h >> 1) & 1u)) << 23) | ((h >> 2) & 0x7FFFFFu);
        }
    }
    fence_proxy_async_shared();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(smem_addr(const_cast<uint32_t *>(tmem_slot)), kMmaCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t d_tmem = *tmem_slot;

    if (threadIdx.x == 0) {
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < K_STEPS; ++kk) {
                const uint64_t adesc = smem_desc(a_base + kk * 32, 16, 1024, kLayoutSw128);
                const uint64_t bdesc = smem_desc(b_base + kk * 32, 16, 1024, kLayoutSw128);
                const uint32_t accumulate = (it > 0 || kk > 0) ? 1u : 0u;
                if (DT == 0)
                    tc_mma_f16(d_tmem, adesc, bdesc, IDESC, accumulate);
                else
                    tc_mma_tf32(d_tmem, adesc, bdesc, IDESC, accumulate);
            }
        }
        tc_commit(bar);
        if (!mbar_wait(bar, 0, abort_flag, status, kWaitDrain, timeout_ns)) {
            // Leave nothing in flight before tensor memory is freed: wait
            // once more, bounded, without a further report.
            int dummy = 0;
            mbar_wait(bar, 0, &dummy, nullptr, kWaitDrain, timeout_ns);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after_sync();
        tmem_dealloc(d_tmem, kMmaCols);
    }
}

int sm_count_of_current_device(int *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_DEVICE;
    if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return GEMM_ERR_DEVICE;
    return GEMM_OK;
}

}  // namespace
}  // namespace dg

extern "C" {

int gemm_peak_fma_run(int packed, int64_t iters, float *sink, cudaStream_t stream, double *flops)
{
    if ((packed != 0 && packed != 1) || iters <= 0 || iters % dg::kFmaUnroll != 0 || !sink)
        return GEMM_ERR_INVALID;
    int sms = 0;
    const int rc = dg::sm_count_of_current_device(&sms);
    if (rc) return rc;
    const int grid = sms * dg::kFmaBlocksPerSm;
    dg::fma_peak_kernel<<<grid, dg::kFmaThreads, 0, stream>>>(packed, iters, sink);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    if (flops) *flops = 4.0 * dg::kFmaChains * static_cast<double>(iters) * grid * dg::kFmaThreads;
    return GEMM_OK;
}

int gemm_peak_mma_run(int dtype, int64_t iters, int *status, uint64_t timeout_ns, cudaStream_t stream,
                      double *flops)
{
    if ((dtype != GEMM_BF16 && dtype != GEMM_TF32) || iters <= 0) return GEMM_ERR_INVALID;
    int sms = 0;
    int rc = dg::sm_count_of_current_device(&sms);
    if (rc) return rc;
    const uint64_t limit = timeout_ns ? timeout_ns : 4000000000ull;
    cudaError_t e;
    if (dtype == GEMM_BF16) {
        e = cudaFuncSetAttribute(dg::mma_peak_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, dg::kMmaSmem);
        if (e == cudaSuccess)
            dg::mma_peak_kernel<0><<<sms, dg::kMmaThreads, dg::kMmaSmem, stream>>>(iters, status, limit);
    } else {
        e = cudaFuncSetAttribute(dg::mma_peak_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, dg::kMmaSmem);
        if (e == cudaSuccess)
            dg::mma_peak_kernel<1><<<sms, dg::kMmaThreads, dg::kMmaSmem, stream>>>(iters, status, limit);
    }
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    // Each iteration is one 128-byte K slice: 128 x 256 x (128 / element size) multiply-adds.
    const int es = dtype == GEMM_BF16 ? 2 : 4;
    if (flops) *flops = 2.0 * 128 * 256 * (128 / es) * static_cast<double>(iters) * sms;
    return GEMM_OK;
}

}  // extern "C"
