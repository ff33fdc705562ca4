// bh_peak.cu -- the measured FP32 fused multiply-add rate of the current GPU.
//
// The walk is bound by plain FP32 arithmetic and instruction issue, not by a
// dense contraction, so its roofline denominator is the FP32 pipe rather
// than the tensor cores. The nominal figure is SMs x 128 lanes x 2 flops x
// clock; this probe measures what the pipes deliver to long, independent
// FMA chains: scalar FFMA, and the packed FFMA2 form (two FMAs per lane per
// instruction) the walk's arithmetic uses. Each thread runs kChains
// independent chains, enough to cover the pipe latency with a full SM of
// warps; the chains converge (|a| < 1), so no value overflows. Every block
// also reads its SM's cycle counter and the global nanosecond timer at its
// start and end, so the clock the pipes ran at during the probe comes out
// beside the rate.
#include <algorithm>
#include <mutex>

#include "../../include/orrery_bh.h"
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSM = 8;    // 2048 threads per SM
constexpr int kChains = 8;
constexpr int kIters = 512;
constexpr int kMaxBlocks = 4096;

__device__ float g_fma_sink[kMaxBlocks];
__device__ double g_fma_mhz[kMaxBlocks];

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

template <bool kPacked>
__global__ void __launch_bounds__(kThreads) k_fma_rate(float seed)
{
    const long long c0 = clock64();
    const unsigned long long t0 = global_ns();
    const float a = 0.999f - 1e-6f * (float)(threadIdx.x & 31);
    float s = 0.0f;
    if (kPacked) {
        const float2 a2 = make_float2(a, a), b2 = make_float2(seed, -seed);
        float2 c[kChains];
#pragma unroll
        for (int i = 0; i < kChains; ++i) c[i] = make_float2(1e-3f * threadIdx.x + i, 0.5f * i);
#pragma unroll 16  // loop control would otherwise take 2 of every 10 issue slots
        for (int it = 0; it < kIters; ++it) {
#pragma unroll
            for (int i = 0; i < kChains; ++i) c[i] = __ffma2_rn(a2, c[i], b2);
        }
#pragma unroll
        for (int i = 0; i < kChains; ++i) s += c[i].x + c[i].y;
    } else {
        float c[kChains];
#pragma unroll
        for (int i = 0; i < kChains; ++i) c[i] = 1e-3f * threadIdx.x + i;
#pragma unroll 16  // loop control would otherwise take 2 of every 10 issue slots
        for (int it = 0; it < kIters; ++it) {
#pragma unroll
            for (int i = 0; i < kChains; ++i) c[i] = __fmaf_rn(a, c[i], seed);
        }
#pragma unroll
        for (int i = 0; i < kChains; ++i) s += c[i];
    }
    g_fma_sink[blockIdx.x % kMaxBlocks] = s;  // keeps the chains live
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long c1 = clock64();
        const unsigned long long t1 = global_ns();
        g_fma_mhz[blockIdx.x % kMaxBlocks] = t1 > t0 ? 1e3 * (double)(c1 - c0) / (double)(t1 - t0) : 0.0;
    }
}

// Times one launch of the probe (after one untimed launch); TFLOP/s or < 0.
// mhz: the median over blocks of their SM cycles per microsecond.
template <bool kPacked>
double time_rate(int blocks, cudaStream_t st, double *mhz)
{
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return -1.0;
    }
    k_fma_rate<kPacked><<<blocks, kThreads, 0, st>>>(0.25f);
    cudaEventRecord(e0, st);
    k_fma_rate<kPacked><<<blocks, kThreads, 0, st>>>(0.25f);
    cudaEventRecord(e1, st);
    g_launches += 2;
    float ms = 0.0f;
    const bool ok = cudaEventSynchronize(e1) == cudaSuccess && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (!ok || ms <= 0.0f) return -1.0;
    static double block_mhz[kMaxBlocks];
    if (cudaMemcpyFromSymbol(block_mhz, g_fma_mhz, sizeof(double) * blocks) != cudaSuccess)
        return -1.0;
    std::nth_element(block_mhz, block_mhz + blocks / 2, block_mhz + blocks);
    *mhz = block_mhz[blocks / 2];
    const double fmas = (double)blocks * kThreads * kIters * kChains * (kPacked ? 2.0 : 1.0);
    return 2.0 * fmas / (ms * 1e-3) / 1e12;
}

}  // namespace
}  // namespace obh

extern "C" int orrery_fp32_fma_rate(double *tflops_scalar, double *tflops_packed, double *sm_mhz,
                                    void *stream)
{
    using namespace obh;
    if (!tflops_scalar || !tflops_packed) return ORRERY_EINVAL;
    static std::mutex mu;  // one probe at a time: the cycle counters are shared
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
        cudaGetLastError();
        return ORRERY_ECUDA;
    }
    const int blocks = sms * kBlocksPerSM < kMaxBlocks ? sms * kBlocksPerSM : kMaxBlocks;
    cudaStream_t st = (cudaStream_t)stream;
    double mhz = 0.0, mhz_packed = 0.0;
    *tflops_scalar = time_rate<false>(blocks, st, &mhz);
    *tflops_packed = time_rate<true>(blocks, st, &mhz_packed);
    if (sm_mhz) *sm_mhz = mhz;
    if (*tflops_scalar <= 0.0 || *tflops_packed <= 0.0 || cudaGetLastError() != cudaSuccess)
        return ORRERY_ECUDA;
    return ORRERY_OK;
}
