// bh_direct.cu -- direct summation of the same softened force law over every
// pair, the comparison solver the pages time the tree against (orrery:
// docs/performance/sycl_tree.md, "Against the two solvers it has to beat":
// the GPU direct kernel of Phase 9, crossover with the tree near 9000
// particles on Xe2).
//
// a_i = sum over j != i, in caller order j = 0, 1, ..., of the term
// r2 = d2 + eps^2, y = rsqrt_newton(r2), f = (m_j y)(y y), a_i += f (x_j - x_i)
// -- the tree walk's particle term, so a CPU restatement reproduces every
// bit. One thread per target; sources are staged through shared memory in
// tiles of kTile, read back as broadcasts. The self pair can only occur in a
// block's diagonal tile, so only that tile carries the j != i check.
#include <math.h>

#include "../../include/orrery_bh.h"
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = kThreads;

__device__ __forceinline__ float rsqrt_newton_d(float x)
{
    const float h = __fmul_rn(0.5f, x);
    float y = __int_as_float(0x5f375a86 - (int)((unsigned)__float_as_int(x) >> 1));
#pragma unroll
    for (int it = 0; it < 3; ++it) y = __fmul_rn(y, __fmaf_rn(-h, __fmul_rn(y, y), 1.5f));
    return y;
}

__device__ __forceinline__ void pair_term(const float4 &p, const float4 &xi, float eps2, float &ax,
                                          float &ay, float &az)
{
    const float dx = __fsub_rn(p.x, xi.x);
    const float dy = __fsub_rn(p.y, xi.y);
    const float dz = __fsub_rn(p.z, xi.z);
    const float d2 = __fmaf_rn(dz, dz, __fmaf_rn(dy, dy, __fmul_rn(dx, dx)));
    const float r2 = __fadd_rn(d2, eps2);
    const float y = rsqrt_newton_d(r2);
    const float f = __fmul_rn(__fmul_rn(p.w, y), __fmul_rn(y, y));
    ax = __fmaf_rn(f, dx, ax);
    ay = __fmaf_rn(f, dy, ay);
    az = __fmaf_rn(f, dz, az);
}

__global__ void __launch_bounds__(kThreads)
k_direct(const float *__restrict__ pos, const float *__restrict__ mass, int n, float eps2,
         float *__restrict__ acc, int *status)
{
    __shared__ float4 tile[kTile];
    const int i = blockIdx.x * kThreads + threadIdx.x;
    const bool valid = i < n;
    float4 xi = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (valid) {
        xi = make_float4(__ldg(pos + 3 * (int64_t)i), __ldg(pos + 3 * (int64_t)i + 1),
                         __ldg(pos + 3 * (int64_t)i + 2), __ldg(mass + i));
        if (!(isfinite(xi.x) && isfinite(xi.y) && isfinite(xi.z) && isfinite(xi.w)))
            atomicOr(status, kStatusNonFinite);
    }
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    const int diag = blockIdx.x * kThreads;
    for (int base = 0; base < n; base += kTile) {
        const int j = base + threadIdx.x;
        tile[threadIdx.x] = (j < n) ? make_float4(__ldg(pos + 3 * (int64_t)j),
                                                  __ldg(pos + 3 * (int64_t)j + 1),
                                                  __ldg(pos + 3 * (int64_t)j + 2), __ldg(mass + j))
                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        __syncthreads();
        const int cnt = min(kTile, n - base);
        if (base != diag) {
#pragma unroll 8
            for (int jj = 0; jj < cnt; ++jj) pair_term(tile[jj], xi, eps2, ax, ay, az);
        } else {
            const int self = i - base;
            for (int jj = 0; jj < cnt; ++jj)
                if (jj != self) pair_term(tile[jj], xi, eps2, ax, ay, az);
        }
        __syncthreads();
    }
    if (valid) {
        acc[3 * (int64_t)i + 0] = ax;
        acc[3 * (int64_t)i + 1] = ay;
        acc[3 * (int64_t)i + 2] = az;
    }
}

}  // namespace

void launch_direct(const float *pos, const float *mass, int64_t n, float eps, float *acc,
                   int *status, cudaStream_t st)
{
    const float eps2 = eps * eps;  // host binary32 product, round to nearest
    k_direct<<<ceil_div(n, kThreads), kThreads, 0, st>>>(pos, mass, (int)n, eps2, acc, status);
    g_launches += 1;
}

}  // namespace obh
