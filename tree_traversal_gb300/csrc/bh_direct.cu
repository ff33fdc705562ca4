// bh_direct.cu -- direct summation of the same softened force law over every
// pair, the comparison solver the pages time the tree against (orrery:
// docs/performance/sycl_tree.md, "Against the two solvers it has to beat":
// the GPU direct kernel of Phase 9, crossover with the tree near 9000
// particles on Xe2).
//
// a_i = sum over j != i, in caller order j = 0, 1, ..., of the term
// r2 = d2 + eps^2, y = rsqrt_newton(r2), f = (m_j y)(y y), a_i += f (x_j - x_i)
// -- the tree walk's particle term with its Newton inverse root: a fixed
// sequence of binary32 operations, so a CPU that repeats it reproduces every
// bit, and within a few ulp per term of the law evaluated plainly. Two
// targets per thread (i and i + kThreads within a block's 2 kThreads
// targets), both summed in packed float2 instructions (__fadd2_rn,
// __fmul2_rn, __ffma2_rn round each component exactly as the scalar forms),
// so one instruction issue does two pairs' arithmetic. Sources are staged
// through shared memory in tiles of kTile and read back as broadcasts. The
// self pair can only occur in the block's two diagonal tiles, so only those
// carry the j != i test, as a zero factor for the self pair (dx = +0 there,
// and fma(+0, +0, a) = a) chosen by a select, which keeps the pair in step.
#include <math.h>

#include "../../include/orrery_bh.h"
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 128;  // 256 targets per block: more blocks for small n
constexpr int kTile = kThreads;

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// rsqrt_newton of the walk, componentwise: Lomont's seed and three
// Newton-Raphson steps y (3/2 - (x/2) y^2); -x/2 is formed as fl(-x/2).
__device__ __forceinline__ float2 rsqrt_newton2(float2 x)
{
    const float2 nh = __fmul2_rn(splat2(-0.5f), x);
    float2 y = make_float2(__int_as_float(0x5f375a86 - (int)((unsigned)__float_as_int(x.x) >> 1)),
                           __int_as_float(0x5f375a86 - (int)((unsigned)__float_as_int(x.y) >> 1)));
#pragma unroll
    for (int it = 0; it < 3; ++it) y = __fmul2_rn(y, __ffma2_rn(nh, __fmul2_rn(y, y), splat2(1.5f)));
    return y;
}

// One source against both of the thread's targets (positions negated);
// kSelf: a target whose own index is the source adds a zero factor.
template <bool kSelf>
__device__ __forceinline__ void pair_term2(const float4 &p, float2 nx, float2 ny, float2 nz,
                                           float2 eps2, bool self0, bool self1, float2 &ax,
                                           float2 &ay, float2 &az)
{
    const float2 dx = __fadd2_rn(splat2(p.x), nx);
    const float2 dy = __fadd2_rn(splat2(p.y), ny);
    const float2 dz = __fadd2_rn(splat2(p.z), nz);
    const float2 d2 = __ffma2_rn(dz, dz, __ffma2_rn(dy, dy, __fmul2_rn(dx, dx)));
    const float2 y = rsqrt_newton2(__fadd2_rn(d2, eps2));
    float2 f = __fmul2_rn(__fmul2_rn(splat2(p.w), y), __fmul2_rn(y, y));
    if (kSelf) f = make_float2(self0 ? 0.0f : f.x, self1 ? 0.0f : f.y);
    ax = __ffma2_rn(f, dx, ax);
    ay = __ffma2_rn(f, dy, ay);
    az = __ffma2_rn(f, dz, az);
}

__device__ __forceinline__ float4 load_particle(const float *__restrict__ pos,
                                                const float *__restrict__ mass, int j)
{
    return make_float4(__ldg(pos + 3 * (int64_t)j), __ldg(pos + 3 * (int64_t)j + 1),
                       __ldg(pos + 3 * (int64_t)j + 2), __ldg(mass + j));
}

__global__ void __launch_bounds__(kThreads)
k_direct(const float *__restrict__ pos, const float *__restrict__ mass, int n, float eps2,
         float *__restrict__ acc, int *status)
{
    __shared__ float4 tile[kTile];
    const int i0 = blockIdx.x * 2 * kThreads + threadIdx.x, i1 = i0 + kThreads;
    const bool v0 = i0 < n, v1 = i1 < n;
    const float4 p0 = v0 ? load_particle(pos, mass, i0) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4 p1 = v1 ? load_particle(pos, mass, i1) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (!(isfinite(p0.x) && isfinite(p0.y) && isfinite(p0.z) && isfinite(p0.w) &&
          isfinite(p1.x) && isfinite(p1.y) && isfinite(p1.z) && isfinite(p1.w)))
        atomicOr(status, kStatusNonFinite);
    const float2 nx = make_float2(-p0.x, -p1.x), ny = make_float2(-p0.y, -p1.y),
                 nz = make_float2(-p0.z, -p1.z), e2 = splat2(eps2);
    float2 ax = splat2(0.0f), ay = splat2(0.0f), az = splat2(0.0f);
    const int diag = blockIdx.x * 2 * kThreads;  // the block's targets span two tiles from here
    for (int base = 0; base < n; base += kTile) {
        const int j = base + threadIdx.x;
        tile[threadIdx.x] = (j < n) ? load_particle(pos, mass, j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        __syncthreads();
        const int cnt = min(kTile, n - base);
        if (base != diag && base != diag + kTile) {
#pragma unroll 8
            for (int jj = 0; jj < cnt; ++jj)
                pair_term2<false>(tile[jj], nx, ny, nz, e2, false, false, ax, ay, az);
        } else {
            const int s0 = i0 - base, s1 = i1 - base;
#pragma unroll 4
            for (int jj = 0; jj < cnt; ++jj)
                pair_term2<true>(tile[jj], nx, ny, nz, e2, jj == s0, jj == s1, ax, ay, az);
        }
        __syncthreads();
    }
    if (v0) {
        acc[3 * (int64_t)i0 + 0] = ax.x;
        acc[3 * (int64_t)i0 + 1] = ay.x;
        acc[3 * (int64_t)i0 + 2] = az.x;
    }
    if (v1) {
        acc[3 * (int64_t)i1 + 0] = ax.y;
        acc[3 * (int64_t)i1 + 1] = ay.y;
        acc[3 * (int64_t)i1 + 2] = az.y;
    }
}

}  // namespace

void launch_direct(const float *pos, const float *mass, int64_t n, float eps, float *acc,
                   int *status, cudaStream_t st)
{
    const float eps2 = eps * eps;  // host binary32 product, round to nearest
    k_direct<<<ceil_div(n, 2 * (int64_t)kThreads), kThreads, 0, st>>>(pos, mass, (int)n, eps2, acc,
                                                                      status);
    g_launches += 1;
}

}  // namespace obh
