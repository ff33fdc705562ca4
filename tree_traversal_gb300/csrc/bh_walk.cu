// bh_walk.cu -- a7: the two stackless traversals of the depth-first octree.
//
// orrery: "sycl_tree_solver.hpp", TreeTraversal:
//   kIndependent -- one thread per target, each following its own node index;
//   kCoherent    -- one node index per warp, advanced by agreement.
// ADR-0029 ("Mask the accepted cells rather than descending together"),
// Decision: the group advances to the smallest node index any lane still
// wants; a lane that accepts a cell records the index its own walk would jump
// to (the escape index) and contributes nothing until the group reaches it.
// The group's visited sequence is therefore the union of its lanes' walks and
// every target is summed over exactly its own nodes, in the same order, so
// the two kernels below produce bit-identical sums and counters.
//
// Per target i at node k of level L (a visit is one acceptance test):
//   accept iff (side 2^-L)^2 < theta^2 |CoM_k - x_i|^2  -> cell term, escape
//   else if k is a leaf -> particle terms over its particles j != i, escape
//   else -> k + 1 (first child)
// Term: r2 = d2 + eps^2, y = the binary32 value nearest 1/sqrt(r2),
// f = (m y)(y y), a += f (x_src - x_i) by fused multiply-add. Every
// floating-point step is one correctly rounded binary32 operation (explicit
// _rn intrinsics), so decisions and sums do not depend on contraction choices.
//
// GB300 shape of the coherent kernel: the node k is warp-uniform, so its two
// 16-byte records are read once per warp step and broadcast. The walk record
// {escape, first, leaf count (0 = internal), squared side bits} carries
// everything a step decides on, so a step needs no table lookup and no leaf
// test beyond one compare. An opened leaf's particles are staged into shared
// memory once (one coalesced 16-byte load per lane) and read back as
// broadcasts by every lane that opened it. The loop is warp-uniform and
// bounded: k strictly increases, so a walk takes at most num_nodes steps; the
// loop stops there and raises a status bit rather than spin.
//
// The self term. When the target's own leaf is opened the oracle skips j = i.
// Summing it instead changes nothing, bit for bit, whenever its force factor
// is finite: dx = dy = dz = +0, so fma(f, +0, a) = a (a is never -0: it
// starts at +0 and round-to-nearest never produces -0 from a sum of unlike
// signs). The factor is finite iff eps > 0 and (m_max y)(y y) does not
// overflow for y = rsqrt(eps^2); the kernels test that once per block and
// drop the per-particle self comparison when it holds.
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

struct WalkArgs {
    const float4 *ps;     // sorted particles {x, y, z, m}
    const float4 *com;    // {CoM_x, CoM_y, CoM_z, M}
    const int4 *wnode;    // {escape, first, leaf count or 0, squared side bits}
    int n;
    float theta2;
    float eps2;
    DeviceParams *P;
    float *acc_s;
    uint32_t *cnt_s;
};

__device__ __forceinline__ void add_term(float dx, float dy, float dz, float d2, float m,
                                         float eps2, float &ax, float &ay, float &az)
{
    const float r2 = __fadd_rn(d2, eps2);
    const float y = __frsqrt_rn(r2);
    const float f = __fmul_rn(__fmul_rn(m, y), __fmul_rn(y, y));
    ax = __fmaf_rn(f, dx, ax);
    ay = __fmaf_rn(f, dy, ay);
    az = __fmaf_rn(f, dz, az);
}

__device__ __forceinline__ float dist2(float dx, float dy, float dz)
{
    return __fmaf_rn(dz, dz, __fmaf_rn(dy, dy, __fmul_rn(dx, dx)));
}

__device__ __forceinline__ void particle_term(const float4 &p, const float4 &xi, float eps2,
                                              float &ax, float &ay, float &az)
{
    const float dx = __fsub_rn(p.x, xi.x);
    const float dy = __fsub_rn(p.y, xi.y);
    const float dz = __fsub_rn(p.z, xi.z);
    add_term(dx, dy, dz, dist2(dx, dy, dz), p.w, eps2, ax, ay, az);
}

// Block prologue shared by both kernels: status, node count and whether the
// self term may be summed (see the file comment). Returns false to skip.
__device__ __forceinline__ bool prologue(const WalkArgs &a, int &num_nodes, bool &self_free)
{
    __shared__ int s_state[3];
    if (threadIdx.x == 0) {
        const DeviceParams *P = a.P;
        s_state[0] = P->status;
        s_state[1] = P->num_nodes;
        bool ok = a.eps2 > 0.0f;
        if (ok) {
            const float y = __frsqrt_rn(a.eps2);
            const float f = __fmul_rn(__fmul_rn(P->mmax, y), __fmul_rn(y, y));
            ok = isfinite(f);
        }
        s_state[2] = ok ? 1 : 0;
    }
    __syncthreads();
    num_nodes = s_state[1];
    self_free = s_state[2] != 0;
    return s_state[0] == 0;
}

template <bool kCount, bool kSelfFree>
__device__ __forceinline__ void coherent_walk(const WalkArgs &a, int num_nodes, float4 *stage)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kThreads + threadIdx.x;
    const bool valid = t < a.n;
    const float4 xi = valid ? __ldg(a.ps + t) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int next = valid ? 0 : num_nodes;
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    uint32_t pc = 0, pp = 0;
    int steps = 0;
    for (; steps <= num_nodes; ++steps) {
        const int k = __reduce_min_sync(0xffffffffu, next);
        if (k >= num_nodes) break;
        const float4 c = __ldg(a.com + k);
        const int4 w = __ldg(a.wnode + k);
        bool open = false;
        if (next == k) {
            const float dx = __fsub_rn(c.x, xi.x);
            const float dy = __fsub_rn(c.y, xi.y);
            const float dz = __fsub_rn(c.z, xi.z);
            const float d2 = dist2(dx, dy, dz);
            if (__int_as_float(w.w) < __fmul_rn(a.theta2, d2)) {
                add_term(dx, dy, dz, d2, c.w, a.eps2, ax, ay, az);
                if (kCount) ++pc;
                next = w.x;
            } else {
                open = w.z != 0;
                next = open ? w.x : k + 1;
            }
        }
        if (__any_sync(0xffffffffu, open)) {
            const int first = w.y, count = w.z;
            if (first < 0 || first > a.n - count) {  // warp-uniform consistency check
                if (lane == 0) atomicOr(&a.P->status, kStatusInternal);
                break;
            }
            if (kCount && open) pp += count - ((unsigned)(t - first) < (unsigned)count ? 1u : 0u);
            for (int base = 0; base < count; base += 32) {
                const int chunk = min(32, count - base);
                if (lane < chunk) stage[lane] = __ldg(a.ps + first + base + lane);
                __syncwarp();
                if (open) {
                    if (kSelfFree) {
#pragma unroll 4
                        for (int j = 0; j < chunk; ++j)
                            particle_term(stage[j], xi, a.eps2, ax, ay, az);
                    } else {
                        const int self = t - (first + base);
                        for (int j = 0; j < chunk; ++j)
                            if (j != self) particle_term(stage[j], xi, a.eps2, ax, ay, az);
                    }
                }
                __syncwarp();
            }
        }
    }
    if (steps > num_nodes && lane == 0) atomicOr(&a.P->status, kStatusWalkBound);
    if (valid) {
        a.acc_s[3 * (int64_t)t + 0] = ax;
        a.acc_s[3 * (int64_t)t + 1] = ay;
        a.acc_s[3 * (int64_t)t + 2] = az;
        if (kCount) {
            a.cnt_s[3 * (int64_t)t + 0] = pc;
            a.cnt_s[3 * (int64_t)t + 1] = pp;
            a.cnt_s[3 * (int64_t)t + 2] = (uint32_t)steps;  // every step visits the union
        }
    }
}

template <bool kCount>
__global__ void __launch_bounds__(kThreads) k_walk_coherent(WalkArgs a)
{
    __shared__ float4 s_leaf[kWarpsPerBlock][32];
    int num_nodes;
    bool self_free;
    if (!prologue(a, num_nodes, self_free)) return;  // block-uniform
    float4 *stage = s_leaf[threadIdx.x >> 5];
    if (self_free)
        coherent_walk<kCount, true>(a, num_nodes, stage);
    else
        coherent_walk<kCount, false>(a, num_nodes, stage);
}

template <bool kCount, bool kSelfFree>
__device__ __forceinline__ void independent_walk(const WalkArgs &a, int num_nodes)
{
    const int t = blockIdx.x * kThreads + threadIdx.x;
    if (t >= a.n) return;
    const float4 xi = __ldg(a.ps + t);
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    uint32_t pc = 0, pp = 0;
    int k = 0, steps = 0;
    for (; steps <= num_nodes && k < num_nodes; ++steps) {
        const float4 c = __ldg(a.com + k);
        const int4 w = __ldg(a.wnode + k);
        const float dx = __fsub_rn(c.x, xi.x);
        const float dy = __fsub_rn(c.y, xi.y);
        const float dz = __fsub_rn(c.z, xi.z);
        const float d2 = dist2(dx, dy, dz);
        if (__int_as_float(w.w) < __fmul_rn(a.theta2, d2)) {
            add_term(dx, dy, dz, d2, c.w, a.eps2, ax, ay, az);
            if (kCount) ++pc;
            k = w.x;
        } else if (w.z != 0) {
            const int first = w.y, count = w.z;
            if (first < 0 || first > a.n - count) {
                atomicOr(&a.P->status, kStatusInternal);
                break;
            }
            if (kCount) pp += count - ((unsigned)(t - first) < (unsigned)count ? 1u : 0u);
            for (int j = first; j < first + count; ++j)
                if (kSelfFree || j != t) particle_term(__ldg(a.ps + j), xi, a.eps2, ax, ay, az);
            k = w.x;
        } else {
            k = k + 1;
        }
    }
    if (k < num_nodes) atomicOr(&a.P->status, kStatusWalkBound);
    a.acc_s[3 * (int64_t)t + 0] = ax;
    a.acc_s[3 * (int64_t)t + 1] = ay;
    a.acc_s[3 * (int64_t)t + 2] = az;
    if (kCount) {
        a.cnt_s[3 * (int64_t)t + 0] = pc;
        a.cnt_s[3 * (int64_t)t + 1] = pp;
        a.cnt_s[3 * (int64_t)t + 2] = (uint32_t)steps;
    }
}

template <bool kCount>
__global__ void __launch_bounds__(kThreads) k_walk_independent(WalkArgs a)
{
    int num_nodes;
    bool self_free;
    if (!prologue(a, num_nodes, self_free)) return;
    if (self_free)
        independent_walk<kCount, true>(a, num_nodes);
    else
        independent_walk<kCount, false>(a, num_nodes);
}

}  // namespace

void launch_walk(int traversal, float theta, float eps, int32_t leaf_cap, bool count,
                 const Buffers &b, cudaStream_t st)
{
    (void)leaf_cap;  // leaf-ness is carried by the walk records
    WalkArgs a;
    a.ps = b.ps;
    a.com = b.com;
    a.wnode = b.wnode;
    a.n = (int)b.n;
    a.theta2 = theta * theta;  // host binary32 products, round to nearest
    a.eps2 = eps * eps;
    a.P = b.params;
    a.acc_s = b.acc_s;
    a.cnt_s = b.cnt_s;
    const unsigned grid = ceil_div(b.n, kThreads);
    if (traversal == 1) {
        if (count)
            k_walk_coherent<true><<<grid, kThreads, 0, st>>>(a);
        else
            k_walk_coherent<false><<<grid, kThreads, 0, st>>>(a);
    } else {
        if (count)
            k_walk_independent<true><<<grid, kThreads, 0, st>>>(a);
        else
            k_walk_independent<false><<<grid, kThreads, 0, st>>>(a);
    }
    g_launches += 1;
}

}  // namespace obh
