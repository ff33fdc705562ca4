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
// Term: r2 = d2 + eps^2, f = m / (r2 sqrt(r2)), a += f (x_src - x_i).
// Every floating-point step is one correctly rounded binary32 operation
// (explicit _rn intrinsics), so decisions and sums do not depend on the
// compiler's contraction choices.
//
// GB300 shape of the coherent kernel: the node k is warp-uniform, so its two
// 16-byte records (CoM/M and escape/first/count/level) are read once per warp
// step and broadcast; the per-level squared side comes from a shared table;
// an opened leaf's particles are staged into shared memory once (one
// coalesced 16-byte load per lane) and read back as broadcasts by every lane
// that opened it. The loop is warp-uniform: the step count is bounded by the
// node count because k strictly increases, and the kernel still carries an
// explicit iteration bound that raises a status bit instead of spinning.
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

__device__ __forceinline__ void add_term(float dx, float dy, float dz, float d2, float m,
                                         float eps2, float &ax, float &ay, float &az)
{
    const float r2 = __fadd_rn(d2, eps2);
    const float f = __fdiv_rn(m, __fmul_rn(r2, __fsqrt_rn(r2)));
    ax = __fmaf_rn(f, dx, ax);
    ay = __fmaf_rn(f, dy, ay);
    az = __fmaf_rn(f, dz, az);
}

__device__ __forceinline__ float dist2(float dx, float dy, float dz)
{
    return __fmaf_rn(dz, dz, __fmaf_rn(dy, dy, __fmul_rn(dx, dx)));
}

template <bool kCount>
__global__ void __launch_bounds__(kThreads)
k_walk_coherent(const float4 *__restrict__ ps, const float4 *__restrict__ com,
                const int4 *__restrict__ meta, int n, int cap, float theta2, float eps2,
                DeviceParams *P, float *__restrict__ acc_s, uint32_t *__restrict__ cnt_s)
{
    __shared__ float s_side2[kLevels + 1];
    __shared__ float4 s_leaf[kWarpsPerBlock][32];
    __shared__ int s_state[2];
    if (threadIdx.x <= kLevels) s_side2[threadIdx.x] = P->s2[threadIdx.x];
    if (threadIdx.x == 0) {
        s_state[0] = P->status;
        s_state[1] = P->num_nodes;
    }
    __syncthreads();
    if (s_state[0] != 0) return;  // block-uniform: skip the walk on a bad input
    const int num_nodes = s_state[1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kThreads + threadIdx.x;
    const bool valid = t < n;
    const float4 xi = valid ? __ldg(ps + t) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int next = valid ? 0 : num_nodes;
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    uint32_t pc = 0, pp = 0, vis = 0;
    float4 *stage = s_leaf[warp];

    for (int step = 0;; ++step) {
        const int k = __reduce_min_sync(0xffffffffu, next);
        if (k >= num_nodes) break;
        if (step > num_nodes) {  // unreachable: k strictly increases
            if (lane == 0) atomicOr(&P->status, kStatusWalkBound);
            break;
        }
        const float4 c = __ldg(com + k);
        const int4 m = __ldg(meta + k);  // {escape, first, count, level}
        if (kCount) vis += valid ? 1u : 0u;
        bool open_leaf = false;
        if (next == k) {
            const float dx = __fsub_rn(c.x, xi.x);
            const float dy = __fsub_rn(c.y, xi.y);
            const float dz = __fsub_rn(c.z, xi.z);
            const float d2 = dist2(dx, dy, dz);
            if (s_side2[m.w] < __fmul_rn(theta2, d2)) {
                add_term(dx, dy, dz, d2, c.w, eps2, ax, ay, az);
                if (kCount) ++pc;
                next = m.x;
            } else if (m.z <= cap || m.w == kLevels) {
                open_leaf = true;
                next = m.x;
            } else {
                next = k + 1;
            }
        }
        if (__ballot_sync(0xffffffffu, open_leaf)) {
            if (m.y < 0 || m.z < 0 || m.y + m.z > n) {  // warp-uniform consistency check
                if (lane == 0) atomicOr(&P->status, kStatusInternal);
                break;
            }
            for (int base = 0; base < m.z; base += 32) {
                const int chunk = min(32, m.z - base);
                if (lane < chunk) stage[lane] = __ldg(ps + m.y + base + lane);
                __syncwarp();
                if (open_leaf) {
                    const int self = t - (m.y + base);
                    for (int j = 0; j < chunk; ++j) {
                        if (j == self) continue;
                        const float4 p = stage[j];
                        const float dx = __fsub_rn(p.x, xi.x);
                        const float dy = __fsub_rn(p.y, xi.y);
                        const float dz = __fsub_rn(p.z, xi.z);
                        add_term(dx, dy, dz, dist2(dx, dy, dz), p.w, eps2, ax, ay, az);
                        if (kCount) ++pp;
                    }
                }
                __syncwarp();
            }
        }
    }
    if (valid) {
        acc_s[3 * (int64_t)t + 0] = ax;
        acc_s[3 * (int64_t)t + 1] = ay;
        acc_s[3 * (int64_t)t + 2] = az;
        if (kCount) {
            cnt_s[3 * (int64_t)t + 0] = pc;
            cnt_s[3 * (int64_t)t + 1] = pp;
            cnt_s[3 * (int64_t)t + 2] = vis;
        }
    }
}

template <bool kCount>
__global__ void __launch_bounds__(kThreads)
k_walk_independent(const float4 *__restrict__ ps, const float4 *__restrict__ com,
                   const int4 *__restrict__ meta, int n, int cap, float theta2, float eps2,
                   DeviceParams *P, float *__restrict__ acc_s, uint32_t *__restrict__ cnt_s)
{
    __shared__ float s_side2[kLevels + 1];
    __shared__ int s_state[2];
    if (threadIdx.x <= kLevels) s_side2[threadIdx.x] = P->s2[threadIdx.x];
    if (threadIdx.x == 0) {
        s_state[0] = P->status;
        s_state[1] = P->num_nodes;
    }
    __syncthreads();
    if (s_state[0] != 0) return;
    const int num_nodes = s_state[1];
    const int t = blockIdx.x * kThreads + threadIdx.x;
    if (t >= n) return;
    const float4 xi = __ldg(ps + t);
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    uint32_t pc = 0, pp = 0, vis = 0;
    int k = 0;
    for (int step = 0; k < num_nodes; ++step) {
        if (step > num_nodes) {  // unreachable: k strictly increases
            atomicOr(&P->status, kStatusWalkBound);
            break;
        }
        const float4 c = __ldg(com + k);
        const int4 m = __ldg(meta + k);
        if (kCount) ++vis;
        const float dx = __fsub_rn(c.x, xi.x);
        const float dy = __fsub_rn(c.y, xi.y);
        const float dz = __fsub_rn(c.z, xi.z);
        const float d2 = dist2(dx, dy, dz);
        if (s_side2[m.w] < __fmul_rn(theta2, d2)) {
            add_term(dx, dy, dz, d2, c.w, eps2, ax, ay, az);
            if (kCount) ++pc;
            k = m.x;
        } else if (m.z <= cap || m.w == kLevels) {
            if (m.y < 0 || m.z < 0 || m.y + m.z > n) {
                atomicOr(&P->status, kStatusInternal);
                break;
            }
            for (int j = m.y; j < m.y + m.z; ++j) {
                if (j == t) continue;
                const float4 p = __ldg(ps + j);
                const float ex = __fsub_rn(p.x, xi.x);
                const float ey = __fsub_rn(p.y, xi.y);
                const float ez = __fsub_rn(p.z, xi.z);
                add_term(ex, ey, ez, dist2(ex, ey, ez), p.w, eps2, ax, ay, az);
                if (kCount) ++pp;
            }
            k = m.x;
        } else {
            k = k + 1;
        }
    }
    acc_s[3 * (int64_t)t + 0] = ax;
    acc_s[3 * (int64_t)t + 1] = ay;
    acc_s[3 * (int64_t)t + 2] = az;
    if (kCount) {
        cnt_s[3 * (int64_t)t + 0] = pc;
        cnt_s[3 * (int64_t)t + 1] = pp;
        cnt_s[3 * (int64_t)t + 2] = vis;
    }
}

}  // namespace

void launch_walk(int traversal, float theta, float eps, int32_t leaf_cap, bool count,
                 const Buffers &b, cudaStream_t st)
{
    const float theta2 = theta * theta;  // host binary32 products, round to nearest
    const float eps2 = eps * eps;
    const unsigned grid = ceil_div(b.n, kThreads);
    const int n = (int)b.n;
    if (traversal == 1) {
        if (count)
            k_walk_coherent<true><<<grid, kThreads, 0, st>>>(b.ps, b.com, b.meta, n, leaf_cap,
                                                             theta2, eps2, b.params, b.acc_s,
                                                             b.cnt_s);
        else
            k_walk_coherent<false><<<grid, kThreads, 0, st>>>(b.ps, b.com, b.meta, n, leaf_cap,
                                                              theta2, eps2, b.params, b.acc_s,
                                                              b.cnt_s);
    } else {
        if (count)
            k_walk_independent<true><<<grid, kThreads, 0, st>>>(b.ps, b.com, b.meta, n,
                                                                leaf_cap, theta2, eps2, b.params,
                                                                b.acc_s, b.cnt_s);
        else
            k_walk_independent<false><<<grid, kThreads, 0, st>>>(b.ps, b.com, b.meta, n,
                                                                 leaf_cap, theta2, eps2,
                                                                 b.params, b.acc_s, b.cnt_s);
    }
    g_launches += 1;
}

}  // namespace obh
