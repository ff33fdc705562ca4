// bh_walk.cu -- a7 (with a8 fused): the stackless traversals of the depth-first
// octree; each target writes its results to its caller-order slot.
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
// Term: r2 = d2 + eps^2, y = rsqrt_newton(r2), f = (m y)(y y), a += f
// (x_src - x_i) by fused multiply-add. Every floating-point step is one
// correctly rounded binary32 operation (explicit _rn intrinsics), so
// decisions and sums do not depend on contraction choices, and a CPU
// restatement of the same steps reproduces them bit for bit.
//
// GB300 shape of the coherent kernel: the node k is group-uniform, so its two
// 16-byte records are read once per group step and broadcast. The walk record
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
#include <type_traits>

#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

struct WalkArgs {
    const float4 *ps;      // sorted particles {x, y, z, m}
    const float4 *com;     // {CoM_x, CoM_y, CoM_z, M}
    const int4 *wnode;     // {escape, first, leaf count or 0, squared side bits}
    const uint32_t *perm;  // caller index of each sorted slot
    int n;
    float theta2;
    float eps2;
    DeviceParams *P;
    float *acc;            // caller order [n][3]
    uint32_t *inter;       // caller order [n][2] or null
    uint32_t *visits;      // caller order [n] or null
};

// a8, fused: a target's results go straight to its caller-order slot.
template <bool kCount>
__device__ __forceinline__ void store_target(const WalkArgs &a, int t, float ax, float ay, float az,
                                             uint32_t pc, uint32_t pp, uint32_t visits)
{
    const uint32_t o = __ldg(a.perm + t);
    if (o >= (uint32_t)a.n) {
        atomicOr(&a.P->status, kStatusInternal);
        return;
    }
    a.acc[3 * (int64_t)o + 0] = ax;
    a.acc[3 * (int64_t)o + 1] = ay;
    a.acc[3 * (int64_t)o + 2] = az;
    if (kCount) {
        if (a.inter) {
            a.inter[2 * (int64_t)o + 0] = pc;
            a.inter[2 * (int64_t)o + 1] = pp;
        }
        if (a.visits) a.visits[o] = visits;
    }
}

// 1/sqrt(x) by a fixed binary32 recipe: the bit-level seed of C. Lomont,
// "Fast Inverse Square Root" (2003) -- the integer 0x5f375a86 minus half the
// bits of x -- then three Newton-Raphson steps y <- y (3/2 - (x/2) y^2), each
// as fl(y * fma(-h, fl(y y), 3/2)) with h = fl(x/2). Within 2 ulp of 1/sqrt(x)
// for normal x; no MUFU and no branch, and reproducible on any IEEE CPU.
__device__ __forceinline__ float rsqrt_newton(float x)
{
    const float h = __fmul_rn(0.5f, x);
    float y = __int_as_float(0x5f375a86 - (int)((unsigned)__float_as_int(x) >> 1));
#pragma unroll
    for (int it = 0; it < 3; ++it) y = __fmul_rn(y, __fmaf_rn(-h, __fmul_rn(y, y), 1.5f));
    return y;
}

// kFast selects the hardware approximate inverse square root (rsqrtf, a few
// ulp) in place of the Newton sequence: faster, no longer reproducible bit for
// bit on a CPU (the caller opts in with ORRERY_FAST_TERM).
template <bool kFast>
__device__ __forceinline__ float inv_sqrt(float x)
{
    return kFast ? rsqrtf(x) : rsqrt_newton(x);
}

template <bool kFast>
__device__ __forceinline__ void add_term(float dx, float dy, float dz, float d2, float m,
                                         float eps2, float &ax, float &ay, float &az)
{
    const float r2 = __fadd_rn(d2, eps2);
    const float y = inv_sqrt<kFast>(r2);
    const float f = __fmul_rn(__fmul_rn(m, y), __fmul_rn(y, y));
    ax = __fmaf_rn(f, dx, ax);
    ay = __fmaf_rn(f, dy, ay);
    az = __fmaf_rn(f, dz, az);
}

__device__ __forceinline__ float dist2(float dx, float dy, float dz)
{
    return __fmaf_rn(dz, dz, __fmaf_rn(dy, dy, __fmul_rn(dx, dx)));
}

template <bool kFast>
__device__ __forceinline__ void particle_term(const float4 &p, const float4 &xi, float eps2,
                                              float &ax, float &ay, float &az)
{
    const float dx = __fsub_rn(p.x, xi.x);
    const float dy = __fsub_rn(p.y, xi.y);
    const float dz = __fsub_rn(p.z, xi.z);
    add_term<kFast>(dx, dy, dz, dist2(dx, dy, dz), p.w, eps2, ax, ay, az);
}

// Block prologue shared by both kernels: status, node count and whether the
// self term may be summed (see the file comment). Returns false to skip.
template <bool kFast>
__device__ __forceinline__ bool prologue(const WalkArgs &a, int &num_nodes, bool &self_free)
{
    __shared__ int s_state[3];
    if (threadIdx.x == 0) {
        const DeviceParams *P = a.P;
        s_state[0] = P->status;
        s_state[1] = P->num_nodes;
        bool ok = a.eps2 > 0.0f;
        if (ok) {
            const float y = inv_sqrt<kFast>(a.eps2);
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

// One coherence group = W consecutive sorted targets sharing one node index.
// W = 16: half a warp per group (two groups per warp, each advancing on its
// own, like the pages' sub-group width of 16); W = 32: one warp; W = 64: one
// warp with two targets per lane (the width the pages could not measure).
// Lane l of a group holds targets base + i*G + l for i < T, with G lanes per
// group and T targets per lane.
template <int W>
struct Group {
    static constexpr int G = W < 32 ? W : 32;
    static constexpr int T = W > 32 ? W / 32 : 1;
};

// kBallot selects how the group finds its next node. The default takes the
// minimum over the lanes' wanted indices (ADR-0029, Decision). The ballot form
// (ADR-0029, Alternatives considered: "Vote on whether to descend, and
// otherwise follow the current node's escape index") goes to k + 1 if any
// lane active at k descends and to escape(k) otherwise. With per-lane skip
// indices both pick the same node -- a lane inactive at k waits at the escape
// of an accepted ancestor of k, which is never below escape(k) -- so the
// ballot form visits exactly the same union; it is kept to measure the cost
// of the two instructions against each other.
template <int W, bool kCount, bool kSelfFree, bool kBallot, bool kFast>
__device__ __forceinline__ void coherent_walk(const WalkArgs &a, int num_nodes, float4 *stage)
{
    constexpr int G = Group<W>::G;
    constexpr int T = Group<W>::T;
    const int lane = threadIdx.x & 31;
    const int glane = lane & (G - 1);
    const unsigned gmask = (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    const int base = ((blockIdx.x * kThreads + threadIdx.x) / G) * W;

    int tgt[T], next[T];
    bool valid[T];
    float4 xi[T];
    float ax[T], ay[T], az[T];
    uint32_t pc[T], pp[T];
#pragma unroll
    for (int i = 0; i < T; ++i) {
        tgt[i] = base + i * G + glane;
        valid[i] = tgt[i] < a.n;
        xi[i] = valid[i] ? __ldg(a.ps + tgt[i]) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        next[i] = valid[i] ? 0 : num_nodes;
        ax[i] = ay[i] = az[i] = 0.0f;
        pc[i] = pp[i] = 0;
    }
    int steps = 0;
    int kb = __any_sync(gmask, valid[0]) ? 0 : num_nodes;  // the ballot form's node
    for (; steps <= num_nodes; ++steps) {
        int k;
        if (kBallot) {
            k = kb;
        } else {
            int v = next[0];
#pragma unroll
            for (int i = 1; i < T; ++i) v = min(v, next[i]);
            k = __reduce_min_sync(gmask, v);
        }
        if (k >= num_nodes) break;
        const float4 c = __ldg(a.com + k);
        const int4 w = __ldg(a.wnode + k);
        bool open[T];
        bool any_open = false;
        bool descend = false;
#pragma unroll
        for (int i = 0; i < T; ++i) {
            open[i] = false;
            if (next[i] == k) {
                const float dx = __fsub_rn(c.x, xi[i].x);
                const float dy = __fsub_rn(c.y, xi[i].y);
                const float dz = __fsub_rn(c.z, xi[i].z);
                const float d2 = dist2(dx, dy, dz);
                if (__int_as_float(w.w) < __fmul_rn(a.theta2, d2)) {
                    add_term<kFast>(dx, dy, dz, d2, c.w, a.eps2, ax[i], ay[i], az[i]);
                    if (kCount) ++pc[i];
                    next[i] = w.x;
                } else {
                    open[i] = w.z != 0;
                    next[i] = open[i] ? w.x : k + 1;
                    descend |= !open[i];
                }
            }
            any_open |= open[i];
        }
        if (kBallot) kb = __any_sync(gmask, descend) ? k + 1 : w.x;
        if (__any_sync(gmask, any_open)) {
            const int first = w.y, count = w.z;
            if (first < 0 || first > a.n - count) {  // group-uniform consistency check
                if (glane == 0) atomicOr(&a.P->status, kStatusInternal);
                break;
            }
#pragma unroll
            for (int i = 0; i < T; ++i)
                if (kCount && open[i])
                    pp[i] += count - ((unsigned)(tgt[i] - first) < (unsigned)count ? 1u : 0u);
            for (int b = 0; b < count; b += G) {
                const int chunk = min(G, count - b);
                if (glane < chunk) stage[glane] = __ldg(a.ps + first + b + glane);
                __syncwarp(gmask);
#pragma unroll
                for (int i = 0; i < T; ++i) {
                    if (!open[i]) continue;
                    if (kSelfFree) {
#pragma unroll 4
                        for (int j = 0; j < chunk; ++j)
                            particle_term<kFast>(stage[j], xi[i], a.eps2, ax[i], ay[i], az[i]);
                    } else {
                        const int self = tgt[i] - (first + b);
                        for (int j = 0; j < chunk; ++j)
                            if (j != self) particle_term<kFast>(stage[j], xi[i], a.eps2, ax[i], ay[i], az[i]);
                    }
                }
                __syncwarp(gmask);
            }
        }
    }
    if (steps > num_nodes && glane == 0) atomicOr(&a.P->status, kStatusWalkBound);
#pragma unroll
    for (int i = 0; i < T; ++i)  // every step visits the group's union
        if (valid[i]) store_target<kCount>(a, tgt[i], ax[i], ay[i], az[i], pc[i], pp[i], steps);
}

template <int W, bool kCount, bool kBallot, bool kFast>
__global__ void __launch_bounds__(kThreads) k_walk_coherent(WalkArgs a)
{
    __shared__ float4 s_leaf[kWarpsPerBlock][32];
    int num_nodes;
    bool self_free;
    if (!prologue<kFast>(a, num_nodes, self_free)) return;  // block-uniform
    constexpr int G = Group<W>::G;
    float4 *stage = &s_leaf[threadIdx.x >> 5][(threadIdx.x & 31) & ~(G - 1)];
    if (self_free)
        coherent_walk<W, kCount, true, kBallot, kFast>(a, num_nodes, stage);
    else
        coherent_walk<W, kCount, false, kBallot, kFast>(a, num_nodes, stage);
}

// The scheme the pages reject, kept as a measured contrast (ADR-0029,
// Alternatives considered: "Descend wherever any lane must, and let the
// accepting lanes descend too"). One node index per warp; at node k the warp
// accepts only if every target accepts (each then adds the cell term),
// otherwise a leaf is opened for every target and an internal node is
// entered by all. Each target's sum depends on which targets share its warp,
// so this is a different function of the input from the walks above.
template <bool kCount, bool kSelfFree, bool kFast>
__device__ __forceinline__ void together_walk(const WalkArgs &a, int num_nodes, float4 *stage)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kThreads + threadIdx.x;
    const bool valid = t < a.n;
    const float4 xi = valid ? __ldg(a.ps + t) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    uint32_t pc = 0, pp = 0;
    int k = 0, steps = 0;
    for (; k < num_nodes && steps <= num_nodes; ++steps) {
        const float4 c = __ldg(a.com + k);
        const int4 w = __ldg(a.wnode + k);
        const float dx = __fsub_rn(c.x, xi.x);
        const float dy = __fsub_rn(c.y, xi.y);
        const float dz = __fsub_rn(c.z, xi.z);
        const float d2 = dist2(dx, dy, dz);
        const bool accept = __int_as_float(w.w) < __fmul_rn(a.theta2, d2);
        if (__all_sync(0xffffffffu, accept || !valid)) {
            if (valid) {
                add_term<kFast>(dx, dy, dz, d2, c.w, a.eps2, ax, ay, az);
                if (kCount) ++pc;
            }
            k = w.x;
        } else if (w.z != 0) {
            const int first = w.y, count = w.z;
            if (first < 0 || first > a.n - count) {  // warp-uniform consistency check
                if (lane == 0) atomicOr(&a.P->status, kStatusInternal);
                break;
            }
            if (kCount && valid)
                pp += count - ((unsigned)(t - first) < (unsigned)count ? 1u : 0u);
            for (int b = 0; b < count; b += 32) {
                const int chunk = min(32, count - b);
                if (lane < chunk) stage[lane] = __ldg(a.ps + first + b + lane);
                __syncwarp();
                if (valid) {
                    if (kSelfFree) {
#pragma unroll 4
                        for (int j = 0; j < chunk; ++j)
                            particle_term<kFast>(stage[j], xi, a.eps2, ax, ay, az);
                    } else {
                        const int self = t - (first + b);
                        for (int j = 0; j < chunk; ++j)
                            if (j != self) particle_term<kFast>(stage[j], xi, a.eps2, ax, ay, az);
                    }
                }
                __syncwarp();
            }
            k = w.x;
        } else {
            k = k + 1;
        }
    }
    if (k < num_nodes && lane == 0) atomicOr(&a.P->status, kStatusWalkBound);
    if (valid) store_target<kCount>(a, t, ax, ay, az, pc, pp, steps);
}

template <bool kCount, bool kFast>
__global__ void __launch_bounds__(kThreads) k_walk_together(WalkArgs a)
{
    __shared__ float4 s_leaf[kWarpsPerBlock][32];
    int num_nodes;
    bool self_free;
    if (!prologue<kFast>(a, num_nodes, self_free)) return;  // block-uniform
    float4 *stage = s_leaf[threadIdx.x >> 5];
    if (self_free)
        together_walk<kCount, true, kFast>(a, num_nodes, stage);
    else
        together_walk<kCount, false, kFast>(a, num_nodes, stage);
}

template <bool kCount, bool kSelfFree, bool kFast>
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
            add_term<kFast>(dx, dy, dz, d2, c.w, a.eps2, ax, ay, az);
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
                if (kSelfFree || j != t) particle_term<kFast>(__ldg(a.ps + j), xi, a.eps2, ax, ay, az);
            k = w.x;
        } else {
            k = k + 1;
        }
    }
    if (k < num_nodes) atomicOr(&a.P->status, kStatusWalkBound);
    store_target<kCount>(a, t, ax, ay, az, pc, pp, steps);
}

template <bool kCount, bool kFast>
__global__ void __launch_bounds__(kThreads) k_walk_independent(WalkArgs a)
{
    int num_nodes;
    bool self_free;
    if (!prologue<kFast>(a, num_nodes, self_free)) return;
    if (self_free)
        independent_walk<kCount, true, kFast>(a, num_nodes);
    else
        independent_walk<kCount, false, kFast>(a, num_nodes);
}

template <bool kFast>
void launch_kernels(int traversal, bool count, unsigned grid, const WalkArgs &a, cudaStream_t st)
{
    // coherent groups of W targets: kThreads lanes cover kThreads * T targets
    auto coherent = [&](auto wtag) {
        constexpr int W = decltype(wtag)::value;
        const unsigned g = ceil_div(a.n, (int64_t)kThreads * Group<W>::T);
        if (count)
            k_walk_coherent<W, true, false, kFast><<<g, kThreads, 0, st>>>(a);
        else
            k_walk_coherent<W, false, false, kFast><<<g, kThreads, 0, st>>>(a);
    };
    switch (traversal) {
    case 1: coherent(std::integral_constant<int, 32>{}); break;
    case 2: coherent(std::integral_constant<int, 16>{}); break;
    case 3: coherent(std::integral_constant<int, 64>{}); break;
    case 4:
        if (count)
            k_walk_together<true, kFast><<<grid, kThreads, 0, st>>>(a);
        else
            k_walk_together<false, kFast><<<grid, kThreads, 0, st>>>(a);
        break;
    case 5:
        if (count)
            k_walk_coherent<32, true, true, kFast><<<grid, kThreads, 0, st>>>(a);
        else
            k_walk_coherent<32, false, true, kFast><<<grid, kThreads, 0, st>>>(a);
        break;
    default:
        if (count)
            k_walk_independent<true, kFast><<<grid, kThreads, 0, st>>>(a);
        else
            k_walk_independent<false, kFast><<<grid, kThreads, 0, st>>>(a);
    }
}

}  // namespace

void launch_walk(int traversal_flags, float theta, float eps, const uint32_t *perm,
                 const Buffers &b, float *acc, uint32_t *inter, uint32_t *visits, cudaStream_t st)
{
    const int traversal = traversal_flags & kTraversalMask;
    const bool fast = (traversal_flags & kFastTermFlag) != 0;
    const bool count = inter != nullptr || visits != nullptr;
    WalkArgs a;
    a.ps = b.ps;
    a.com = b.com;
    a.wnode = b.wnode;
    a.perm = perm;
    a.n = (int)b.n;
    a.theta2 = theta * theta;  // host binary32 products, round to nearest
    a.eps2 = eps * eps;
    a.P = b.params;
    a.acc = acc;
    a.inter = inter;
    a.visits = visits;
    const unsigned grid = ceil_div(b.n, kThreads);
    if (fast)
        launch_kernels<true>(traversal, count, grid, a, st);
    else
        launch_kernels<false>(traversal, count, grid, a, st);
    g_launches += 1;
}

}  // namespace obh
