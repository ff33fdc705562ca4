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
// the independent and the coherent kernels below produce bit-identical sums
// and counters.
//
// Per target i at node k of level L (a visit is one acceptance test):
//   accept iff (side 2^-L)^2 < theta^2 |CoM_k - x_i|^2  -> cell term, escape
//   else if k is a leaf -> particle terms over its particles j != i, escape
//   else -> k + 1 (first child)
// Term (the softened law a = m r / (r^2 + eps^2)^(3/2)): r2 = d2 + eps^2,
// y = 1/sqrt(r2) (a fixed Newton sequence, or the hardware approximation
// with the fast-term flag), f = (m y)(y y), a += f (x_src - x_i) by fused
// multiply-add, in walk order. Every floating-point step is one correctly
// rounded binary32 operation (explicit _rn intrinsics), so decisions and sums
// do not depend on contraction choices: a CPU restatement of the decisions
// reproduces the counts bit for bit, and of the Newton term the sums.
//
// GB300 shape of the coherent kernels: the node k is group-uniform, so its
// 32-byte record (one sector) is read once per group step and broadcast. The
// record {escape, next node when not accepted, leaf count (0 = internal),
// squared side bits; CoM, M} carries everything a step decides on, so a step
// needs no table lookup and no select on the leaf flag. An opened leaf's
// particles are staged into shared memory once (one coalesced 16-byte load
// per lane) and read back as broadcasts by every lane that opened it. The
// loop is warp-uniform and ends within num_nodes steps without a per-step
// bound: every record's next nodes lie in (k, num_nodes] (the build checks
// each one), so the group's node index strictly increases, and the record
// at num_nodes is a sentinel leaf that no target accepts, so a group whose
// targets are all done opens it and stops there, in the leaf branch, with no
// per-step test of k. The default width-64 kernel (k_walk_paired, below)
// holds two targets per lane and does their arithmetic in packed float2
// instructions.
//
// The self term. When the target's own leaf is opened the oracle skips j = i.
// Summing it instead changes nothing, bit for bit, whenever its force factor
// is finite: dx = dy = dz = +0, so fma(f, +0, a) = a (a is never -0: it
// starts at +0 and round-to-nearest never produces -0 from a sum of unlike
// signs). The kernels test once per block that eps^2 is a normal number and
// that twice the largest particle factor, (m_max y)(y y) at y = rsqrt(eps^2),
// is finite; then every factor is finite (r2 >= eps^2 and the roots are within
// a few ulp of monotone), every r2 is normal (so the fast term may use the
// flush-to-zero hardware root), and the per-particle self comparison is
// dropped.
#include <atomic>
#include <cfloat>
#include <type_traits>

#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;

struct WalkArgs {
    const float4 *ps;      // sorted particles {x, y, z, m}
    const WalkNode *wnode; // {escape, next if not accepted, leaf count or 0, side^2 bits}, {CoM, M}
    const int4 *meta;      // node table {escape, first, count, level}: a leaf's first particle
    const uint32_t *perm;  // caller index of each sorted slot
    int n;                 // particles (sources)
    int t_begin, t_end;    // the sorted targets walked: [t_begin, t_end)
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

// The hardware approximate inverse square root with subnormal inputs flushed:
// the same value as rsqrtf for every normal input, without rsqrtf's extra
// handling of subnormal ones.
__device__ __forceinline__ float rsqrt_ftz(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// kFast selects the hardware approximate inverse square root (a few ulp) in
// place of the Newton sequence: faster, no longer reproducible bit for bit on
// a CPU (the caller opts in with ORRERY_FAST_TERM). kNormal: the argument is
// known to be a normal number (every r2 >= eps^2 >= FLT_MIN).
template <bool kFast, bool kNormal = false>
__device__ __forceinline__ float inv_sqrt(float x)
{
    return kFast ? (kNormal ? rsqrt_ftz(x) : rsqrtf(x)) : rsqrt_newton(x);
}

template <bool kFast, bool kNormal = false>
__device__ __forceinline__ void add_term(float dx, float dy, float dz, float d2, float m,
                                         float eps2, float &ax, float &ay, float &az)
{
    const float r2 = __fadd_rn(d2, eps2);
    const float y = inv_sqrt<kFast, kNormal>(r2);
    const float f = __fmul_rn(__fmul_rn(m, y), __fmul_rn(y, y));
    ax = __fmaf_rn(f, dx, ax);
    ay = __fmaf_rn(f, dy, ay);
    az = __fmaf_rn(f, dz, az);
}

__device__ __forceinline__ float dist2(float dx, float dy, float dz)
{
    return __fmaf_rn(dz, dz, __fmaf_rn(dy, dy, __fmul_rn(dx, dx)));
}

template <bool kFast, bool kNormal = false>
__device__ __forceinline__ void particle_term(const float4 &p, const float4 &xi, float eps2,
                                              float &ax, float &ay, float &az)
{
    const float dx = __fsub_rn(p.x, xi.x);
    const float dy = __fsub_rn(p.y, xi.y);
    const float dz = __fsub_rn(p.z, xi.z);
    add_term<kFast, kNormal>(dx, dy, dz, dist2(dx, dy, dz), p.w, eps2, ax, ay, az);
}

// The same two functions for one target with its x and y components in one
// packed pair (__fadd2_rn and __ffma2_rn round each component exactly like
// the scalar forms, and d2 keeps its sequential order): the same results bit
// for bit, in two fewer instructions per term. nxy = (-x_i, -y_i): a
// separation is then one packed add.
template <bool kFast, bool kNormal = false>
__device__ __forceinline__ void add_term_xy(float2 dxy, float dz, float d2, float m, float eps2,
                                            float2 &axy, float &az)
{
    const float r2 = __fadd_rn(d2, eps2);
    const float y = inv_sqrt<kFast, kNormal>(r2);
    const float f = __fmul_rn(__fmul_rn(m, y), __fmul_rn(y, y));
    axy = __ffma2_rn(make_float2(f, f), dxy, axy);
    az = __fmaf_rn(f, dz, az);
}

template <bool kFast, bool kNormal = false>
__device__ __forceinline__ void particle_term_xy(const float4 &p, float2 nxy, float z, float eps2,
                                                 float2 &axy, float &az)
{
    const float2 dxy = __fadd2_rn(make_float2(p.x, p.y), nxy);
    const float dz = __fsub_rn(p.z, z);
    add_term_xy<kFast, kNormal>(dxy, dz, dist2(dxy.x, dxy.y, dz), p.w, eps2, axy, az);
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
        bool ok = a.eps2 >= FLT_MIN;
        if (ok) {
            const float y = inv_sqrt<kFast>(a.eps2);
            const float f = __fmul_rn(__fmul_rn(P->mmax, y), __fmul_rn(y, y));
            ok = isfinite(__fmul_rn(f, 2.0f));
        }
        s_state[2] = ok ? 1 : 0;
    }
    __syncthreads();
    num_nodes = s_state[1];
    self_free = s_state[2] != 0;
    return s_state[0] == 0;
}

// Shared-memory copies of everything a walk step reads, for small problems.
struct LocalTree {
    const WalkNode *nodes;  // [num_nodes]
    const int *first;       // [num_nodes] first particle of each node
    const float4 *ps;       // [n] sorted particles, or null: leaves read global memory
};

// One coherence group = W consecutive sorted targets sharing one node index,
// one target per lane. W = 16: half a warp per group (two groups per warp,
// each advancing on its own, like the pages' sub-group width of 16); W = 32:
// one warp. (Width 64 -- two targets per lane -- is the packed walk below.)
//
// kBallot selects how the group finds its next node. The default takes the
// minimum over the lanes' wanted indices (ADR-0029, Decision). The ballot form
// (ADR-0029, Alternatives considered: "Vote on whether to descend, and
// otherwise follow the current node's escape index") goes to k + 1 if any
// lane active at k descends and to escape(k) otherwise. With per-lane skip
// indices both pick the same node -- a lane inactive at k waits at the escape
// of an accepted ancestor of k, which is never below escape(k) -- so the
// ballot form visits exactly the same union; it is kept to measure the cost
// of the two instructions against each other.
template <int W, bool kCount, bool kSelfFree, bool kBallot, bool kFast, bool kLocal = false>
__device__ __forceinline__ void coherent_walk(const WalkArgs &a, int num_nodes, float4 *stage,
                                              LocalTree loc = LocalTree{})
{
    static_assert(W == 16 || W == 32, "one target per lane");
    constexpr int G = W;
    const int lane = threadIdx.x & 31;
    const int glane = lane & (G - 1);
    const unsigned gmask = (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    const int tgt = a.t_begin + blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = tgt < a.t_end;
    const float4 xi = valid ? __ldg(a.ps + tgt) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float2 nxy = make_float2(-xi.x, -xi.y);
    int next = valid ? 0 : num_nodes;
    float2 axy = make_float2(0.0f, 0.0f);
    float az = 0.0f;
    uint32_t pc = 0, pp = 0;
    int steps = 0;
    int kb = __any_sync(gmask, valid) ? 0 : num_nodes;  // the ballot form's node
    // k <= num_nodes: the group ends at the sentinel record after the last
    // node (a leaf no target accepts), in the leaf branch, as the packed walk
    for (;; ++steps) {  // ends: the node index strictly increases
        const int k = kBallot ? kb : __reduce_min_sync(gmask, next);
        const int4 w = kLocal ? loc.nodes[k].w : __ldg(&a.wnode[k].w);
        const float4 c = kLocal ? loc.nodes[k].c : __ldg(&a.wnode[k].c);
        bool open = false, descend = false;
        if (next == k) {
            const float2 dxy = __fadd2_rn(make_float2(c.x, c.y), nxy);
            const float dz = __fsub_rn(c.z, xi.z);
            const float d2 = dist2(dxy.x, dxy.y, dz);
            if (__int_as_float(w.w) < __fmul_rn(a.theta2, d2)) {
                add_term_xy<kFast, kSelfFree>(dxy, dz, d2, c.w, a.eps2, axy, az);
                if (kCount) ++pc;
                next = w.x;
            } else {
                open = w.z != 0;
                next = w.y;
                descend = !open;
            }
        }
        if (kBallot) kb = __any_sync(gmask, descend) ? k + 1 : w.x;
        if (w.z != 0 && __any_sync(gmask, open)) {  // w.z: group-uniform
            if (k >= num_nodes) break;  // the sentinel
            const int first = kLocal ? loc.first[k] : __ldg(&a.meta[k].y), count = w.z;
            if (first < 0 || first > a.n - count) {  // group-uniform consistency check
                if (glane == 0) atomicOr(&a.P->status, kStatusInternal);
                break;
            }
            if (kCount && open) pp += count - ((unsigned)(tgt - first) < (unsigned)count ? 1u : 0u);
            if (kLocal && loc.ps) {  // the particles are in shared memory: read them as broadcasts
                if (open) {
                    const int self = tgt - first;
#pragma unroll 4
                    for (int j = 0; j < count; ++j)
                        if (kSelfFree || j != self)
                            particle_term_xy<kFast, kSelfFree>(loc.ps[first + j], nxy, xi.z, a.eps2, axy, az);
                }
                continue;
            }
            for (int b = 0; b < count; b += G) {
                const int chunk = min(G, count - b);
                if (glane < chunk) stage[glane] = __ldg(a.ps + first + b + glane);
                __syncwarp(gmask);
                if (open) {
                    if (kSelfFree) {
#pragma unroll 4
                        for (int j = 0; j < chunk; ++j)
                            particle_term_xy<kFast, kSelfFree>(stage[j], nxy, xi.z, a.eps2, axy, az);
                    } else {
                        const int self = tgt - (first + b);
                        for (int j = 0; j < chunk; ++j)
                            if (j != self) particle_term_xy<kFast, kSelfFree>(stage[j], nxy, xi.z, a.eps2, axy, az);
                    }
                }
                __syncwarp(gmask);
            }
        }
    }
    if (steps > num_nodes && glane == 0) atomicOr(&a.P->status, kStatusWalkBound);
    if (valid) store_target<kCount>(a, tgt, axy.x, axy.y, az, pc, pp, steps);  // every step visits the union
}

template <int W, bool kCount, bool kBallot, bool kFast>
__global__ void __launch_bounds__(kThreads) k_walk_coherent(WalkArgs a)
{
    __shared__ float4 s_leaf[kWarpsPerBlock][32];
    int num_nodes;
    bool self_free;
    if (!prologue<kFast>(a, num_nodes, self_free)) return;  // block-uniform
    float4 *stage = &s_leaf[threadIdx.x >> 5][(threadIdx.x & 31) & ~(W - 1)];
    if (self_free)
        coherent_walk<W, kCount, true, kBallot, kFast>(a, num_nodes, stage);
    else
        coherent_walk<W, kCount, false, kBallot, kFast>(a, num_nodes, stage);
}

// ---------------------------------------------------------------------------
// Width 64: one warp, two targets per lane, in packed pairs. Blackwell issues
// two binary32 operations of one thread in one instruction (__fadd2_rn,
// __fmul2_rn, __ffma2_rn; each component is rounded exactly like its scalar
// form), so a lane does both of its targets' acceptance tests and terms in
// the issue slots of one. The warp still shares one node index, the minimum
// over its 64 targets' wanted indices, and each target still follows its own
// walk. To keep a pair in step, the cell term at node k is evaluated for both
// targets of every lane, and a target that does not accept k (or is not at k)
// adds it with a zero factor: fma(+0, dx, a) = a exactly for any finite dx (a
// is never -0, see the file comment), so its sum is unchanged bit for bit.
// Leaf particles are handled the same way for targets that did not open the
// leaf. Every separation is finite because coordinates below 2^125 and node
// centres of mass below 2^126 are checked before the walk runs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

template <bool kFast, bool kNormal = false>
__device__ __forceinline__ float2 inv_sqrt2(float2 x)
{
    if (kFast) return make_float2(inv_sqrt<true, kNormal>(x.x), inv_sqrt<true, kNormal>(x.y));
    // rsqrt_newton componentwise; -h is formed as fl(-x/2), which equals
    // -fl(x/2) bit for bit
    const float2 nh = __fmul2_rn(splat(-0.5f), x);
    float2 y = make_float2(__int_as_float(0x5f375a86 - (int)((unsigned)__float_as_int(x.x) >> 1)),
                           __int_as_float(0x5f375a86 - (int)((unsigned)__float_as_int(x.y) >> 1)));
#pragma unroll
    for (int it = 0; it < 3; ++it) y = __fmul2_rn(y, __ffma2_rn(nh, __fmul2_rn(y, y), splat(1.5f)));
    return y;
}

// Separations of a lane's two targets from one source (a cell's CoM or a
// leaf particle), and their squared distances in the order of dist2.
struct Sep2 {
    float2 dx, dy, dz, d2;
};

__device__ __forceinline__ Sep2 separation2(float sx, float sy, float sz, float2 nx, float2 ny, float2 nz)
{
    Sep2 s;
    s.dx = __fadd2_rn(splat(sx), nx);  // sx - x_i, formed as sx + (-x_i): the same rounding
    s.dy = __fadd2_rn(splat(sy), ny);
    s.dz = __fadd2_rn(splat(sz), nz);
    s.d2 = __ffma2_rn(s.dz, s.dz, __ffma2_rn(s.dy, s.dy, __fmul2_rn(s.dx, s.dx)));
    return s;
}

// add_term for both targets; a target with use == false adds a zero factor.
template <bool kFast, bool kNormal = false>
__device__ __forceinline__ void add_term2(const Sep2 &s, float m, bool use0, bool use1, float2 eps2,
                                          float2 &ax, float2 &ay, float2 &az)
{
    const float2 y = inv_sqrt2<kFast, kNormal>(__fadd2_rn(s.d2, eps2));
    const float2 fp = __fmul2_rn(__fmul2_rn(splat(m), y), __fmul2_rn(y, y));
    const float2 f = make_float2(use0 ? fp.x : 0.0f, use1 ? fp.y : 0.0f);
    ax = __ffma2_rn(f, s.dx, ax);
    ay = __ffma2_rn(f, s.dy, ay);
    az = __ffma2_rn(f, s.dz, az);
}


// Lane l of warp w holds sorted targets 64w + l and 64w + 32 + l. kLocal:
// nodes, first indices and leaf particles are read from the block's
// shared-memory copies (loc) instead of global memory.
template <bool kCount, bool kSelfFree, bool kFast, bool kLocal = false>
__device__ __forceinline__ void paired_walk(const WalkArgs &a, int num_nodes, float4 *stage,
                                            LocalTree loc = LocalTree{})
{
    constexpr unsigned kFull = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int base = a.t_begin + ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 64;
    const int t0 = base + lane, t1 = base + 32 + lane;
    const bool v0 = t0 < a.t_end, v1 = t1 < a.t_end;
    const float4 p0 = v0 ? __ldg(a.ps + t0) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4 p1 = v1 ? __ldg(a.ps + t1) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // negated positions: every separation is then one packed add
    const float2 nx = make_float2(-p0.x, -p1.x), ny = make_float2(-p0.y, -p1.y),
                 nz = make_float2(-p0.z, -p1.z);
    const float2 theta2 = splat(a.theta2), eps2 = splat(a.eps2);
    float2 ax = splat(0.0f), ay = splat(0.0f), az = splat(0.0f);
    uint32_t pc0 = 0, pc1 = 0, pp0 = 0, pp1 = 0;
    int next0 = v0 ? 0 : num_nodes, next1 = v1 ? 0 : num_nodes;
    int steps = 0;
    // k <= num_nodes: the record at num_nodes is a sentinel leaf that no
    // target accepts (side^2 = +inf, zero mass), so when every target is done
    // the group opens it, and the leaf branch ends the walk there
    for (;; ++steps) {  // ends: the node index strictly increases
        const int k = __reduce_min_sync(kFull, min(next0, next1));
        const int4 w = kLocal ? loc.nodes[k].w : __ldg(&a.wnode[k].w);
        const float4 c = kLocal ? loc.nodes[k].c : __ldg(&a.wnode[k].c);
        const bool act0 = next0 == k, act1 = next1 == k;
        const Sep2 s = separation2(c.x, c.y, c.z, nx, ny, nz);
        const float2 lim = __fmul2_rn(theta2, s.d2);
        const float s2 = __int_as_float(w.w);
        const bool acc0 = act0 && s2 < lim.x, acc1 = act1 && s2 < lim.y;
        // unconditional: nine steps in ten have an accepting target, and
        // skipping the rest costs more in branching than it saves
        add_term2<kFast, kSelfFree>(s, c.w, acc0, acc1, eps2, ax, ay, az);
        if (kCount) {
            pc0 += acc0;
            pc1 += acc1;
        }
        // a target that neither accepts nor waits opens k if it is a leaf;
        // the leaf test comes first: it is warp-uniform and skips the vote
        // at internal nodes
        const bool open0 = act0 && !acc0, open1 = act1 && !acc1;
        if (act0) next0 = acc0 ? w.x : w.y;
        if (act1) next1 = acc1 ? w.x : w.y;
        if (w.z != 0 && __any_sync(kFull, open0 || open1)) {
            if (k >= num_nodes) break;  // the sentinel
            const int first = kLocal ? loc.first[k] : __ldg(&a.meta[k].y), count = w.z;
            if (first < 0 || first > a.n - count) {  // warp-uniform consistency check
                if (lane == 0) atomicOr(&a.P->status, kStatusInternal);
                break;
            }
            if (kCount) {
                pp0 += open0 ? count - ((unsigned)(t0 - first) < (unsigned)count ? 1u : 0u) : 0u;
                pp1 += open1 ? count - ((unsigned)(t1 - first) < (unsigned)count ? 1u : 0u) : 0u;
            }
            if (kLocal && loc.ps) {  // the particles are in shared memory: read them as broadcasts
                const int self0 = t0 - first, self1 = t1 - first;
#pragma unroll 4
                for (int j = 0; j < count; ++j) {
                    const float4 q = loc.ps[first + j];
                    const Sep2 sj = separation2(q.x, q.y, q.z, nx, ny, nz);
                    add_term2<kFast, kSelfFree>(sj, q.w, open0 && (kSelfFree || j != self0),
                                                open1 && (kSelfFree || j != self1), eps2, ax, ay, az);
                }
                continue;
            }
            for (int b = 0; b < count; b += 32) {
                const int chunk = min(32, count - b);
                if (lane < chunk) stage[lane] = __ldg(a.ps + first + b + lane);
                __syncwarp();
                const int self0 = t0 - (first + b), self1 = t1 - (first + b);
#pragma unroll 4
                for (int j = 0; j < chunk; ++j) {
                    const float4 q = stage[j];
                    const Sep2 sj = separation2(q.x, q.y, q.z, nx, ny, nz);
                    add_term2<kFast, kSelfFree>(sj, q.w, open0 && (kSelfFree || j != self0),
                                     open1 && (kSelfFree || j != self1), eps2, ax, ay, az);
                }
                __syncwarp();
            }
        }
    }
    if (steps > num_nodes && lane == 0) atomicOr(&a.P->status, kStatusWalkBound);
    if (v0) store_target<kCount>(a, t0, ax.x, ay.x, az.x, pc0, pp0, steps);
    if (v1) store_target<kCount>(a, t1, ax.y, ay.y, az.y, pc1, pp1, steps);
}

template <bool kCount, bool kFast>
__global__ void __launch_bounds__(kThreads) k_walk_paired(WalkArgs a)
{
    __shared__ float4 s_leaf[kWarpsPerBlock][32];
    int num_nodes;
    bool self_free;
    if (!prologue<kFast>(a, num_nodes, self_free)) return;  // block-uniform
    float4 *stage = s_leaf[threadIdx.x >> 5];
    if (self_free)
        paired_walk<kCount, true, kFast>(a, num_nodes, stage);
    else
        paired_walk<kCount, false, kFast>(a, num_nodes, stage);
}

// Small and mid-size problems: too few warps to hide the latency of the L2
// reads every step makes (the node, a leaf's first index, its particles),
// which then sets the pace of the whole walk. Each block first copies into
// shared memory the nodes and the leaves' first indices and, when they fit
// too, all sorted particles (the node count is only known on the device, so
// the fit is decided there), then walks from there. Up to kLocalMaxTargets
// targets the blocks have kLocalThreads threads to spread the few warps over
// more SMs; up to kLocalWaveTargets (one block of kThreads per SM) they have
// kThreads, so one SM's warps share its L1 for the leaves read from global
// memory. Above that the plain kernel runs: enough warps to hide latency.
constexpr int kLocalThreads = 64;
constexpr int kLocalBytes = 200 * 1024;
constexpr int64_t kLocalMaxTargets = 16384;
constexpr int64_t kLocalMaxN = kLocalBytes / (int64_t)sizeof(float4);
constexpr int64_t kLocalWaveTargets = 152 * 2 * kThreads;
// Above about 40 000 particles the nodes of a leaf-32 tree no longer fit
// (about 0.13 nodes per particle, 36 bytes each), and a block that falls back
// to global memory with this much shared memory reserved was measured slower
// than the plain kernel (65 536 particles: 0.99 vs 0.82 ms).
constexpr int64_t kLocalMidMaxN = 40000;

// W = 64: the packed walk; W = 32 or 16: the one-target-per-lane walk.
template <int W, bool kCount, bool kSelfFree, bool kFast, bool kLocal>
__device__ __forceinline__ void any_walk(const WalkArgs &a, int num_nodes, float4 *stage, LocalTree loc)
{
    if constexpr (W == 64)
        paired_walk<kCount, kSelfFree, kFast, kLocal>(a, num_nodes, stage, loc);
    else
        coherent_walk<W, kCount, kSelfFree, false, kFast, kLocal>(a, num_nodes, stage, loc);
}

template <int kBlock, int W, bool kCount, bool kFast>
__global__ void __launch_bounds__(kBlock) k_walk_local(WalkArgs a)
{
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ float4 s_leaf[kBlock / 32][32];
    int num_nodes;
    bool self_free;
    if (!prologue<kFast>(a, num_nodes, self_free)) return;  // block-uniform
    // the node records with the sentinel, then the first indices
    const int64_t tree_bytes = ((int64_t)num_nodes + 1) * sizeof(WalkNode) + (int64_t)num_nodes * sizeof(int);
    const int64_t ps_offset = (tree_bytes + 15) & ~int64_t(15);
    const bool with_ps = ps_offset + (int64_t)a.n * (int64_t)sizeof(float4) <= kLocalBytes;  // block-uniform
    // the group's slots of the per-warp leaf stage (a half warp at W = 16)
    float4 *stage = &s_leaf[threadIdx.x >> 5][(threadIdx.x & 31) & ~((W < 32 ? W : 32) - 1)];
    if (tree_bytes > kLocalBytes) {  // block-uniform: walk from global memory
        if (self_free)
            any_walk<W, kCount, true, kFast, false>(a, num_nodes, stage, LocalTree{});
        else
            any_walk<W, kCount, false, kFast, false>(a, num_nodes, stage, LocalTree{});
        return;
    }
    WalkNode *nodes = reinterpret_cast<WalkNode *>(s_dyn);
    int *first = reinterpret_cast<int *>(nodes + num_nodes + 1);
    float4 *ps = with_ps ? reinterpret_cast<float4 *>(s_dyn + ps_offset) : nullptr;
    {
        const int4 *src = reinterpret_cast<const int4 *>(a.wnode);
        int4 *dst = reinterpret_cast<int4 *>(nodes);
        for (int i = threadIdx.x; i < 2 * (num_nodes + 1); i += kBlock) dst[i] = __ldg(src + i);
        for (int i = threadIdx.x; i < num_nodes; i += kBlock) first[i] = __ldg(&a.meta[i].y);
        if (with_ps)
            for (int i = threadIdx.x; i < a.n; i += kBlock) ps[i] = __ldg(a.ps + i);
    }
    __syncthreads();
    const LocalTree loc{nodes, first, ps};
    if (self_free)
        any_walk<W, kCount, true, kFast, true>(a, num_nodes, stage, loc);
    else
        any_walk<W, kCount, false, kFast, true>(a, num_nodes, stage, loc);
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
    const int t = a.t_begin + blockIdx.x * kThreads + threadIdx.x;
    const bool valid = t < a.t_end;
    const float4 xi = valid ? __ldg(a.ps + t) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float ax = 0.0f, ay = 0.0f, az = 0.0f;
    uint32_t pc = 0, pp = 0;
    int k = 0, steps = 0;
    for (; k < num_nodes; ++steps) {
        const int4 w = __ldg(&a.wnode[k].w);
        const float4 c = __ldg(&a.wnode[k].c);
        const float dx = __fsub_rn(c.x, xi.x);
        const float dy = __fsub_rn(c.y, xi.y);
        const float dz = __fsub_rn(c.z, xi.z);
        const float d2 = dist2(dx, dy, dz);
        const bool accept = __int_as_float(w.w) < __fmul_rn(a.theta2, d2);
        if (__all_sync(0xffffffffu, accept || !valid)) {
            if (valid) {
                add_term<kFast, kSelfFree>(dx, dy, dz, d2, c.w, a.eps2, ax, ay, az);
                if (kCount) ++pc;
            }
            k = w.x;
        } else if (w.z != 0) {
            const int first = __ldg(&a.meta[k].y), count = w.z;
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
                            particle_term<kFast, kSelfFree>(stage[j], xi, a.eps2, ax, ay, az);
                    } else {
                        const int self = t - (first + b);
                        for (int j = 0; j < chunk; ++j)
                            if (j != self) particle_term<kFast, kSelfFree>(stage[j], xi, a.eps2, ax, ay, az);
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
    const int t = a.t_begin + blockIdx.x * kThreads + threadIdx.x;
    if (t >= a.t_end) return;
    const float4 xi = __ldg(a.ps + t);
    const float2 nxy = make_float2(-xi.x, -xi.y);
    float2 axy = make_float2(0.0f, 0.0f);
    float az = 0.0f;
    uint32_t pc = 0, pp = 0;
    int k = 0, steps = 0;
    for (; k < num_nodes; ++steps) {
        const int4 w = __ldg(&a.wnode[k].w);
        const float4 c = __ldg(&a.wnode[k].c);
        const float2 dxy = __fadd2_rn(make_float2(c.x, c.y), nxy);
        const float dz = __fsub_rn(c.z, xi.z);
        const float d2 = dist2(dxy.x, dxy.y, dz);
        if (__int_as_float(w.w) < __fmul_rn(a.theta2, d2)) {
            add_term_xy<kFast, kSelfFree>(dxy, dz, d2, c.w, a.eps2, axy, az);
            if (kCount) ++pc;
            k = w.x;
        } else if (w.z != 0) {
            const int first = __ldg(&a.meta[k].y), count = w.z;
            if (first < 0 || first > a.n - count) {
                atomicOr(&a.P->status, kStatusInternal);
                break;
            }
            if (kCount) pp += count - ((unsigned)(t - first) < (unsigned)count ? 1u : 0u);
            for (int j = first; j < first + count; ++j)
                if (kSelfFree || j != t) particle_term_xy<kFast, kSelfFree>(__ldg(a.ps + j), nxy, xi.z, a.eps2, axy, az);
            k = w.x;
        } else {
            k = k + 1;
        }
    }
    if (k < num_nodes) atomicOr(&a.P->status, kStatusWalkBound);
    store_target<kCount>(a, t, axy.x, axy.y, az, pc, pp, steps);
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
    const int64_t targets = a.t_end - a.t_begin;
    // the shared-memory walks for small and mid-size problems (see above);
    // returns false when the plain kernels should run
    auto local = [&](auto wtag) -> bool {
        constexpr int W = decltype(wtag)::value;
        constexpr int per_thread = W == 64 ? 2 : 1;
        if (targets <= kLocalMaxTargets && a.n <= kLocalMaxN) {
            const unsigned g = ceil_div(targets, (int64_t)kLocalThreads * per_thread);
            if (count)
                k_walk_local<kLocalThreads, W, true, kFast><<<g, kLocalThreads, kLocalBytes, st>>>(a);
            else
                k_walk_local<kLocalThreads, W, false, kFast><<<g, kLocalThreads, kLocalBytes, st>>>(a);
            return true;
        }
        if (targets <= kLocalWaveTargets && a.n <= kLocalMidMaxN) {
            const unsigned g = ceil_div(targets, (int64_t)kThreads * per_thread);
            if (count)
                k_walk_local<kThreads, W, true, kFast><<<g, kThreads, kLocalBytes, st>>>(a);
            else
                k_walk_local<kThreads, W, false, kFast><<<g, kThreads, kLocalBytes, st>>>(a);
            return true;
        }
        return false;
    };
    auto coherent = [&](auto wtag) {
        constexpr int W = decltype(wtag)::value;
        if (local(wtag)) return;
        if (count)
            k_walk_coherent<W, true, false, kFast><<<grid, kThreads, 0, st>>>(a);
        else
            k_walk_coherent<W, false, false, kFast><<<grid, kThreads, 0, st>>>(a);
    };
    switch (traversal) {
    case 1: coherent(std::integral_constant<int, 32>{}); break;
    case 2: coherent(std::integral_constant<int, 16>{}); break;
    case 3: {
        if (local(std::integral_constant<int, 64>{})) break;
        const unsigned g = ceil_div(targets, (int64_t)kThreads * 2);  // 64 targets per warp
        if (count)
            k_walk_paired<true, kFast><<<g, kThreads, 0, st>>>(a);
        else
            k_walk_paired<false, kFast><<<g, kThreads, 0, st>>>(a);
        break;
    }
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

// The local walk's shared memory exceeds the default 48 KB: opted in once
// per device, outside any stream capture.
void prepare_walk()
{
    static std::atomic<bool> configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && configured[dev].load()) return;
    auto opt_in = [](const void *f) {
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kLocalBytes);
    };
    auto each = [&](auto btag, auto wtag) {
        constexpr int B = decltype(btag)::value, W = decltype(wtag)::value;
        opt_in((const void *)k_walk_local<B, W, true, true>);
        opt_in((const void *)k_walk_local<B, W, true, false>);
        opt_in((const void *)k_walk_local<B, W, false, true>);
        opt_in((const void *)k_walk_local<B, W, false, false>);
    };
    using L = std::integral_constant<int, kLocalThreads>;
    using T = std::integral_constant<int, kThreads>;
    each(L{}, std::integral_constant<int, 64>{});
    each(L{}, std::integral_constant<int, 32>{});
    each(L{}, std::integral_constant<int, 16>{});
    each(T{}, std::integral_constant<int, 64>{});
    each(T{}, std::integral_constant<int, 32>{});
    each(T{}, std::integral_constant<int, 16>{});
    if (dev >= 0 && dev < 64) configured[dev] = true;
}

void launch_walk(int traversal_flags, float theta, float eps, const uint32_t *perm,
                 const Buffers &b, int64_t t_begin, int64_t t_end, float *acc, uint32_t *inter,
                 uint32_t *visits, cudaStream_t st)
{
    if (t_end <= t_begin) return;  // no targets: nothing to launch
    const int traversal = traversal_flags & kTraversalMask;
    const bool fast = (traversal_flags & kFastTermFlag) != 0;
    const bool count = inter != nullptr || visits != nullptr;
    WalkArgs a;
    a.ps = b.ps;
    a.wnode = b.wnode;
    a.meta = b.meta;
    a.perm = perm;
    a.n = (int)b.n;
    a.t_begin = (int)t_begin;
    a.t_end = (int)t_end;
    a.theta2 = theta * theta;  // host binary32 products, round to nearest
    a.eps2 = eps * eps;
    a.P = b.params;
    a.acc = acc;
    a.inter = inter;
    a.visits = visits;
    const unsigned grid = ceil_div(t_end - t_begin, kThreads);
    prepare_walk();
    if (fast)
        launch_kernels<true>(traversal, count, grid, a, st);
    else
        launch_kernels<false>(traversal, count, grid, a, st);
    g_launches += 1;
}

}  // namespace obh
