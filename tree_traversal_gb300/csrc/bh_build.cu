// bh_build.cu -- a5 octree build from sorted Morton keys and a6 upward
// monopole moments.
//
// Tree definition (orrery: "sycl_tree_solver.hpp", "Where the tree comes
// from"; ADR-0029, Decision; the workload's "split any cell above leaf
// capacity"): a cell of level L is the run of sorted keys sharing their top L
// octant digits. The root is a node; any other cell is a node iff its parent
// cell holds more than leaf_cap particles (and so do all its ancestors,
// since counts only grow upwards). A node is a leaf iff it holds at most
// leaf_cap particles or its level is 21. Nodes are stored in depth-first
// preorder with the escape index of each node = first node after its subtree.
//
// The build is flat rather than recursive. Two observations make it so:
//  * in preorder, nodes are ordered by (first particle, level), so the index
//    of a node is (nodes starting at earlier positions) + (its rank among
//    the nested nodes that start at the same position): one exclusive scan of
//    a per-position node count;
//  * the nodes starting at position i are the cells of levels D+1 .. L_last,
//    where D is the number of levels key[i-1] and key[i] share, provided the
//    level-D cell around them is over capacity; the chain stops at the first
//    level whose cell does not contain key[i + leaf_cap] (or at level 21).
// escape(node) = scan value at the first position past the node's range.
#include <cfloat>

#include <cuda/atomic>

#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;

// The child table: for every node, its children's indices by octant (-1
// where the octant holds no child), so that the moments climb reads a
// node's children at once instead of following their escape indices one by
// one. It takes 32 bytes per node and lives in the radix key buffer the
// sort did not leave its result in (8 bytes per particle), so it is used
// when the tree has at most n / 4 nodes (a leaf capacity of 32 gives about
// n / 8); larger trees climb by the escape indices.
__device__ __forceinline__ bool child_table_fits(int64_t nodes, int64_t n) { return 4 * nodes <= n; }

// Per position: D (levels shared with the previous key), the number of
// nodes starting here (from D and W, the levels shared with the key leaf_cap
// ahead), and the start of the parent cell of the first of them.
__global__ void __launch_bounds__(kThreads)
k_build_levels(const uint64_t *__restrict__ K, int64_t n, int32_t cap,
               int8_t *__restrict__ lev_d,
               uint8_t *__restrict__ ncount, int32_t *__restrict__ pstart, const int *status)
{
    if (*status & kStatusInternal) return;  // the keys are not sorted: build nothing
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i > n) return;
    if (i == n) {  // the scan runs over n + 1 entries; the last contributes 0
        ncount[n] = 0;
        return;
    }
    const uint64_t key = K[i];
    const int D = (i == 0) ? -1 : common_levels(K[i - 1], key);
    const int W = (i + cap < n) ? common_levels(key, K[i + cap]) : -1;
    int cnt = 0;
    int64_t s = 0;
    if (i == 0) {
        cnt = (W < 0) ? 1 : min(kLevels, W + 1) + 1;  // levels 0 .. L_last
    } else if (D < kLevels) {
        // start of the level-D cell holding key[i-1] and key[i]: the first
        // position whose key is >= key with its low 3(21-D) bits cleared
        const uint64_t prefix = key & ~((1ull << (3 * (kLevels - D))) - 1ull);
        uint32_t lo = 0, hi = (uint32_t)i;  // n < 2^31: 32-bit indices (fewer instructions per step)
        while (lo < hi) {
            const uint32_t mid = (lo + hi) >> 1;
            if (K[mid] < prefix)
                lo = mid + 1;
            else
                hi = mid;
        }
        s = lo;
        const int Ws = (s + cap < n) ? common_levels(K[s], K[s + cap]) : -1;
        if (Ws >= D) cnt = min(kLevels, max(D + 1, W + 1)) - D;  // parent over capacity
    }
    lev_d[i] = (int8_t)D;
    ncount[i] = (uint8_t)cnt;
    pstart[i] = (int32_t)s;
}

// Writes the nodes that start at each position: their first particle and
// level, and the parent index (the first node's parent is the level-D cell
// found by k_build_levels, every later one's is the node before it: the
// cells starting at one position are nested). The cells' ends come from
// k_build_ends, one node per thread, so no thread walks a chain of searches.
// A thread takes four consecutive positions and reads each per-position
// array with one load (4 bytes of counts, 4 of levels, 16 of scan values and
// of parent-cell starts), then the parent cells' entries of all four at once:
// two rounds of independent loads instead of a chain per position.
constexpr int kEmitPositions = 4;

__global__ void __launch_bounds__(kThreads)
k_build_emit(int64_t n, const int8_t *__restrict__ lev_d, const uint8_t *__restrict__ ncount,
             const int32_t *__restrict__ pstart, const uint32_t *__restrict__ node_start,
             int64_t max_nodes, int4 *__restrict__ meta, int32_t *__restrict__ parent,
             int4 *__restrict__ ctab, DeviceParams *P)
{
    // warp-uniform exit (the warp's lanes meet in a reduction below)
    if (__shfl_sync(0xffffffffu, P->status, 0) & kStatusInternal) return;
    const int64_t i0 = kEmitPositions * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
    const uint32_t total = node_start[n];
    if (i0 == 0) {
        P->num_nodes = (int)total;
        if ((int64_t)total > max_nodes) atomicOr(&P->status, kStatusNodeBound);
    }
    int cnt[kEmitPositions] = {}, D[kEmitPositions] = {}, s[kEmitPositions] = {};
    uint32_t base[kEmitPositions] = {};
    if (i0 < n && (int64_t)total <= max_nodes) {
        if (i0 + kEmitPositions <= n) {  // the buffers are 256-byte aligned, i0 a multiple of 4
            const uint32_t c4 = *reinterpret_cast<const uint32_t *>(ncount + i0);
            const uint32_t d4 = *reinterpret_cast<const uint32_t *>(lev_d + i0);
            const uint4 b4 = *reinterpret_cast<const uint4 *>(node_start + i0);
            const int4 s4 = *reinterpret_cast<const int4 *>(pstart + i0);
#pragma unroll
            for (int j = 0; j < kEmitPositions; ++j) {
                cnt[j] = (int)((c4 >> (8 * j)) & 0xffu);
                D[j] = (int)(int8_t)((d4 >> (8 * j)) & 0xffu);
            }
            base[0] = b4.x; base[1] = b4.y; base[2] = b4.z; base[3] = b4.w;
            s[0] = s4.x; s[1] = s4.y; s[2] = s4.z; s[3] = s4.w;
        } else {
            for (int j = 0; j < kEmitPositions && i0 + j < n; ++j) {
                cnt[j] = ncount[i0 + j];
                D[j] = lev_d[i0 + j];
                base[j] = node_start[i0 + j];
                s[j] = pstart[i0 + j];
            }
        }
    }
    // the parent cell of each position's first node: its first node and level
    int s_level[kEmitPositions] = {};
    uint32_t s_base[kEmitPositions] = {};
#pragma unroll
    for (int j = 0; j < kEmitPositions; ++j) {
        if (cnt[j] > 0 && i0 + j > 0) {
            s_level[j] = (s[j] == 0) ? 0 : lev_d[s[j]] + 1;
            s_base[j] = node_start[s[j]];
        }
    }
    const bool table = child_table_fits(total, n);
    int deepest = -1;  // the deepest node of these positions, for the tree depth
#pragma unroll
    for (int j = 0; j < kEmitPositions; ++j) {
        if (cnt[j] == 0) continue;
        const int64_t i = i0 + j;
        const int first_level = (i == 0) ? 0 : D[j] + 1;
        int32_t par = -1;
        if (i > 0) {
            par = (int32_t)(s_base[j] + (uint32_t)(D[j] - s_level[j]));
            if (par < 0 || par >= (int32_t)base[j]) {  // a parent precedes its children
                atomicOr(&P->status, kStatusInternal);
                continue;
            }
        }
        for (int l = 0; l < cnt[j]; ++l) {
            const int64_t k = (int64_t)base[j] + l;
            meta[k] = make_int4(0, (int)i, 0, first_level + l);  // escape and count: k_build_ends
            parent[k] = par;
            if (table) {  // no children yet: k_build_ends enters them
                ctab[2 * k] = make_int4(-1, -1, -1, -1);
                ctab[2 * k + 1] = make_int4(-1, -1, -1, -1);
            }
            par = (int32_t)k;
        }
        deepest = max(deepest, first_level + cnt[j] - 1);
    }
    // one atomic per warp for the depth, not one per node-starting position
    deepest = __reduce_max_sync(0xffffffffu, deepest);
    if ((threadIdx.x & 31) == 0 && deepest >= 0) atomicMax(&P->depth, deepest);
}

__device__ __forceinline__ void node_end(const uint64_t *__restrict__ K, int64_t n,
                                         const uint32_t *__restrict__ node_start, int64_t total,
                                         int32_t leaf_cap, int4 *__restrict__ meta,
                                         WalkNode *__restrict__ wnode, int32_t *__restrict__ arrive,
                                         const int32_t *__restrict__ parent, int32_t *__restrict__ ctab,
                                         DeviceParams *P, int64_t k)
{
    const int4 m = meta[k];
    const int64_t i = m.y;
    const int L = m.w;
    if (i < 0 || i >= n || L < 0 || L > kLevels) {
        atomicOr(&P->status, kStatusInternal);
        return;
    }
    int64_t end = n;
    if (L > 0) {
        const uint64_t upper = K[i] | ((1ull << (3 * (kLevels - L))) - 1ull);
        uint32_t lo = (uint32_t)i + 1, hi = (uint32_t)n;  // n < 2^31: 32-bit indices
        while (lo < hi) {
            const uint32_t mid = (lo + hi) >> 1;
            if (K[mid] <= upper)
                lo = mid + 1;
            else
                hi = mid;
        }
        end = lo;
    }
    int esc = (int)node_start[end];
    if (!(esc > k && esc <= total)) {
        atomicOr(&P->status, kStatusInternal);
        esc = (int)total;
    }
    const int count = (int)(end - i);
    const bool leaf = count <= leaf_cap || L == kLevels;
    meta[k] = make_int4(esc, (int)i, count, L);
    arrive[k] = 0;
    // this node in its parent's row of the child table, under its octant
    // (the parent's cell split by the level-L digit; children in key order
    // are children in octant order)
    if (ctab && L > 0) {
        const int32_t par = parent[k];
        if (par >= 0 && par < k) ctab[8 * (int64_t)par + (int)((K[i] >> (3 * (kLevels - L))) & 7u)] = (int32_t)k;
    }
    wnode[k].w = make_int4(esc, leaf ? esc : (int)k + 1, leaf ? count : 0, __float_as_int(P->s2[L]));
}

// One thread per node (a grid-stride loop over the node count the scan
// produced, so the grid follows the tree rather than its bound): the end of
// its cell (the first position past the keys that share the node's top L
// octal digits; a binary search over the sorted keys), hence its particle
// count and escape index (the node index at that position), and the node's
// walk record {escape, the node a target that does not accept it goes to
// next (escape for a leaf, which it opens; k + 1 for an internal node, which
// it enters), leaf count (0 for an internal node), bits of (side
// 2^-level)^2}. Every node k < num_nodes gets its record here, and every
// record's next nodes are checked to lie in (k, num_nodes]: so a walk's node
// index strictly increases and every walk ends within num_nodes steps (an
// escape outside that range is flagged and replaced by num_nodes). The
// node's arrival count for the moments climb is cleared here too.
__global__ void __launch_bounds__(kThreads)
k_build_ends(const uint64_t *__restrict__ K, int64_t n, const uint32_t *__restrict__ node_start,
             int64_t max_nodes, int32_t leaf_cap, int4 *__restrict__ meta,
             WalkNode *__restrict__ wnode, int32_t *__restrict__ arrive,
             const int32_t *__restrict__ parent, int32_t *__restrict__ ctab, DeviceParams *P)
{
    if (P->status & kStatusInternal) return;
    const int64_t total = node_start[n];
    if (total > max_nodes) return;
    const int64_t first_k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (first_k == 0) {
        // a sentinel after the last node: a leaf no target accepts (side^2 =
        // +inf) with zero mass, where the packed walk's group ends
        wnode[total].w = make_int4((int)total, (int)total, 1, 0x7f800000);
        wnode[total].c = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    int32_t *table = child_table_fits(total, n) ? ctab : nullptr;
    for (int64_t k = first_k; k < total; k += (int64_t)gridDim.x * blockDim.x)
        node_end(K, n, node_start, total, leaf_cap, meta, wnode, arrive, parent, table, P, k);
}
// A node whose mass is not finite or whose CoM lies at 2^126 or beyond is
// reported as non-finite: with every coordinate below 2^125 (checked with the
// bounding box), every separation the walks form is then a finite number.
__device__ __forceinline__ float4 store_moments(int64_t k, float sx, float sy, float sz, float M,
                                                float4 *sums, DeviceParams *P)
{
    __stcg(sums + k, make_float4(sx, sy, sz, M));
    float4 c = make_float4(0.0f, 0.0f, 0.0f, M);
    if (M > 0.0f) {
        c.x = __fdiv_rn(sx, M);
        c.y = __fdiv_rn(sy, M);
        c.z = __fdiv_rn(sz, M);
    }
    const float lim = 0x1p126f;
    if (!(fabsf(M) <= FLT_MAX && fabsf(c.x) < lim && fabsf(c.y) < lim && fabsf(c.z) < lim))
        atomicOr((int *)&P->status, kStatusNonFinite);
    return c;
}

// Stores a node's moments: its sums, and {CoM, M} in its walk record (the
// rest of the record comes from k_build_ends).
__device__ __forceinline__ void store_node(int64_t k, float sx, float sy, float sz, float M,
                                           float4 *sums, WalkNode *wnode, DeviceParams *P)
{
    wnode[k].c = store_moments(k, sx, sy, sz, M, sums, P);
}

// a6: one thread per leaf (a grid-stride loop over the nodes) sums its
// particles in sorted order, then climbs: each child adds its particle count
// to its parent's arrival count, and the child that completes it (the
// children's ranges partition the parent's, so their counts add up to the
// parent's) sums all of the parent's children in child order. No thread
// ever waits for another.
__device__ __forceinline__ void leaf_and_climb(const float4 *__restrict__ ps, int64_t n,
                                               const int4 *__restrict__ meta,
                                               const int32_t *__restrict__ parent,
                                               int32_t *__restrict__ arrive, float4 *sums,
                                               WalkNode *__restrict__ wnode,
                                               const int4 *__restrict__ ctab, DeviceParams *P,
                                               int total, int64_t k, int4 m)
{
    if (m.y < 0 || m.z < 0 || (int64_t)m.y + m.z > n) {
        atomicOr((int *)&P->status, kStatusInternal);
        return;
    }
    float M = 0.0f, sx = 0.0f, sy = 0.0f, sz = 0.0f;
    const float4 *src = ps + m.y;
    int j = 0;
    // four loads in flight, then the additions in order
    for (; j + 4 <= m.z; j += 4) {
        float4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = __ldg(src + j + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            M = __fadd_rn(M, q[u].w);
            sx = __fmaf_rn(q[u].w, q[u].x, sx);
            sy = __fmaf_rn(q[u].w, q[u].y, sy);
            sz = __fmaf_rn(q[u].w, q[u].z, sz);
        }
    }
    for (; j < m.z; ++j) {
        const float4 q = __ldg(src + j);
        M = __fadd_rn(M, q.w);
        sx = __fmaf_rn(q.w, q.x, sx);
        sy = __fmaf_rn(q.w, q.y, sy);
        sz = __fmaf_rn(q.w, q.z, sz);
    }
    store_node(k, sx, sy, sz, M, sums, wnode, P);
    int carried = m.z;
    int64_t node = parent[k];
    while (node >= 0) {
        // release: this child's sums before the count; acquire: the child
        // that completes the count sees every sibling's sums
        cuda::atomic_ref<int32_t, cuda::thread_scope_device> count(arrive[node]);
        const int prev = count.fetch_add(carried, cuda::std::memory_order_acq_rel);
        const int4 pm = meta[node];
        if (prev + carried != pm.z) return;
        const int esc = pm.x;
        M = sx = sy = sz = 0.0f;
        if (esc > total) {
            atomicOr((int *)&P->status, kStatusInternal);
            return;
        }
        if (ctab) {  // the children by octant, read at once, summed in octant order
            const int4 lo = ctab[2 * node], hi = ctab[2 * node + 1];
            const int ch[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            float4 cs[8];
#pragma unroll
            for (int o = 0; o < 8; ++o) {
                const bool in = ch[o] > node && ch[o] < esc;  // a child lies inside its parent's range
                if (ch[o] >= 0 && !in) {
                    atomicOr((int *)&P->status, kStatusInternal);
                    return;
                }
                cs[o] = in ? __ldcg(sums + ch[o]) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int o = 0; o < 8; ++o) {
                if (ch[o] < 0) continue;
                M = __fadd_rn(M, cs[o].w);
                sx = __fadd_rn(sx, cs[o].x);
                sy = __fadd_rn(sy, cs[o].y);
                sz = __fadd_rn(sz, cs[o].z);
            }
            store_node(node, sx, sy, sz, M, sums, wnode, P);
            carried = pm.z;
            node = parent[node];
            continue;
        }
        for (int c = (int)node + 1; c < esc;) {
            const float4 s = __ldcg(sums + c);
            M = __fadd_rn(M, s.w);
            sx = __fadd_rn(sx, s.x);
            sy = __fadd_rn(sy, s.y);
            sz = __fadd_rn(sz, s.z);
            const int nc = meta[c].x;
            if (nc <= c) {  // escapes strictly increase; stop rather than loop
                atomicOr((int *)&P->status, kStatusInternal);
                return;
            }
            c = nc;
        }
        store_node(node, sx, sy, sz, M, sums, wnode, P);
        carried = pm.z;
        node = parent[node];
    }
}

__global__ void __launch_bounds__(kThreads)
k_moments(const float4 *__restrict__ ps, int64_t n, int32_t leaf_cap,
          const int4 *__restrict__ meta, const int32_t *__restrict__ parent,
          int32_t *__restrict__ arrive, float4 *sums, WalkNode *__restrict__ wnode,
          const int4 *__restrict__ ctab, DeviceParams *P)
{
    if (P->status & (kStatusNodeBound | kStatusInternal)) return;
    const int total = P->num_nodes;
    const int4 *table = child_table_fits(total, n) ? ctab : nullptr;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int4 m = meta[k];
        if (m.z <= leaf_cap || m.w == kLevels)  // a leaf
            leaf_and_climb(ps, n, meta, parent, arrive, sums, wnode, table, P, total, k, m);
    }
}

}  // namespace

// Grid of the kernels that loop over the nodes: the node count is only
// known on the device, so they stride over it with at most a few waves of
// blocks (and no more blocks than the bound needs).
static unsigned node_grid(const Buffers &b)
{
    const unsigned want = ceil_div(b.max_nodes, kThreads);
    return want < 152u * 8u ? want : 152u * 8u;
}

// The child table's storage: the radix key buffer that does not hold the
// sorted keys (free once the sort is done).
static void *child_table(const uint64_t *keys_sorted, const Buffers &b)
{
    return keys_sorted == b.keys_a ? (void *)b.keys_b : (void *)b.keys_a;
}

void launch_build(const uint64_t *keys_sorted, int32_t leaf_cap, const Buffers &b,
                  cudaStream_t st)
{
    int4 *ctab = (int4 *)child_table(keys_sorted, b);
    k_build_levels<<<ceil_div(b.n + 1, kThreads), kThreads, 0, st>>>(
        keys_sorted, b.n, leaf_cap, b.lev_d, b.ncount, b.pstart, &b.params->status);
    g_launches += 1;
    // node_start = exclusive scan of ncount over n + 1 entries
    launch_scan_u8(b.ncount, b.node_start, b.n + 1, b.scan_partial, st);
    k_build_emit<<<ceil_div(b.n, (int64_t)kThreads * kEmitPositions), kThreads, 0, st>>>(
        b.n, b.lev_d, b.ncount, b.pstart, b.node_start, b.max_nodes, b.meta, b.parent, ctab, b.params);
    k_build_ends<<<node_grid(b), kThreads, 0, st>>>(keys_sorted, b.n, b.node_start, b.max_nodes,
                                                   leaf_cap, b.meta, b.wnode, b.arrive, b.parent,
                                                   (int32_t *)ctab, b.params);
    g_launches += 2;
}

void launch_moments(const uint64_t *keys_sorted, int32_t leaf_cap, const Buffers &b, cudaStream_t st)
{
    k_moments<<<node_grid(b), kThreads, 0, st>>>(b.ps, b.n, leaf_cap, b.meta, b.parent, b.arrive,
                                                b.sums, b.wnode, (const int4 *)child_table(keys_sorted, b),
                                                b.params);
    g_launches += 1;
}

}  // namespace obh
