// bh_common.cuh -- types and helpers shared by the CUDA translation units of
// the Barnes-Hut library (never by the oracle).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace obh {

constexpr int kLevels = 21;          // bits per axis; deepest octree level

// The traversal argument: the low byte selects the walk, a flag bit the fast
// force term (see include/orrery_bh.h).
constexpr int kTraversalMask = 0xff;
constexpr int kFastTermFlag = 0x100;

// Bits of the device status word.
constexpr int kStatusNonFinite = 1;  // a position or mass is not finite
constexpr int kStatusWalkBound = 2;  // a walk hit its iteration bound
constexpr int kStatusNodeBound = 4;  // more nodes than the workspace holds
constexpr int kStatusInternal = 8;   // an index failed a consistency check (access skipped)

// Per-evaluation parameters that the device computes for itself.
struct DeviceParams {
    float lo[3];
    float side;
    float inv;
    float s2[kLevels + 1];  // (side * 2^-L)^2 for L = 0..21
    float mmax;             // largest |m|: bounds the self term (see the walk)
    int status;
    int num_nodes;
    int depth;
};

// Device pointers carved out of one workspace allocation.
// One node as the walks read it: 32 bytes, one sector, so a step's two
// 16-byte loads touch one cache line. w = {escape, next node when not
// accepted (escape for a leaf, k + 1 otherwise), leaf count or 0, bits of the
// node's squared side}; c = {CoM_x, CoM_y, CoM_z, M}. A leaf's first particle
// is read from the node table (meta) when the leaf is opened.
struct alignas(32) WalkNode {
    int4 w;
    float4 c;
};

struct Buffers {
    int64_t n;
    int64_t max_nodes;
    int bbox_blocks;
    // a1
    float *bbox_partial;      // [bbox_blocks][8]
    DeviceParams *params;
    // a2, a3
    uint64_t *keys_a, *keys_b;
    uint32_t *idx_a, *idx_b;
    uint32_t *sort_ctl;       // [sort_ctl_words()] digit counts of every pass, tile tickets
    uint32_t *sort_look;      // look-back words of alternate passes, [2][tiles][512]
    // a4
    float4 *ps;               // sorted {x, y, z, m}
    // a5
    int8_t *lev_d;            // common levels with the previous key (-1 at 0)
    uint8_t *ncount;          // nodes starting at each position
    int32_t *pstart;          // start of the parent cell of the first node at i
    uint32_t *node_start;     // [n + 1] exclusive scan of ncount
    uint32_t *scan_partial;   // scan block sums
    int4 *meta;               // [max_nodes] {escape, first, count, level}
    int32_t *parent;          // [max_nodes]
    int32_t *arrive;          // [max_nodes] particles of the children summed so far (moments)
    // a6
    float4 *sums;             // [max_nodes] {S_x, S_y, S_z, M}
    WalkNode *wnode;          // [max_nodes + 1] everything a walk step reads of a node, then a sentinel
};

// The node bound of n particles at leaf capacity cap: the most nodes a tree
// can have (n leaves' worth of cells plus a chain of single-child cells of
// length up to 21 above every cap + 1 particles), plus one.
int64_t node_bound(int64_t n, int32_t cap);
// Lays the buffers of one evaluation of n particles and up to `nodes` nodes
// out over `base` (nullptr: computes the size only); returns the bytes used.
size_t carve(Buffers &b, char *base, int64_t n, int64_t nodes);

// Kernel-launch counter (every launch site increments it).
extern std::atomic<uint64_t> g_launches;

// --- launchers, one per phase (all enqueue on `st`) ----------------------
void launch_bbox(const float *pos, const float *mass, const Buffers &b, cudaStream_t st);
void launch_morton(const float *pos, const Buffers &b, cudaStream_t st);
void launch_sort(const Buffers &b, cudaStream_t st, uint64_t **keys_sorted, uint32_t **perm);
void launch_gather(const float *pos, const float *mass, const uint32_t *perm, const Buffers &b,
                   cudaStream_t st);
void launch_build(const uint64_t *keys_sorted, int32_t leaf_cap, const Buffers &b,
                  cudaStream_t st);
// keys_sorted: the buffer launch_sort left the keys in (the other one holds
// the moments' child table).
void launch_moments(const uint64_t *keys_sorted, int32_t leaf_cap, const Buffers &b,
                    cudaStream_t st);
// a7 with the a8 scatter fused: results land in the caller's order. Walks
// the sorted targets [t_begin, t_end) against the whole tree.
void launch_walk(int traversal, float theta, float eps, const uint32_t *perm, const Buffers &b,
                 int64_t t_begin, int64_t t_end, float *acc, uint32_t *inter, uint32_t *visits,
                 cudaStream_t st);
void launch_direct(const float *pos, const float *mass, int64_t n, float eps, float *acc,
                   int *status, cudaStream_t st);
void launch_scan_u8(const uint8_t *in, uint32_t *out, int64_t count, uint32_t *partial,
                    cudaStream_t st);
int64_t scan_partial_count(int64_t count);
int64_t sort_look_words(int64_t n);  // both look-back arrays
int sort_ctl_words();  // cleared by launch_bbox at the start of every evaluation
unsigned *bbox_ticket(const Buffers &b);  // the last of them: the bounding box's fold ticket
void prepare_sort();  // sets the sort kernels' function attributes on this device
void prepare_walk();  // sets the walk kernels' function attributes on this device

// --- small device helpers -------------------------------------------------
// Number of leading 3-bit groups (levels) two 63-bit keys share: 0..21.
__device__ __forceinline__ int common_levels(uint64_t a, uint64_t b)
{
    uint64_t x = a ^ b;
    if (x == 0) return kLevels;
    int msb = 63 - __clzll((long long)x);
    return (kLevels - 1) - msb / 3;
}

inline unsigned ceil_div(int64_t a, int64_t b) { return (unsigned)((a + b - 1) / b); }

}  // namespace obh
