// bh_prep.cu -- the data-movement phases before the tree: bounding cube,
// gather into tree order, and a device-wide exclusive scan used by the
// build. (The Morton keys are made in bh_sort.cu, together with the digit
// counts of their sort; the scatter back to the caller's order is fused into
// the walk's epilogue.)
//
// Pages: "sycl_tree_solver.hpp" (Detailed Description, "Where the tree comes
// from": particles are copied into the tree's sorted order before the walk
// and the accelerations scattered back to the caller's order afterwards).
// The bounding cube follows the workload definition that accompanies the
// pages (a quantised bounding cube, 21 bits per axis).
#include <math.h>

#include "bh_common.cuh"

namespace obh {

std::atomic<uint64_t> g_launches{0};

namespace {

constexpr int kBBoxThreads = 256;

__device__ __forceinline__ void warp_minmax(float &lo, float &hi)
{
    for (int off = 16; off > 0; off >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
}

// Folds one value set per thread over the block; thread 0 writes
// {lo[3], hi[3], bad, mmax} to out.
__device__ __forceinline__ void block_fold(float lo[3], float hi[3], float mmax, int bad, float *out)
{
    __shared__ float s_lo[3][kBBoxThreads / 32], s_hi[3][kBBoxThreads / 32];
    __shared__ float s_m[kBBoxThreads / 32];
    __shared__ int s_bad[kBBoxThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int a = 0; a < 3; ++a) warp_minmax(lo[a], hi[a]);
    for (int off = 16; off > 0; off >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, off));
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        for (int a = 0; a < 3; ++a) {
            s_lo[a][warp] = lo[a];
            s_hi[a][warp] = hi[a];
        }
        s_m[warp] = mmax;
        s_bad[warp] = bad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kBBoxThreads / 32; ++w) {
            for (int a = 0; a < 3; ++a) {
                lo[a] = fminf(lo[a], s_lo[a][w]);
                hi[a] = fmaxf(hi[a], s_hi[a][w]);
            }
            mmax = fmaxf(mmax, s_m[w]);
            bad |= s_bad[w];
        }
        for (int a = 0; a < 3; ++a) {
            out[a] = lo[a];
            out[3 + a] = hi[a];
        }
        out[6] = bad ? 1.0f : 0.0f;
        out[7] = mmax;
    }
}

// Adds particle {x, y, z} of mass m to a thread's running extent.
__device__ __forceinline__ void extend(float x, float y, float z, float m, float lo[3], float hi[3],
                                       float &mmax, int &bad)
{
    const float v[3] = {x, y, z};
    bad |= !isfinite(m);
    mmax = fmaxf(mmax, fabsf(m));
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        bad |= !(fabsf(v[a]) < 0x1p125f);  // non-finite, or beyond the supported range
        lo[a] = fminf(lo[a], v[a]);
        hi[a] = fmaxf(hi[a], v[a]);
    }
}

// a1: per-block min / max per axis, max |m| and a non-finite flag, then the
// last block to finish folds all blocks' partials and derives the cube:
// side = max_a (hi_a - lo_a), inv = 2^21 / side, and the per-level squared
// cell side s2[L] = (side * side) * 2^(-2L) (an exact power-of-two scaling).
// It also resets the status word, node count and depth of this evaluation.
// A thread reads four particles at a time with 16-byte loads when the
// arrays allow it. ticket: zero on entry (cleared with the sort's control
// words before the launch).
__global__ void __launch_bounds__(kBBoxThreads)
k_bbox(const float *__restrict__ pos, const float *__restrict__ mass, int64_t n,
       float *__restrict__ partial, unsigned *ticket, DeviceParams *P)
{
    float lo[3] = {INFINITY, INFINITY, INFINITY};
    float hi[3] = {-INFINITY, -INFINITY, -INFINITY};
    float mmax = 0.0f;
    int bad = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool vec = ((reinterpret_cast<uintptr_t>(pos) | reinterpret_cast<uintptr_t>(mass)) & 15u) == 0;
    int64_t done = 0;  // particles covered by the four-at-a-time loop
    if (vec) {
        const float4 *p4 = reinterpret_cast<const float4 *>(pos);
        const float4 *m4 = reinterpret_cast<const float4 *>(mass);
        const int64_t quads = n / 4;
        for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += stride) {
            const float4 a = __ldg(p4 + 3 * q), b = __ldg(p4 + 3 * q + 1), c = __ldg(p4 + 3 * q + 2);
            const float4 m = __ldg(m4 + q);
            extend(a.x, a.y, a.z, m.x, lo, hi, mmax, bad);
            extend(a.w, b.x, b.y, m.y, lo, hi, mmax, bad);
            extend(b.z, b.w, c.x, m.z, lo, hi, mmax, bad);
            extend(c.y, c.z, c.w, m.w, lo, hi, mmax, bad);
        }
        done = 4 * quads;
    }
    for (int64_t i = done + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        extend(__ldg(pos + 3 * i), __ldg(pos + 3 * i + 1), __ldg(pos + 3 * i + 2), __ldg(mass + i), lo, hi,
               mmax, bad);
    block_fold(lo, hi, mmax, bad, partial + 8 * blockIdx.x);

    // the last block: fold the partials (they were written before each
    // block's ticket, and are read past L1)
    __shared__ bool s_last;
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    __shared__ float s_out[8];
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        lo[a] = INFINITY;
        hi[a] = -INFINITY;
    }
    mmax = 0.0f;
    bad = 0;
    for (int b = threadIdx.x; b < (int)gridDim.x; b += blockDim.x) {
        const float *o = partial + 8 * b;
        for (int a = 0; a < 3; ++a) {
            lo[a] = fminf(lo[a], __ldcg(o + a));
            hi[a] = fmaxf(hi[a], __ldcg(o + 3 + a));
        }
        bad |= (__ldcg(o + 6) != 0.0f);
        mmax = fmaxf(mmax, __ldcg(o + 7));
    }
    block_fold(lo, hi, mmax, bad, s_out);
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int a = 0; a < 3; ++a) {
        lo[a] = s_out[a];
        hi[a] = s_out[3 + a];
    }
    bad = s_out[6] != 0.0f;
    P->mmax = s_out[7];
    float side = 0.0f;
    for (int a = 0; a < 3; ++a) {
        float ext = __fsub_rn(hi[a], lo[a]);
        if (ext > side) side = ext;
        P->lo[a] = lo[a];
    }
    P->side = side;
    P->inv = (side > 0.0f) ? __fdiv_rn(2097152.0f, side) : 0.0f;
    float s2 = __fmul_rn(side, side);
    for (int L = 0; L <= kLevels; ++L) P->s2[L] = __fmul_rn(s2, ldexpf(1.0f, -2 * L));
    P->status = bad ? kStatusNonFinite : 0;
    P->num_nodes = 0;
    P->depth = 0;
}

// a4: sorted particles {x, y, z, m}. (Four slots per thread, with the
// sixteen gathers issued together, measured the same: the gather is bound by
// its traffic, not by load latency.)
__global__ void __launch_bounds__(256)
k_gather(const float *__restrict__ pos, const float *__restrict__ mass,
         const uint32_t *__restrict__ perm, int64_t n, float4 *__restrict__ ps, int *status)
{
    int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n || (*status & kStatusInternal)) return;  // no permutation to follow
    uint32_t i = __ldg(perm + k);
    if (i >= (uint64_t)n) {
        atomicOr(status, kStatusInternal);
        return;
    }
    ps[k] = make_float4(__ldg(pos + 3 * (int64_t)i), __ldg(pos + 3 * (int64_t)i + 1),
                        __ldg(pos + 3 * (int64_t)i + 2), __ldg(mass + i));
}

// ---- exclusive scan into uint32 (three launches, no inter-block waiting) ----
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

// Block-wide exclusive scan of one value per thread; returns the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t &total)
{
    __shared__ uint32_t s_warp[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = (lane < kScanThreads / 32) ? s_warp[lane] : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        if (lane < kScanThreads / 32) s_warp[lane] = w;
    }
    __syncthreads();
    uint32_t before = (warp > 0) ? s_warp[warp - 1] : 0u;
    total = s_warp[kScanThreads / 32 - 1];
    __syncthreads();
    return before + x - v;
}

template <typename T>
__global__ void __launch_bounds__(kScanThreads)
k_scan_reduce(const T *__restrict__ in, int64_t count, uint32_t *__restrict__ partial)
{
    int64_t base = (int64_t)blockIdx.x * kScanTile + threadIdx.x * kScanItems;
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < kScanItems; ++j)
        if (base + j < count) s += in[base + j];
    uint32_t total;
    block_exclusive_scan(s, total);
    if (threadIdx.x == 0) partial[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads)
k_scan_partials(uint32_t *__restrict__ partial, int64_t parts)
{
    uint32_t carry = 0;
    for (int64_t base = 0; base < parts; base += kScanThreads) {
        int64_t i = base + threadIdx.x;
        uint32_t v = (i < parts) ? partial[i] : 0u;
        uint32_t total;
        uint32_t ex = block_exclusive_scan(v, total);
        if (i < parts) partial[i] = carry + ex;
        carry += total;
    }
}

// kItems per thread; partial == null: a single block scans everything.
template <typename T, int kItems>
__global__ void __launch_bounds__(kScanThreads)
k_scan_down(const T *__restrict__ in, uint32_t *__restrict__ out, int64_t count,
            const uint32_t *__restrict__ partial)
{
    int64_t base = (int64_t)blockIdx.x * kScanThreads * kItems + threadIdx.x * kItems;
    uint32_t v[kItems];
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        v[j] = (base + j < count) ? in[base + j] : 0u;
        s += v[j];
    }
    uint32_t total;
    uint32_t run = block_exclusive_scan(s, total) + (partial ? partial[blockIdx.x] : 0u);
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        if (base + j < count) out[base + j] = run;
        run += v[j];
    }
}

// Up to this many entries one block scans in one launch instead of three.
constexpr int kScanSingleItems = 32;
constexpr int64_t kScanSingle = (int64_t)kScanThreads * kScanSingleItems;  // 8192

}  // namespace

int64_t scan_partial_count(int64_t count) { return (count + kScanTile - 1) / kScanTile; }

template <typename T>
static void scan_exclusive(const T *in, uint32_t *out, int64_t count, uint32_t *partial,
                           cudaStream_t st)
{
    if (count <= kScanSingle) {
        k_scan_down<T, kScanSingleItems><<<1, kScanThreads, 0, st>>>(in, out, count, nullptr);
        g_launches += 1;
        return;
    }
    int64_t parts = scan_partial_count(count);
    k_scan_reduce<T><<<(unsigned)parts, kScanThreads, 0, st>>>(in, count, partial);
    k_scan_partials<<<1, kScanThreads, 0, st>>>(partial, parts);
    k_scan_down<T, kScanItems><<<(unsigned)parts, kScanThreads, 0, st>>>(in, out, count, partial);
    g_launches += 3;
}

void launch_scan_u8(const uint8_t *in, uint32_t *out, int64_t count, uint32_t *partial,
                    cudaStream_t st)
{
    scan_exclusive<uint8_t>(in, out, count, partial, st);
}

// Clears the sort's control words (and with them the fold ticket), then
// finds the cube.
void launch_bbox(const float *pos, const float *mass, const Buffers &b, cudaStream_t st)
{
    cudaMemsetAsync(b.sort_ctl, 0, sizeof(uint32_t) * (size_t)sort_ctl_words(), st);
    k_bbox<<<b.bbox_blocks, kBBoxThreads, 0, st>>>(pos, mass, b.n, b.bbox_partial, bbox_ticket(b),
                                                   b.params);
    g_launches += 1;
}

void launch_gather(const float *pos, const float *mass, const uint32_t *perm, const Buffers &b,
                   cudaStream_t st)
{
    k_gather<<<ceil_div(b.n, 256), 256, 0, st>>>(pos, mass, perm, b.n, b.ps, &b.params->status);
    g_launches += 1;
}

}  // namespace obh
