// bh_sort.cu -- a3: stable least-significant-digit radix sort of (key, index).
//
// The pages name the host Morton sort as the limit of their solver (orrery:
// docs/performance/sycl_tree.md, the five findings and "Where one evaluation
// goes": 40-46 per cent of every evaluation) and a device radix sort as the
// first thing to do about it. Eight passes of 8 bits cover the 63-bit keys.
// Each pass is three launches with no inter-block waiting: per-tile digit
// counts, a per-digit scan over tiles, and a stable scatter in which every
// warp ranks its elements with a match-any vote.
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;                      // per lane
constexpr int kTile = kThreads * kItems;        // 4096 keys per block
constexpr int kWarpSpan = 32 * kItems;          // 512 consecutive keys per warp
constexpr int kPasses = 8;

__global__ void __launch_bounds__(kThreads)
k_radix_hist(const uint64_t *__restrict__ keys, int64_t n, int shift,
             uint32_t *__restrict__ hist, int nblocks)
{
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    int64_t base = (int64_t)blockIdx.x * kTile;
#pragma unroll 4
    for (int it = 0; it < kItems; ++it) {
        int64_t e = base + it * kThreads + threadIdx.x;
        if (e < n) atomicAdd(&h[(keys[e] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[(int64_t)threadIdx.x * nblocks + blockIdx.x] = h[threadIdx.x];
}

// One block per digit: exclusive scan of that digit's tile counts, in place.
__global__ void __launch_bounds__(kThreads)
k_radix_scan(uint32_t *__restrict__ hist, int nblocks, uint32_t *__restrict__ total)
{
    __shared__ uint32_t s_warp[kWarps];
    uint32_t *row = hist + (int64_t)blockIdx.x * nblocks;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t carry = 0;
    for (int base = 0; base < nblocks; base += kThreads) {
        int i = base + threadIdx.x;
        uint32_t v = (i < nblocks) ? row[i] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        uint32_t before = 0, all = 0;
        for (int w = 0; w < kWarps; ++w) {
            if (w < warp) before += s_warp[w];
            all += s_warp[w];
        }
        if (i < nblocks) row[i] = carry + before + x - v;
        carry += all;
        __syncthreads();
    }
    if (threadIdx.x == 0) total[blockIdx.x] = carry;
}

// Stable scatter. The block's tile is split into one contiguous 512-key span
// per warp, walked 32 keys at a time in order, so a key's rank among equal
// digits is (keys of that digit in earlier spans of the block) + (in earlier
// rounds of this span) + (lower lanes of this round).
__global__ void __launch_bounds__(kThreads)
k_radix_scatter(const uint64_t *__restrict__ kin, const uint32_t *__restrict__ vin,
                uint64_t *__restrict__ kout, uint32_t *__restrict__ vout, int64_t n, int shift,
                const uint32_t *__restrict__ hist, const uint32_t *__restrict__ total,
                int nblocks, int first_pass, int *status)
{
    __shared__ uint32_t s_base[256];
    __shared__ uint32_t s_cnt[kWarps][256];
    __shared__ uint32_t s_warp[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;

    // global start of each digit = exclusive scan of the digit totals + this
    // block's offset within the digit
    {
        uint32_t v = total[threadIdx.x];
        uint32_t x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        uint32_t before = 0;
        for (int w = 0; w < warp; ++w) before += s_warp[w];
        s_base[threadIdx.x] =
            before + x - v + hist[(int64_t)threadIdx.x * nblocks + blockIdx.x];
        for (int w = 0; w < kWarps; ++w) s_cnt[w][threadIdx.x] = 0;
    }
    __syncthreads();

    const int64_t span = (int64_t)blockIdx.x * kTile + warp * kWarpSpan;
    uint64_t key[kItems];
    uint32_t val[kItems];
    uint32_t dig[kItems];
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        int64_t e = span + r * 32 + lane;
        bool ok = e < n;
        key[r] = ok ? kin[e] : 0ull;
        val[r] = ok ? (first_pass ? (uint32_t)e : vin[e]) : 0u;
        dig[r] = ok ? (uint32_t)((key[r] >> shift) & 255u) : 256u;
        unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        int leader = __ffs(peers) - 1;
        if (lane == leader && dig[r] < 256u) s_cnt[warp][dig[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {
        uint32_t run = s_base[threadIdx.x];
        for (int w = 0; w < kWarps; ++w) {
            uint32_t c = s_cnt[w][threadIdx.x];
            s_cnt[w][threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        int leader = __ffs(peers) - 1;
        if (dig[r] < 256u) {
            uint32_t pos = s_cnt[warp][dig[r]] + __popc(peers & lt);
            if (pos < (uint64_t)n) {
                kout[pos] = key[r];
                vout[pos] = val[r];
            } else {
                atomicOr(status, kStatusInternal);
            }
        }
        __syncwarp();
        if (lane == leader && dig[r] < 256u) s_cnt[warp][dig[r]] += __popc(peers);
        __syncwarp();
    }
}

}  // namespace

// Sorts b.keys_a (filled by the key phase) with the original indices as
// values. The result lands back in keys_a / idx_a (an even number of passes).
void launch_sort(const Buffers &b, cudaStream_t st, uint64_t **keys_sorted, uint32_t **perm)
{
    const int nb = b.radix_blocks;
    uint64_t *kin = b.keys_a, *kout = b.keys_b;
    uint32_t *vin = b.idx_a, *vout = b.idx_b;
    for (int p = 0; p < kPasses; ++p) {
        const int shift = 8 * p;
        k_radix_hist<<<nb, kThreads, 0, st>>>(kin, b.n, shift, b.radix_hist, nb);
        k_radix_scan<<<256, kThreads, 0, st>>>(b.radix_hist, nb, b.radix_total);
        k_radix_scatter<<<nb, kThreads, 0, st>>>(kin, vin, kout, vout, b.n, shift, b.radix_hist,
                                                 b.radix_total, nb, p == 0,
                                                 &b.params->status);
        g_launches += 3;
        uint64_t *tk = kin;
        kin = kout;
        kout = tk;
        uint32_t *tv = vin;
        vin = vout;
        vout = tv;
    }
    *keys_sorted = kin;
    *perm = vin;
}

int radix_blocks_for(int64_t n) { return (int)((n + kTile - 1) / kTile); }

}  // namespace obh
