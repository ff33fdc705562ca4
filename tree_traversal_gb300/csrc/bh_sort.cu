// bh_sort.cu -- a3: stable least-significant-digit radix sort of (key, index).
//
// The pages name the host Morton sort as the limit of their solver (orrery:
// docs/performance/sycl_tree.md, the five findings and "Where one evaluation
// goes": 40-46 per cent of every evaluation) and a device radix sort as the
// first thing to do about it. Seven passes of 9 bits cover the 63-bit keys.
// Each pass is three launches with no inter-block waiting: per-tile digit
// counts, a per-digit scan over tiles, and a stable scatter. The scatter
// ranks every key of its 2048-key tile (each warp walks a contiguous 256-key
// span 32 keys at a time, ranking equal digits with a match-any vote), puts
// the tile in digit order in shared memory, and then writes each digit's run
// to its global slot with consecutive threads on consecutive addresses.
#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 8;                       // per lane
constexpr int kTile = kThreads * kItems;        // 2048 keys per block
constexpr int kWarpSpan = 32 * kItems;          // 256 consecutive keys per warp
constexpr int kBits = 9;
constexpr int kBins = 1 << kBits;               // 512 digits
constexpr int kPasses = 7;                      // 7 x 9 = 63 key bits
constexpr int kBinsPerThread = kBins / kThreads;

// dynamic shared memory of the scatter: digit counters and the reordered tile
struct ScatterSmem {
    uint32_t cnt[kWarps][kBins];  // per-warp digit counts, then offsets
    uint32_t base[kBins];         // global start of each digit's run for this tile
    uint32_t loc[kBins];          // start of each digit's run inside the tile
    uint32_t warp_sum[kWarps];
    uint64_t key[kTile];
    uint32_t val[kTile];
};

__device__ __forceinline__ uint32_t digit_of(uint64_t key, int shift)
{
    return (uint32_t)((key >> shift) & (kBins - 1));
}

__global__ void __launch_bounds__(kThreads)
k_radix_hist(const uint64_t *__restrict__ keys, int64_t n, int shift,
             uint32_t *__restrict__ hist, int nblocks)
{
    __shared__ uint32_t h[kBins];
    for (int d = threadIdx.x; d < kBins; d += kThreads) h[d] = 0;
    __syncthreads();
    int64_t base = (int64_t)blockIdx.x * kTile;
#pragma unroll 4
    for (int it = 0; it < kItems; ++it) {
        int64_t e = base + it * kThreads + threadIdx.x;
        if (e < n) atomicAdd(&h[digit_of(keys[e], shift)], 1u);
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kBins; d += kThreads)
        hist[(int64_t)d * nblocks + blockIdx.x] = h[d];
}

// Block-wide exclusive scan of one value per thread; also returns the total.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *warp_sum, uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    total = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before += warp_sum[w];
        total += warp_sum[w];
    }
    __syncthreads();
    return before + x - v;
}

// One block per digit: exclusive scan of that digit's tile counts, in place.
__global__ void __launch_bounds__(kThreads)
k_radix_scan(uint32_t *__restrict__ hist, int nblocks, uint32_t *__restrict__ total)
{
    __shared__ uint32_t warp_sum[kWarps];
    uint32_t *row = hist + (int64_t)blockIdx.x * nblocks;
    uint32_t carry = 0;
    for (int base = 0; base < nblocks; base += kThreads) {
        int i = base + threadIdx.x;
        uint32_t v = (i < nblocks) ? row[i] : 0u;
        uint32_t all;
        uint32_t ex = block_scan(v, warp_sum, all);
        if (i < nblocks) row[i] = carry + ex;
        carry += all;
    }
    if (threadIdx.x == 0) total[blockIdx.x] = carry;
}

__global__ void __launch_bounds__(kThreads)
k_radix_scatter(const uint64_t *__restrict__ kin, const uint32_t *__restrict__ vin,
                uint64_t *__restrict__ kout, uint32_t *__restrict__ vout, int64_t n, int shift,
                const uint32_t *__restrict__ hist, const uint32_t *__restrict__ total,
                int nblocks, int first_pass, int *status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScatterSmem &S = *reinterpret_cast<ScatterSmem *>(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const int64_t tile0 = (int64_t)blockIdx.x * kTile;
    const int tile_n = (n - tile0 < (int64_t)kTile) ? (int)(n - tile0) : kTile;

    // global start of each digit = exclusive scan of the digit totals, plus
    // this tile's offset within the digit
    {
        uint32_t v[kBinsPerThread], sum = 0;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            v[q] = total[threadIdx.x * kBinsPerThread + q];
            sum += v[q];
        }
        uint32_t all;
        uint32_t run = block_scan(sum, S.warp_sum, all);
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            const int d = threadIdx.x * kBinsPerThread + q;
            S.base[d] = run + hist[(int64_t)d * nblocks + blockIdx.x];
            run += v[q];
        }
        for (int d = threadIdx.x; d < kBins; d += kThreads)
            for (int w = 0; w < kWarps; ++w) S.cnt[w][d] = 0;
    }
    __syncthreads();

    // phase A: per-warp digit counts, spans walked in order
    const int span = warp * kWarpSpan;
    uint64_t key[kItems];
    uint32_t val[kItems];
    uint32_t dig[kItems];
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int e = span + r * 32 + lane;
        const bool ok = e < tile_n;
        key[r] = ok ? kin[tile0 + e] : 0ull;
        val[r] = ok ? (first_pass ? (uint32_t)(tile0 + e) : vin[tile0 + e]) : 0u;
        dig[r] = ok ? digit_of(key[r], shift) : (uint32_t)kBins;
        const unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        const int leader = __ffs(peers) - 1;
        if (lane == leader && dig[r] < (uint32_t)kBins) S.cnt[warp][dig[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // per digit: offsets of each warp's first key inside the digit's run, and
    // the start of each digit's run inside the tile
    {
        uint32_t c[kBinsPerThread], sum = 0;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            const int d = threadIdx.x * kBinsPerThread + q;
            uint32_t run = 0;
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t x = S.cnt[w][d];
                S.cnt[w][d] = run;
                run += x;
            }
            c[q] = run;
            sum += run;
        }
        uint32_t all;
        uint32_t run = block_scan(sum, S.warp_sum, all);
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            S.loc[threadIdx.x * kBinsPerThread + q] = run;
            run += c[q];
        }
    }
    __syncthreads();

    // phase B: place every key at its stable position inside the tile
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
        const int leader = __ffs(peers) - 1;
        if (dig[r] < (uint32_t)kBins) {
            const uint32_t p = S.loc[dig[r]] + S.cnt[warp][dig[r]] + __popc(peers & lt);
            if (p < (uint32_t)tile_n) {
                S.key[p] = key[r];
                S.val[p] = val[r];
            } else {
                atomicOr(status, kStatusInternal);
            }
        }
        __syncwarp();
        if (lane == leader && dig[r] < (uint32_t)kBins) S.cnt[warp][dig[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // phase C: write each digit's run contiguously
    for (int p = threadIdx.x; p < tile_n; p += kThreads) {
        const uint64_t k = S.key[p];
        const uint32_t d = digit_of(k, shift);
        const uint64_t g = (uint64_t)S.base[d] + (uint32_t)(p - S.loc[d]);
        if (g < (uint64_t)n) {
            kout[g] = k;
            vout[g] = S.val[p];
        } else {
            atomicOr(status, kStatusInternal);
        }
    }
}

// Up to 4096 keys: the whole sort in one block, all seven passes in
// shared memory. Each pass ranks the keys exactly as the scatter above (per-
// warp digit counts with match-any votes, spans and rounds walked in key
// order, so equal digits keep their order), writes every key to its rank in
// shared memory and reads its new keys back. One launch instead of 21: at
// these sizes the sort is bound by launch latency, not by work.
constexpr int kSmallThreads = 512;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallItems = 8;                           // rounds per lane at most
// 4096 keys at most: the cost grows with the rounds per lane (about 6 us per
// round over the seven passes, scattering keys into shared memory; measured
// 31 / 68 us at 1024 / 4096 keys against 76 / 101 us for the multi-block
// passes), so beyond 4096 keys it would no longer win.
constexpr int kSmallN = kSmallThreads * kSmallItems;     // 4096

struct SmallSortSmem {
    uint64_t key[kSmallN];
    uint32_t val[kSmallN];
    uint32_t cnt[kSmallWarps][kBins];  // per-warp digit counts, then offsets
    uint32_t loc[kBins];               // start of each digit's run
};

// Exclusive scan of one value per thread over a 512-thread block.
__device__ __forceinline__ uint32_t block_scan_512(uint32_t v, uint32_t &total)
{
    __shared__ uint32_t sums[kSmallWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) sums[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    total = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
        if (w < warp) before += sums[w];
        total += sums[w];
    }
    __syncthreads();
    return before + x - v;
}

__global__ void __launch_bounds__(kSmallThreads)
k_radix_sort_small(const uint64_t *__restrict__ kin, uint64_t *__restrict__ kout,
                   uint32_t *__restrict__ vout, int n, int *status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmallSortSmem &S = *reinterpret_cast<SmallSortSmem *>(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    // each warp takes a contiguous span of rounds * 32 keys, just enough to
    // cover n; rounds walk the span in key order (round-major, then lane)
    const int rounds = (n + kSmallThreads - 1) / kSmallThreads;
    const int span = warp * 32 * rounds;
    uint64_t key[kSmallItems];
    uint32_t val[kSmallItems];
#pragma unroll
    for (int r = 0; r < kSmallItems; ++r) {
        const int e = span + r * 32 + lane;
        key[r] = (r < rounds && e < n) ? kin[e] : 0ull;
        val[r] = (uint32_t)e;
    }
    for (int pass = 0; pass < kPasses; ++pass) {
        const int shift = kBits * pass;
        for (int i = threadIdx.x; i < kSmallWarps * kBins; i += kSmallThreads) (&S.cnt[0][0])[i] = 0;
        __syncthreads();
        uint32_t dig[kSmallItems];
#pragma unroll
        for (int r = 0; r < kSmallItems; ++r) {  // per-warp digit counts
            const int e = span + r * 32 + lane;
            dig[r] = (r < rounds && e < n) ? digit_of(key[r], shift) : (uint32_t)kBins;
            if (r >= rounds) continue;  // warp-uniform
            const unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
            if (lane == __ffs(peers) - 1 && dig[r] < (uint32_t)kBins) S.cnt[warp][dig[r]] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        {  // thread d owns digit d: offsets of each warp's first key in the run
            const int d = threadIdx.x;
            uint32_t run = 0;
            for (int w = 0; w < kSmallWarps; ++w) {
                const uint32_t x = S.cnt[w][d];
                S.cnt[w][d] = run;
                run += x;
            }
            uint32_t all;
            S.loc[d] = block_scan_512(run, all);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kSmallItems; ++r) {  // every key to its stable rank
            if (r >= rounds) break;  // warp-uniform
            const unsigned peers = __match_any_sync(0xffffffffu, dig[r]);
            if (dig[r] < (uint32_t)kBins) {
                const uint32_t p = S.loc[dig[r]] + S.cnt[warp][dig[r]] + __popc(peers & lt);
                if (p < (uint32_t)n) {
                    S.key[p] = key[r];
                    S.val[p] = val[r];
                } else {
                    atomicOr(status, kStatusInternal);
                }
            }
            __syncwarp();
            if (lane == __ffs(peers) - 1 && dig[r] < (uint32_t)kBins) S.cnt[warp][dig[r]] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kSmallItems; ++r) {  // read back in rank order
            const int e = span + r * 32 + lane;
            if (r < rounds && e < n) {
                key[r] = S.key[e];
                val[r] = S.val[e];
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < kSmallItems; ++r) {
        const int e = span + r * 32 + lane;
        if (r < rounds && e < n) {
            kout[e] = key[r];
            vout[e] = val[r];
        }
    }
}

}  // namespace

// Sorts b.keys_a (filled by the key phase) with the original indices as
// values. Seven passes: the result lands in keys_b / idx_b.
void prepare_sort()
{
    static std::atomic<bool> configured[64];  // the opt-in is set once per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev].load()) {
        cudaFuncSetAttribute(k_radix_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(ScatterSmem));
        cudaFuncSetAttribute(k_radix_sort_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SmallSortSmem));
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
}

void launch_sort(const Buffers &b, cudaStream_t st, uint64_t **keys_sorted, uint32_t **perm)
{
    const int nb = b.radix_blocks;
    const size_t smem = sizeof(ScatterSmem);
    prepare_sort();
    if (b.n <= kSmallN) {  // one block, one launch; the result lands where the passes' would
        k_radix_sort_small<<<1, kSmallThreads, sizeof(SmallSortSmem), st>>>(
            b.keys_a, b.keys_b, b.idx_b, (int)b.n, &b.params->status);
        g_launches += 1;
        *keys_sorted = b.keys_b;
        *perm = b.idx_b;
        return;
    }
    uint64_t *kin = b.keys_a, *kout = b.keys_b;
    uint32_t *vin = b.idx_a, *vout = b.idx_b;
    for (int p = 0; p < kPasses; ++p) {
        const int shift = kBits * p;
        k_radix_hist<<<nb, kThreads, 0, st>>>(kin, b.n, shift, b.radix_hist, nb);
        k_radix_scan<<<kBins, kThreads, 0, st>>>(b.radix_hist, nb, b.radix_total);
        k_radix_scatter<<<nb, kThreads, smem, st>>>(kin, vin, kout, vout, b.n, shift,
                                                    b.radix_hist, b.radix_total, nb, p == 0,
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

int radix_bins() { return kBins; }

}  // namespace obh
