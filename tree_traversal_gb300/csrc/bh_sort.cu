// bh_sort.cu -- a2 Morton keys and a3 their stable least-significant-digit
// radix sort of (key, index).
//
// The pages name the host Morton sort as the limit of their solver (orrery:
// docs/performance/sycl_tree.md, the five findings and "Where one evaluation
// goes": 40-46 per cent of every evaluation) and a device radix sort as the
// first thing to do about it. The 21-bit quantisation per axis follows the
// workload definition that accompanies the pages (a quantised bounding cube,
// 21 bits per axis). Seven passes of 9 bits cover the 63-bit keys.
//
// The key kernel also counts the digits of all seven passes at once (seven
// 512-bin histograms), so every pass is a single launch in the manner of the
// published "Onesweep" radix sort (Adinets and Merrill, 2022) with its
// decoupled look-back (Merrill and Garland, 2016): a block takes the next
// tile (4096 to 8192 keys, sized to the SM count) by ticket, counts its
// digits, publishes the counts, and adds up the counts of the tiles before
// it by reading their published words backwards until it meets a tile that
// has already published its inclusive prefix. A block only ever waits for
// tiles with smaller tickets, which are already running, so every wait
// ends; each is still bounded, and a wait that runs out flags an internal
// error instead of spinning on. The tile is then ranked (each warp walks a
// contiguous span of 256 to 512 keys, 32 keys at a time, finding the lanes
// with equal digits by one vote per digit bit), put in digit order in shared
// memory, and each digit's run is written to its global slot with
// consecutive threads on consecutive addresses.
#include <stdlib.h>

#include <type_traits>

#include <cuda/atomic>

#include "bh_common.cuh"

namespace obh {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBits = 9;
constexpr int kBins = 1 << kBits;               // 512 digits
constexpr int kPasses = 7;                      // 7 x 9 = 63 key bits
constexpr int kBinsPerThread = kBins / kThreads;

// One pass's tile: kItems keys per lane, so kThreads * kItems keys per block
// and a contiguous span of 32 * kItems keys per warp. A pass is a chain of
// latencies inside each tile (load, rank, look-back, place, write), so the
// fastest tiling is the smallest tile that still fills whole waves of one
// block per SM: kItems is the smallest even count in [8, 16] for which the
// tiles fill no more than the waves that 16 would need. (Up to 622 592 keys
// on 152 SMs that is 8: 4096-key tiles, two blocks per SM.) Measured at
// 1M: 0.106 ms with 7168-key tiles (147 tiles on 152 SMs) against 0.111
// with 8192 (128 tiles) and 0.129 with 4096; at 2M 0.192 (293 tiles, two
// waves) against 0.201 (256).
template <int kItemsT>
struct Tiling {
    static constexpr int kItems = kItemsT;
    static constexpr int kTile = kThreads * kItems;
    static constexpr int kWarpSpan = 32 * kItems;
    // a key's rank inside its warp's run of a digit is below the warp's
    // span: one byte per key up to 256 keys per warp, else 16 bits
    static constexpr int kRankBits = kWarpSpan <= 256 ? 8 : 16;
    static constexpr int kRanksPerWord = 32 / kRankBits;
    static constexpr uint32_t kRankMask = (1u << kRankBits) - 1u;
};
constexpr int kMinTileItems = 8;    // 4096-key tiles
constexpr int kMaxTileItems = 16;   // 8192-key tiles

// Control words of one evaluation, cleared before the bounding box: the
// digit counts of every pass, one tile ticket per pass, and the bounding
// box's fold ticket.
constexpr int kCtlCounts = kPasses * kBins;
constexpr int kCtlWords = kCtlCounts + kPasses + 1;

// A look-back word: bit 31 set = the inclusive count of the digit over this
// tile and all before it (at most 2^30, the largest n); bit 30 set = this
// tile's own count only (at most 8192); zero = not yet published.
constexpr uint32_t kLookInclusive = 0x80000000u;
constexpr uint32_t kLookTileOnly = 0x40000000u;
constexpr int kLookSpins = 1 << 20;  // polls of an unpublished word before giving up
// ORRERY_TEST_SORT_STALL=1 (failure-path tests): tile 0 of the first pass
// never publishes its counts, and the tiles after it give up after this many
// polls, flag an internal error and go on
constexpr int kTestLookSpins = 64;
constexpr int kLookWindow = 4;       // earlier tiles' words read at once

// Spreads the low 21 bits of v so that bit b lands at bit 3b.
__device__ __forceinline__ uint64_t spread3(uint32_t v)
{
    uint64_t x = v & 0x1fffffu;
    x = (x | (x << 32)) & 0x001f00000000ffffull;
    x = (x | (x << 16)) & 0x001f0000ff0000ffull;
    x = (x | (x << 8)) & 0x100f00f00f00f00full;
    x = (x | (x << 4)) & 0x10c30c30c30c30c3ull;
    x = (x | (x << 2)) & 0x1249249249249249ull;
    return x;
}

// q = min(floor(fl(fl(x - lo) * inv)), 2^21 - 1)
__device__ __forceinline__ uint32_t quantise(float x, float lo, float inv)
{
    float t = __fmul_rn(__fsub_rn(x, lo), inv);
    if (!(t >= 0.0f)) t = 0.0f;
    if (t >= 2097151.0f) return 2097151u;
    return (uint32_t)t;  // truncation is floor for t >= 0
}

// 63-bit Morton key of particle i, x the high bit of each level's triple.
__device__ __forceinline__ uint64_t morton_key(const float *__restrict__ pos, int64_t i,
                                               const float lo[3], float inv)
{
    const uint32_t qx = quantise(__ldg(pos + 3 * i + 0), lo[0], inv);
    const uint32_t qy = quantise(__ldg(pos + 3 * i + 1), lo[1], inv);
    const uint32_t qz = quantise(__ldg(pos + 3 * i + 2), lo[2], inv);
    return (spread3(qx) << 2) | (spread3(qy) << 1) | spread3(qz);
}

__device__ __forceinline__ uint32_t digit_of(uint64_t key, int shift)
{
    return (uint32_t)((key >> shift) & (kBins - 1));
}

// The lanes of this warp holding a valid key with this lane's digit: one vote
// per digit bit. (A match-any vote gives the same set, but its cost grows
// with the number of distinct digits in the warp: measured at about 1 000
// cycles per 32 random 9-bit digits, against a few dozen for the votes.)
__device__ __forceinline__ unsigned digit_peers(uint32_t dig, bool valid)
{
    unsigned peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 0; b < kBits; ++b) {
        const bool bit = (dig >> b) & 1u;
        const unsigned vote = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? vote : ~vote;
    }
    return peers;
}

// Rank of this lane's key among the warp's keys with the same digit, counting
// the keys of earlier rounds in cnt[digit] (updated here for the next round).
__device__ __forceinline__ uint32_t warp_rank(uint32_t *cnt, uint32_t dig, bool valid)
{
    const unsigned lane_lt = (1u << (threadIdx.x & 31)) - 1u;
    const unsigned peers = digit_peers(dig, valid);
    const uint32_t before = valid ? cnt[dig] : 0u;
    __syncwarp();
    if (valid && (threadIdx.x & 31) == __ffs(peers) - 1) cnt[dig] = before + __popc(peers);
    __syncwarp();
    return before + __popc(peers & lane_lt);
}

// Keys only (the single-block sort counts its own digits).
__global__ void __launch_bounds__(256)
k_morton(const float *__restrict__ pos, int64_t n, const DeviceParams *__restrict__ P,
         uint64_t *__restrict__ keys)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float lo[3] = {P->lo[0], P->lo[1], P->lo[2]};
    keys[i] = morton_key(pos, i, lo, P->inv);
}

// Keys and the digit counts of all seven passes. Each block counts its keys
// in shared memory and adds its histograms to the global ones; the grid also
// clears the look-back words of the first pass.
constexpr int kCountThreads = 512;
constexpr int kCountKeysPerThread = 4;   // more blocks, more keys in flight
constexpr int kCountMaxBlocks = 2 * 152;

__global__ void __launch_bounds__(kCountThreads)
k_keys_count(const float *__restrict__ pos, int64_t n, const DeviceParams *__restrict__ P,
             uint64_t *__restrict__ keys, uint32_t *__restrict__ counts,
             uint32_t *__restrict__ look0, int64_t look_words)
{
    __shared__ uint32_t h[kCtlCounts];
    for (int i = threadIdx.x; i < kCtlCounts; i += kCountThreads) h[i] = 0;
    __syncthreads();
    const float lo[3] = {P->lo[0], P->lo[1], P->lo[2]};
    const float inv = P->inv;
    const int64_t stride = (int64_t)gridDim.x * kCountThreads;
    for (int64_t i = (int64_t)blockIdx.x * kCountThreads + threadIdx.x; i < n; i += stride) {
        const uint64_t key = morton_key(pos, i, lo, inv);
        keys[i] = key;
#pragma unroll
        for (int p = 0; p < kPasses; ++p) atomicAdd(&h[p * kBins + digit_of(key, kBits * p)], 1u);
    }
    for (int64_t i = (int64_t)blockIdx.x * kCountThreads + threadIdx.x; i < look_words; i += stride)
        look0[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < kCtlCounts; i += kCountThreads)
        if (h[i]) atomicAdd(&counts[i], h[i]);
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


// dynamic shared memory of one pass: digit counters and the reordered tile
template <int kItems>
struct PassSmem {
    uint32_t cnt[kWarps][kBins];  // per-warp digit counts, then offsets
    uint32_t base[kBins];         // global start of each digit's run for this tile
    uint32_t loc[kBins];          // start of each digit's run inside the tile
    uint32_t warp_sum[kWarps];
    uint32_t tile;                // this block's ticket = its tile
    uint64_t key[Tiling<kItems>::kTile];
    uint32_t val[Tiling<kItems>::kTile];
};

// Look-back words are read and written as device-scope relaxed atomics: each
// word carries its whole meaning, so no other memory needs ordering with it.
__device__ __forceinline__ uint32_t look_load(uint32_t *p)
{
    return cuda::atomic_ref<uint32_t, cuda::thread_scope_device>(*p).load(cuda::memory_order_relaxed);
}

__device__ __forceinline__ void look_store(uint32_t *p, uint32_t v)
{
    cuda::atomic_ref<uint32_t, cuda::thread_scope_device>(*p).store(v, cuda::memory_order_relaxed);
}

// One pass over the tile of this block's ticket. counts: the pass's digit
// totals; ticket: the pass's tile counter (zero on entry); look: the pass's
// look-back words [tiles][kBins] (zero on entry); look_next: the next pass's
// words, whose row for this tile is cleared here (null on the last pass);
// silent_tile: a tile that publishes nothing (-1: none; failure-path tests
// only); spin_limit: polls of an unpublished word before giving up.
template <int kItems>
__global__ void __launch_bounds__(kThreads)
k_onesweep(const uint64_t *__restrict__ kin, const uint32_t *__restrict__ vin,
           uint64_t *__restrict__ kout, uint32_t *__restrict__ vout, int64_t n, int pass,
           const uint32_t *__restrict__ counts, uint32_t *ticket, uint32_t *look,
           uint32_t *look_next, int tiles, int silent_tile, int spin_limit, int *status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using T = Tiling<kItems>;
    PassSmem<kItems> &S = *reinterpret_cast<PassSmem<kItems> *>(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int shift = kBits * pass;
    if (threadIdx.x == 0) S.tile = atomicAdd(ticket, 1u);
    for (int d = threadIdx.x; d < kBins; d += kThreads)
        for (int w = 0; w < kWarps; ++w) S.cnt[w][d] = 0;

    // global start of each digit: exclusive scan of the pass's digit totals
    uint32_t start[kBinsPerThread];
    {
        uint32_t v[kBinsPerThread], sum = 0;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            v[q] = counts[threadIdx.x * kBinsPerThread + q];
            sum += v[q];
        }
        uint32_t all;
        uint32_t run = block_scan(sum, S.warp_sum, all);  // its barriers also publish S.tile
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) {
            start[q] = run;
            run += v[q];
        }
    }
    const int tile = (int)S.tile;
    if (tile >= tiles) {  // block-uniform; cannot happen with one block per tile
        if (threadIdx.x == 0) atomicOr(status, kStatusInternal);
        return;
    }
    if (look_next)
        for (int d = threadIdx.x; d < kBins; d += kThreads) look_next[(int64_t)tile * kBins + d] = 0;
    const int64_t tile0 = (int64_t)tile * T::kTile;
    const int tile_n = (n - tile0 < (int64_t)T::kTile) ? (int)(n - tile0) : T::kTile;

    // phase A: per-warp digit counts and each key's rank inside its warp's
    // run of the digit (packed kRanksPerWord to a register), spans walked in
    // order
    const int span = warp * T::kWarpSpan;
    uint64_t key[kItems];
    uint32_t val[kItems];
    uint32_t rank[(kItems + T::kRanksPerWord - 1) / T::kRanksPerWord] = {};
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int e = span + r * 32 + lane;
        const bool ok = e < tile_n;
        key[r] = ok ? kin[tile0 + e] : 0ull;
        val[r] = ok ? (pass == 0 ? (uint32_t)(tile0 + e) : vin[tile0 + e]) : 0u;
    }
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const bool ok = span + r * 32 + lane < tile_n;
        rank[r / T::kRanksPerWord] |= warp_rank(S.cnt[warp], digit_of(key[r], shift), ok)
                                      << (T::kRankBits * (r % T::kRanksPerWord));
    }
    __syncthreads();

    // per digit: offsets of each warp's first key inside the tile's run, and
    // the tile's count, published at once
    uint32_t c[kBinsPerThread];
    uint32_t *row = look + (int64_t)tile * kBins;
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
        if (tile != silent_tile) look_store(row + d, (tile == 0 ? kLookInclusive : kLookTileOnly) | run);
    }

    // look-back: the count of each digit over all earlier tiles, reading the
    // words of kLookWindow tiles at once and adding them nearest first up to
    // the first inclusive one; an unpublished word ends the window and is
    // read again after a growing pause
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) {
        const int d = threadIdx.x * kBinsPerThread + q;
        uint32_t before = 0;
        if (tile > 0) {
            int spins = 0;
            unsigned pause = 32;
            for (int j = tile - 1; j >= 0;) {
                uint32_t s[kLookWindow];
#pragma unroll
                for (int u = 0; u < kLookWindow; ++u)  // past tile 0: an inclusive zero
                    s[u] = j - u >= 0 ? look_load(look + (int64_t)(j - u) * kBins + d) : kLookInclusive;
                int used = 0;
                bool found = false;
#pragma unroll
                for (int u = 0; u < kLookWindow; ++u) {
                    if (found || used < u) break;
                    if (s[u] & kLookInclusive) {
                        before += s[u] & ~kLookInclusive;
                        found = true;
                    } else if (s[u] & kLookTileOnly) {
                        before += s[u] & ~kLookTileOnly;
                        ++used;
                    }
                }
                if (found) break;
                j -= used;
                if (used == 0) {  // tile j has not published yet
                    if (++spins > spin_limit) {  // it never did: give up, flagged
                        atomicOr(status, kStatusInternal);
                        break;
                    }
                    __nanosleep(pause);
                    pause = pause < 1024 ? 2 * pause : pause;
                }
            }
            if (tile != silent_tile) look_store(row + d, kLookInclusive | (before + c[q]));
        }
        S.base[d] = start[q] + before;
    }

    // start of each digit's run inside the tile
    {
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < kBinsPerThread; ++q) sum += c[q];
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
        if (span + r * 32 + lane < tile_n) {
            const uint32_t d = digit_of(key[r], shift);
            const uint32_t p = S.loc[d] + S.cnt[warp][d] +
                               ((rank[r / T::kRanksPerWord] >> (T::kRankBits * (r % T::kRanksPerWord))) &
                                T::kRankMask);
            if (p < (uint32_t)tile_n) {
                S.key[p] = key[r];
                S.val[p] = val[r];
            } else {
                atomicOr(status, kStatusInternal);
            }
        }
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
// shared memory. Each pass ranks the keys exactly as k_onesweep (per-
// warp digit counts and ranks from digit-bit votes, spans and rounds walked
// in key order, so equal digits keep their order), writes every key to its rank in
// shared memory and reads its new keys back. One launch instead of eight:
// at these sizes the sort is bound by launch latency, not by work.
constexpr int kSmallThreads = 512;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallItems = 8;                           // rounds per lane at most
// 4096 keys at most: the cost grows with the rounds per lane (about 6 us per
// round over the seven passes, scattering keys into shared memory; measured
// 31 / 68 us at 1024 / 4096 keys), so beyond 4096 keys it would no longer
// win.
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
        uint32_t rank[kSmallItems / 4] = {};
#pragma unroll
        for (int r = 0; r < kSmallItems; ++r) {  // per-warp digit counts and ranks
            if (r >= rounds) break;  // warp-uniform
            const bool ok = span + r * 32 + lane < n;
            rank[r / 4] |= warp_rank(S.cnt[warp], digit_of(key[r], shift), ok) << (8 * (r % 4));
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
            if (span + r * 32 + lane < n) {
                const uint32_t d = digit_of(key[r], shift);
                const uint32_t p = S.loc[d] + S.cnt[warp][d] + ((rank[r / 4] >> (8 * (r % 4))) & 0xffu);
                if (p < (uint32_t)n) {
                    S.key[p] = key[r];
                    S.val[p] = val[r];
                } else {
                    atomicOr(status, kStatusInternal);
                }
            }
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

// The tile sizes a pass may use, one instantiation each.
template <int kItems>
void opt_in_pass()
{
    cudaFuncSetAttribute(k_onesweep<kItems>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(PassSmem<kItems>));
}

void prepare_sort()
{
    static std::atomic<bool> configured[64];  // the opt-in is set once per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev].load()) {
        opt_in_pass<8>();
        opt_in_pass<10>();
        opt_in_pass<12>();
        opt_in_pass<14>();
        opt_in_pass<16>();
        cudaFuncSetAttribute(k_radix_sort_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SmallSortSmem));
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
}

// SMs of the current device (read once per device).
static int sm_count()
{
    static std::atomic<int> sms[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && sms[dev].load() > 0) return sms[dev].load();
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        v = 1;
    }
    if (dev >= 0 && dev < 64) sms[dev] = v;
    return v;
}

// Keys per lane of a pass over n keys (see Tiling).
static int tile_items(int64_t n)
{
    const int64_t per_wave = (int64_t)kThreads * sm_count();  // keys per item of a wave
    const int64_t waves = (n + per_wave * kMaxTileItems - 1) / (per_wave * kMaxTileItems);
    int64_t items = (n + per_wave * waves - 1) / (per_wave * waves);
    items += items & 1;
    return (int)(items < kMinTileItems ? kMinTileItems : items > kMaxTileItems ? kMaxTileItems : items);
}

// Tiles of the passes for n keys (more than the single-block size).
static int pass_tiles(int64_t n)
{
    const int64_t tile = (int64_t)kThreads * tile_items(n);
    return (int)((n + tile - 1) / tile);
}

// a2: the keys into b.keys_a; above the single-block size also the digit
// counts of every pass, with the sort's control words cleared first.
void launch_morton(const float *pos, const Buffers &b, cudaStream_t st)
{
    if (b.n <= kSmallN) {
        k_morton<<<ceil_div(b.n, 256), 256, 0, st>>>(pos, b.n, b.params, b.keys_a);
        g_launches += 1;
        return;
    }
    int64_t blocks = ((int64_t)b.n + kCountThreads * kCountKeysPerThread - 1) /
                     (kCountThreads * kCountKeysPerThread);
    if (blocks > kCountMaxBlocks) blocks = kCountMaxBlocks;
    k_keys_count<<<(unsigned)blocks, kCountThreads, 0, st>>>(
        pos, b.n, b.params, b.keys_a, b.sort_ctl, b.sort_look, (int64_t)pass_tiles(b.n) * kBins);
    g_launches += 1;
}

// a3: sorts b.keys_a (from launch_morton) with the original indices as
// values; returns where the sorted keys and the permutation landed.
void launch_sort(const Buffers &b, cudaStream_t st, uint64_t **keys_sorted, uint32_t **perm)
{
    prepare_sort();
    if (b.n <= kSmallN) {  // one block, one launch
        k_radix_sort_small<<<1, kSmallThreads, sizeof(SmallSortSmem), st>>>(
            b.keys_a, b.keys_b, b.idx_b, (int)b.n, &b.params->status);
        g_launches += 1;
        *keys_sorted = b.keys_b;
        *perm = b.idx_b;
        return;
    }
    const int tiles = pass_tiles(b.n);
    const int64_t look_words = (int64_t)tiles * kBins;  // the look-back rows of one pass
    const char *stall = getenv("ORRERY_TEST_SORT_STALL");
    const bool stalled = stall && stall[0] == '1';
    uint64_t *kin = b.keys_a, *kout = b.keys_b;
    uint32_t *vin = b.idx_a, *vout = b.idx_b;
    const int items = tile_items(b.n);
    for (int p = 0; p < kPasses; ++p) {
        uint32_t *look = b.sort_look + (p & 1) * look_words;
        uint32_t *look_next = p + 1 < kPasses ? b.sort_look + ((p + 1) & 1) * look_words : nullptr;
        auto pass = [&](auto itag) {
            constexpr int I = decltype(itag)::value;
            k_onesweep<I><<<tiles, kThreads, sizeof(PassSmem<I>), st>>>(
                kin, vin, kout, vout, b.n, p, b.sort_ctl + p * kBins, b.sort_ctl + kCtlCounts + p,
                look, look_next, tiles, stalled && p == 0 ? 0 : -1,
                stalled ? kTestLookSpins : kLookSpins, &b.params->status);
        };
        switch (items) {
        case 8: pass(std::integral_constant<int, 8>{}); break;
        case 10: pass(std::integral_constant<int, 10>{}); break;
        case 12: pass(std::integral_constant<int, 12>{}); break;
        case 14: pass(std::integral_constant<int, 14>{}); break;
        default: pass(std::integral_constant<int, 16>{}); break;
        }
        g_launches += 1;
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

// Both passes' look-back rows, sized for the smaller tiles whatever n (so
// the size only grows with n, as the workspace assumes).
int64_t sort_look_words(int64_t n)
{
    constexpr int tile = Tiling<kMinTileItems>::kTile;
    return 2 * ((n + tile - 1) / tile) * kBins;
}

int sort_ctl_words() { return kCtlWords; }

unsigned *bbox_ticket(const Buffers &b) { return b.sort_ctl + kCtlCounts + kPasses; }

}  // namespace obh
