// Stable LSD radix sort of (key, int32 value) pairs, one 8-bit digit per
// pass, as a single-pass "onesweep" kernel per digit with decoupled
// look-back (the CPU listing's counting pass + exclusive scan + stable
// scatter, gsplat 1.0.0, intersections.c, gs_radix_sort_without_gvl, done
// by every block for its own tile of keys at once).
//
// Per pass, each 256-thread block:
//   1. takes a virtual block id from an atomic ticket (so a block only ever
//      waits on blocks that are already running);
//   2. loads its tile of keys warp-striped (coalesced) into registers, and
//      starts one bulk copy (TMA, cp.async.bulk) of the tile's values into
//      shared memory, which is waited for only when the tile is reordered
//      (bulk-copying the keys too measured 2 % slower: they are needed in
//      registers at once, and the copy adds a shared-memory round trip);
//   3. ranks each key among equal digits of its warp (bit-sliced ballots +
//      popc), keeping input order (stability);
//   4. publishes its 256 digit counts, then walks back over predecessors'
//      words (bounded wait) to get its exclusive prefix per digit;
//   5. reorders the tile by digit in shared memory and writes it out, so
//      that consecutive threads write consecutive addresses of a bucket.
// The global digit histogram that step 4 adds as bucket starts comes from
// one histogram pass over all digits before the first sorting pass.
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kThreads = kSortThreads;
constexpr int kWarps = kThreads / kWarp;

template <typename K>
__device__ __forceinline__ uint32_t digit_of(K k, int shift, uint32_t mask) {
    return (uint32_t)(k >> shift) & mask;
}

// Mask of the digit starting at bit `shift` when only bits below `end_bit`
// take part (the last digit of a range may be narrower than 8 bits).
__host__ __device__ __forceinline__ uint32_t digit_mask(int shift, int end_bit) {
    const int bits = end_bit - shift >= 8 ? 8 : end_bit - shift;
    return bits <= 0 ? 0u : ((1u << bits) - 1u);
}

constexpr int kHistPasses = 4;  // digit passes per histogram launch
constexpr int kBulkPolls = 1 << 20;  // bounded try_wait rounds for a tile's bulk copies

template <typename K>
__global__ void __launch_bounds__(kThreads) k_digit_hist(const K* __restrict__ keys, int64_t n,
                                                         int shift0, int npasses, int end_bit,
                                                         uint32_t* __restrict__ hist) {
    // one private histogram per warp: only lanes of one warp ever contend on
    // an address, and a digit shared by the whole warp (common in high key
    // bits) is added once by lane 0
    __shared__ uint32_t sh[kWarps][kHistPasses][256];
    for (int i = threadIdx.x; i < kWarps * kHistPasses * 256; i += kThreads) (&sh[0][0][0])[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    // every lane of a warp runs the same trip count so the warp votes agree
    const int64_t begin = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t rounds = (n + stride - 1) / stride;
    for (int64_t r = 0; r < rounds; ++r) {
        const int64_t i = begin + r * stride;
        const bool valid = i < n;
        const K k = valid ? keys[i] : K(0);
        const bool full = __all_sync(0xffffffffu, valid);
        for (int p = 0; p < npasses; ++p) {
            const int sh_p = shift0 + 8 * p;
            const uint32_t d = digit_of(k, sh_p, digit_mask(sh_p, end_bit));
            const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
            if (full && __all_sync(0xffffffffu, d == d0)) {
                if (lane == 0) sh[warp][p][d] += 32u;
            } else if (valid) {
                atomicAdd(&sh[warp][p][d], 1u);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < npasses * 256; i += kThreads) {
        uint32_t v = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += (&sh[w][0][0])[i];
        if (v) atomicAdd(&hist[i], v);
    }
}

// How a tile of `count` elements at src splits for a bulk copy: `head`
// elements before the first 16-byte boundary, a `body` of whole 16-byte
// units, the rest after it; `shift` places the body on a 16-byte boundary
// of the destination (dst[shift + j] receives src[j]).
struct TileCopy {
    int shift, head, body;
};

template <typename T>
__device__ __forceinline__ TileCopy plan_copy(const T* src, int count) {
    constexpr int kPer = 16 / (int)sizeof(T);
    const int mis = (int)((reinterpret_cast<uintptr_t>(src) & 15u) / sizeof(T));
    TileCopy c;
    c.head = mis == 0 ? 0 : kPer - mis;
    if (c.head > count) c.head = count;
    c.body = (count - c.head) / kPer * kPer;
    c.shift = (kPer - c.head % kPer) % kPer;
    return c;
}

// The ends the bulk copy leaves (head and tail, under 16 bytes each), one
// element per thread: threads 0 .. head - 1 and 16 .. 16 + tail - 1.
template <typename T>
__device__ __forceinline__ void copy_ends(T* dst, const T* src, const TileCopy& c, int count,
                                          int tid) {
    const int tail = count - c.head - c.body;
    if (tid < c.head) dst[tid] = src[tid];
    const int t = tid - 16;
    if (t >= 0 && t < tail) dst[c.head + c.body + t] = src[c.head + c.body + t];
}

template <typename K, int ITEMS>
struct OnesweepSmem {
    K keys[kThreads * ITEMS];                             // the tile, reordered
    alignas(16) int32_t stage_vals[kThreads * ITEMS + 4];  // the tile's values as loaded
    int32_t vals[kThreads * ITEMS];                    // reordered values
    uint64_t bar;                                      // completes the bulk copies
    uint32_t warp_count[kWarps][256];  // per-warp digit counts, then warp prefixes
    uint32_t local_start[256];         // first slot of each digit in the tile
    int64_t out_base[256];             // output index of slot 0 of each digit
    int64_t scratch_a[32];
    int64_t scratch_b[32];
    uint32_t blk;
};

// WIDEN (32-bit keys only): the output key is the 64-bit key_in << 32 |
// wide_low[value] (into keys_wide instead of keys_out).
template <typename K, int ITEMS, bool IOTA, bool WIDEN = false>
__global__ void __launch_bounds__(kThreads, 4)
    k_onesweep(const K* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
               K* __restrict__ keys_out, int32_t* __restrict__ vals_out, int64_t n, int shift,
               uint32_t dmask, const uint32_t* __restrict__ hist, uint64_t* __restrict__ lookback,
               uint32_t* __restrict__ ticket, ErrorSink err,
               uint64_t* __restrict__ keys_wide = nullptr,
               const uint32_t* __restrict__ wide_low = nullptr) {
    __shared__ OnesweepSmem<K, ITEMS> sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        sm.blk = atomicAdd(ticket, 1u);
        mbar_init(&sm.bar, 1);
    }
    for (int i = tid; i < kWarps * 256; i += kThreads) (&sm.warp_count[0][0])[i] = 0;
    __syncthreads();
    const int64_t blk = sm.blk;
    const int64_t tile_base = blk * (kThreads * ITEMS);
    const int warp_local = warp * (kWarp * ITEMS);
    const int64_t warp_base = tile_base + warp_local;

    // 2. the tile's values into shared memory while the keys are ranked: the
    //    16-byte aligned middle by one bulk copy, the ragged ends (under 16
    //    bytes each) by plain loads; value j lands at stage_vals[shift + j].
    //    The keys come straight into registers, warp-striped.
    // (no keys for a virtual block past the end: a test of the timeout path
    // starts the tickets late)
    const int64_t left = n - tile_base;
    const int tile_n = left <= 0 ? 0 : (left < kThreads * ITEMS ? (int)left : kThreads * ITEMS);
    const TileCopy vc = IOTA ? TileCopy{0, 0, 0} : plan_copy(vals_in + tile_base, tile_n);
    const uint32_t tx = (uint32_t)(vc.body * 4);
    if (tid == 0 && tx) {
        mbar_expect_tx(&sm.bar, tx);
        bulk_to_shared(sm.stage_vals + vc.shift + vc.head, vals_in + tile_base + vc.head, tx,
                       &sm.bar);
    }
    if (!IOTA) copy_ends(sm.stage_vals + vc.shift, vals_in + tile_base, vc, tile_n, tid);

    K key[ITEMS];
    uint32_t rank[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const int local = warp_local + i * kWarp + lane;
        key[i] = local < tile_n ? keys_in[tile_base + local] : K(0);
    }

    // 3. rank within the warp, in element order (i, then lane): for each
    //    item the lowest lane of every group of equal digits adds the group
    //    size to the warp's count with one shared atomic, whose old value
    //    (broadcast to the group) is the group's base.  A warp's atomics on
    //    one address take effect in issue order, so an item need not wait for
    //    the previous one: each atomic's result is collected two items later.
    const unsigned lt = lanemask_lt();
    constexpr int kLag = 2;
    unsigned peers[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS + kLag; ++i) {
        if (i < ITEMS) {
            const bool valid = warp_base + i * kWarp + lane < n;
            const uint32_t d = valid ? digit_of(key[i], shift, dmask) : 0u;
            // every lane calls it; bits above a narrower digit are 0 in every lane
            const unsigned pm = digit_peers(d, valid, 8);
            peers[i] = valid ? pm : (1u << lane);
            uint32_t old = 0;
            if (valid && (peers[i] & lt) == 0)
                old = atomicAdd(&sm.warp_count[warp][d], (uint32_t)__popc(peers[i]));
            rank[i] = old;
        }
        if (i >= kLag) {
            const int j = i - kLag;
            rank[j] = __shfl_sync(0xffffffffu, rank[j], __ffs(peers[j]) - 1) +
                      __popc(peers[j] & lt);
        }
    }
    __syncthreads();

    // 4. per-digit totals, warp prefixes, publication and look-back
    const int d = tid;  // one digit per thread
    uint32_t total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        uint32_t c = sm.warp_count[w][d];
        sm.warp_count[w][d] = total;
        total += c;
    }
    uint64_t* mine = lookback + blk * 256 + d;
    st_relaxed_u64(mine, ((uint64_t)total << 2) | (blk == 0 ? kFlagPrefix : kFlagAggregate));

    int64_t all;
    const int64_t bucket_start = block_exclusive_scan<kThreads>(hist[d], sm.scratch_a, &all);

    // look back over the predecessors' words for this digit, four per round
    // trip (nearest first); a word not yet published is waited for
    int64_t excl = 0;
    if (blk > 0) {
        constexpr int kWin = 4;
        bool found = false;
        for (int64_t top = blk - 1; !found; top -= kWin) {
            uint64_t wv[kWin];
#pragma unroll
            for (int u = 0; u < kWin; ++u)
                wv[u] = top - u >= 0 ? ld_relaxed_u64(lookback + (top - u) * 256 + d) : 0;
#pragma unroll
            for (int u = 0; u < kWin; ++u) {
                if (found) break;
                const int64_t p = top - u;
                uint64_t v = wv[u];
                if ((v & kFlagMask) == 0) v = wait_published(lookback + p * 256 + d, err);
                excl += (int64_t)(v >> 2);
                found = (v & kFlagMask) == kFlagPrefix || p == 0;
            }
        }
        st_relaxed_u64(mine, ((uint64_t)(excl + total) << 2) | kFlagPrefix);
    }
    int64_t tile_count;
    const int64_t lstart = block_exclusive_scan<kThreads>(total, sm.scratch_b, &tile_count);
    sm.local_start[d] = (uint32_t)lstart;
    // the values' bulk copy has had the ranking and the look-back to land
    const bool ok = tx == 0 || mbar_wait(&sm.bar, 0, kBulkPolls);
    sm.out_base[d] = bucket_start + excl - lstart;
    if (__syncthreads_or(!ok)) {
        // the copy never completed: report, give it one more bounded wait
        // (it writes this block's shared memory), and stop
        if (tid == 0) err.raise(GS_ERR_TIMEOUT);
        mbar_wait(&sm.bar, 0, kBulkPolls);
        return;
    }

    // 5. reorder by digit in shared memory, then write out bucket runs
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        if (warp_base + i * kWarp + lane < n) {
            const uint32_t dd = digit_of(key[i], shift, dmask);
            const uint32_t pos = sm.local_start[dd] + sm.warp_count[warp][dd] + rank[i];
            const int local = warp_local + i * kWarp + lane;
            sm.keys[pos] = key[i];
            sm.vals[pos] = IOTA ? (int32_t)(tile_base + local) : sm.stage_vals[vc.shift + local];
        }
    }
    __syncthreads();
    // unrolled over the thread's (at most ITEMS) slots, so the loads (and the
    // gathers of the widening pass) of all of them are in flight together
    const int cnt = (int)tile_count;
    uint32_t low[ITEMS];
    if (WIDEN) {
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
            const int j = it * kThreads + tid;
            low[it] = j < cnt ? wide_low[sm.vals[j]] : 0u;
        }
    }
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int j = it * kThreads + tid;
        if (j >= cnt) break;
        const K k = sm.keys[j];
        const int64_t o = sm.out_base[digit_of(k, shift, dmask)] + j;
        // in range by construction when the histogram matches the keys; the
        // test only matters after a timed-out wait or an inconsistent input
        if ((uint64_t)o < (uint64_t)n) {
            const int32_t v = sm.vals[j];
            if (WIDEN) keys_wide[o] = ((uint64_t)k << 32) | low[it];
            else keys_out[o] = k;
            vals_out[o] = v;
        } else {
            err.raise(GS_ERR_COUNT_MISMATCH);
        }
    }
}

int hist_grid(int64_t n) {
    int64_t g = (n + kThreads * 16 - 1) / (kThreads * 16);
    if (g < 1) g = 1;
    if (g > 152 * 4) g = 152 * 4;
    return (int)g;
}

}  // namespace

template <typename K>
void digit_hist(const K* keys, int64_t n, int shift0, int end_bit, uint32_t* hist,
                cudaStream_t s) {
    const int npasses = (end_bit - shift0 + 7) / 8;
    if (n <= 0 || npasses <= 0) return;
    for (int p0 = 0; p0 < npasses; p0 += kHistPasses) {
        const int np = npasses - p0 < kHistPasses ? npasses - p0 : kHistPasses;
        k_digit_hist<K><<<hist_grid(n), kThreads, 0, s>>>(keys, n, shift0 + 8 * p0, np, end_bit,
                                                         hist + 256 * p0);
    }
}

void launch_digit_hist_u64(const uint64_t* keys, int64_t n, int shift0, int end_bit,
                           uint32_t* hist, cudaStream_t s) {
    digit_hist<uint64_t>(keys, n, shift0, end_bit, hist, s);
}

void launch_digit_hist_u32(const uint32_t* keys, int64_t n, int shift0, int end_bit,
                           uint32_t* hist, cudaStream_t s) {
    digit_hist<uint32_t>(keys, n, shift0, end_bit, hist, s);
}

void launch_onesweep_u64(const uint64_t* keys_in, const int32_t* vals_in, uint64_t* keys_out,
                         int32_t* vals_out, int64_t n, int shift, int end_bit,
                         const uint32_t* hist,
                         LookbackScratch lb, int32_t* abort_flag, int32_t* d_status,
                         cudaStream_t s, int spin_limit) {
    if (n <= 0) return;
    const int64_t blocks = sort_blocks(n, kTile64);
    ErrorSink err{abort_flag, d_status};
    if (spin_limit > 0) err.spin_limit = spin_limit;
    const uint32_t dm = digit_mask(shift, end_bit);
    if (vals_in)
        k_onesweep<uint64_t, kItems64, false><<<(unsigned)blocks, kThreads, 0, s>>>(
            keys_in, vals_in, keys_out, vals_out, n, shift, dm, hist, lb.words, lb.ticket, err);
    else
        k_onesweep<uint64_t, kItems64, true><<<(unsigned)blocks, kThreads, 0, s>>>(
            keys_in, vals_in, keys_out, vals_out, n, shift, dm, hist, lb.words, lb.ticket, err);
}

void launch_onesweep_u32(const uint32_t* keys_in, const int32_t* vals_in, uint32_t* keys_out,
                         int32_t* vals_out, int64_t n, int shift, int end_bit,
                         const uint32_t* hist,
                         LookbackScratch lb, int32_t* abort_flag, int32_t* d_status,
                         cudaStream_t s) {
    if (n <= 0) return;
    const int64_t blocks = sort_blocks(n, kTile32);
    ErrorSink err{abort_flag, d_status};
    const uint32_t dm = digit_mask(shift, end_bit);
    if (vals_in)
        k_onesweep<uint32_t, kItems32, false><<<(unsigned)blocks, kThreads, 0, s>>>(
            keys_in, vals_in, keys_out, vals_out, n, shift, dm, hist, lb.words, lb.ticket, err);
    else
        k_onesweep<uint32_t, kItems32, true><<<(unsigned)blocks, kThreads, 0, s>>>(
            keys_in, vals_in, keys_out, vals_out, n, shift, dm, hist, lb.words, lb.ticket, err);
}

void launch_onesweep_u32_widen(const uint32_t* keys_in, const int32_t* vals_in,
                               uint64_t* keys_out, int32_t* vals_out, int64_t n, int shift,
                               int end_bit, const uint32_t* hist, const uint32_t* wide_low,
                               LookbackScratch lb, int32_t* abort_flag, int32_t* d_status,
                               cudaStream_t s) {
    if (n <= 0) return;
    const int64_t blocks = sort_blocks(n, kTile32);
    ErrorSink err{abort_flag, d_status};
    const uint32_t dm = digit_mask(shift, end_bit);
    k_onesweep<uint32_t, kItems32, false, true><<<(unsigned)blocks, kThreads, 0, s>>>(
        keys_in, vals_in, nullptr, vals_out, n, shift, dm, hist, lb.words, lb.ticket, err,
        keys_out, wide_low);
}

}  // namespace gs
