// Fixed-capacity per-tile bin lists: the bin_faces layout of the pytorch3d
// fine rasterizer (rasterize_meshes.cu, RasterizeMeshesFineCudaKernel:
// (N, BH, BW, M) int32, -1 after a bin's entries), filled with the splats
// that cover each tile in compositing order -- ascending depth bits, ties by
// splat index, i.e. each tile's slice of the stable sort of the 64-bit keys
// -- without a global sort.
//
//   k_bin_fill  512 splats per block, index order: the block's (splat, tile)
//               pairs are expanded cooperatively (as in k_isect_emit) and
//               each appends its splat to the tile's bin with one atomic on
//               the tile's counter.  The order inside a bin is the order the
//               atomics happened to take.
//   k_bin_merge one block per bin of at most kSmallBin entries (every bin when
//               the capacity allows no more): its entries, keyed (depth bits
//               << 32 | splat index), are merge-sorted in shared memory --
//               64-entry chunks in registers with warp shuffles, then runs
//               merged pairwise, each entry placed by a binary search in the
//               partner run -- written back in order and followed by -1s.
//   k_bin_merge_large  the larger bins, 1024 threads, as many blocks as fit
//               on the GPU walking the bins in turn (the small ones skipped):
//               runs of eight sorted in registers, then merged pairwise with
//               each thread writing several consecutive entries from one
//               binary search (merge path); above kMergeMaxCapacity (two key
//               buffers no longer fit in shared memory) a bitonic network on
//               one power-of-two buffer instead.
//   The result does not depend on the append order.
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kFillThreads = 256;
constexpr int kFillSplats = 2 * kFillThreads;
constexpr int kBinSortThreads = 256;       // k_bin_merge
constexpr int kLargeBinThreads = 1024;     // k_bin_merge_large
constexpr int kSmallBin = 2048;            // entries of the largest bin k_bin_merge sorts
// Largest capacity merge-sorted by k_bin_merge_large (two buffers of 64-bit
// keys in shared memory); above it a bitonic network on one buffer.
constexpr int kMergeMaxCapacity = 14336;

struct FillSmem {
    int32_t incl[kFillSplats];  // inclusive prefix of pair counts in the chunk
    int32_t x0[kFillSplats];
    int32_t y0[kFillSplats];
    int32_t w[kFillSplats];     // rect width in tiles
    int64_t tile0[kFillSplats];  // camera * tiles per camera
    int32_t sid[kFillSplats];
    int64_t scratch[32];
};

__global__ void __launch_bounds__(kFillThreads)
    k_bin_fill(const float* __restrict__ means2d, const float* __restrict__ radii, int elliptical,
               int64_t CN, int N, float ts, float inv_ts, int tile_width, int tile_height,
               int capacity,
               int32_t* __restrict__ bins, int32_t* __restrict__ counts) {
    __shared__ FillSmem sm;
    const int tid = threadIdx.x;
    const int64_t per_camera = (int64_t)tile_width * tile_height;
    int cnt[2];
    int64_t local = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int slot = 2 * tid + u;
        const int64_t i = (int64_t)blockIdx.x * kFillSplats + slot;
        cnt[u] = 0;
        if (i < CN) {
            const float2 m = reinterpret_cast<const float2*>(means2d)[i];
            float rx, ry;
            if (elliptical) {
                const float2 rr = reinterpret_cast<const float2*>(radii)[i];
                rx = rr.x;
                ry = rr.y;
            } else {
                rx = ry = radii[i];
            }
            const Rect r = splat_rect(m.x, m.y, rx, ry, ts, inv_ts, tile_width, tile_height);
            cnt[u] = (r.x1 - r.x0) * (r.y1 - r.y0);
            sm.x0[slot] = r.x0;
            sm.y0[slot] = r.y0;
            sm.w[slot] = r.x1 - r.x0;
            sm.tile0[slot] = (i / N) * per_camera;
            sm.sid[slot] = (int32_t)i;
        }
        local += cnt[u];
    }
    int64_t chunk_total;
    const int64_t excl = block_exclusive_scan<kFillThreads>(local, sm.scratch, &chunk_total);
    sm.incl[2 * tid] = (int32_t)(excl + cnt[0]);
    sm.incl[2 * tid + 1] = (int32_t)(excl + cnt[0] + cnt[1]);
    __syncthreads();
    const int total = (int)chunk_total;
    // four pairs per thread and round: their owner searches and atomics are
    // issued together, so the atomics' returns overlap
    constexpr int U = 4;
    for (int q0 = tid; q0 < total; q0 += U * kFillThreads) {
        int64_t t[U];
        int32_t id[U], k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = q0 + u * kFillThreads;
            t[u] = -1;
            if (q < total) {
                int lo = 0, hi = kFillSplats - 1;  // owner: first o with incl[o] > q
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (sm.incl[mid] > q) hi = mid;
                    else lo = mid + 1;
                }
                const int o = lo;
                const int li = q - (o == 0 ? 0 : sm.incl[o - 1]);
                const int dy = li / sm.w[o];
                t[u] = sm.tile0[o] + (int64_t)(sm.y0[o] + dy) * tile_width + sm.x0[o] +
                       (li - dy * sm.w[o]);
                id[u] = sm.sid[o];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) k[u] = t[u] >= 0 ? atomicAdd(&counts[t[u]], 1) : capacity;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (k[u] < capacity) bins[t[u] * capacity + k[u]] = id[u];
    }
}

// One compare-exchange of a bitonic stage between lanes: element i (this
// lane's) and i ^ stride (lane ^ stride, stride < 32) of a 64-element chunk;
// ascending where bit `size` of i is clear.
__device__ __forceinline__ uint64_t cas_lanes(uint64_t x, int i, int size, int stride, int lane) {
    const uint64_t y = ((uint64_t)__shfl_xor_sync(0xffffffffu, (uint32_t)(x >> 32), stride) << 32) |
                       __shfl_xor_sync(0xffffffffu, (uint32_t)x, stride);
    const bool asc = (i & size) == 0;
    const bool lower = (lane & stride) == 0;
    const uint64_t lo = x < y ? x : y, hi = x < y ? y : x;
    return lower == asc ? lo : hi;
}

// Strides 32 .. 1 of bitonic level `size` (or all levels up to 64 when
// full) on a 64-element chunk held as x0 = element lane, x1 = element
// lane + 32.
__device__ __forceinline__ void chunk_stages(uint64_t& x0, uint64_t& x1, int base, int size_lo,
                                             int size_hi, int lane) {
    for (int size = size_lo; size <= size_hi; size <<= 1) {
        for (int stride = (size < 64 ? size : 64) >> 1; stride > 0; stride >>= 1) {
            if (stride == 32) {
                const bool asc = ((base + lane) & size) == 0;
                if ((x0 > x1) == asc) {
                    const uint64_t t = x0;
                    x0 = x1;
                    x1 = t;
                }
            } else {
                x0 = cas_lanes(x0, base + lane, size, stride, lane);
                x1 = cas_lanes(x1, base + lane + 32, size, stride, lane);
            }
        }
    }
}

// Number of entries of the sorted run[0 .. n) below x (its lower bound).
__device__ __forceinline__ int count_below(const uint64_t* run, int n, uint64_t x) {
    int lo = 0;
    while (n > 0) {
        const int half = n >> 1;
        if (run[lo + half] < x) {
            lo += half + 1;
            n -= half + 1;
        } else {
            n = half;
        }
    }
    return lo;
}

__device__ __forceinline__ uint64_t bin_key(const uint32_t* depth_bits, const int32_t* bin, int k) {
    const uint32_t id = (uint32_t)bin[k];
    return ((uint64_t)depth_bits[id] << 32) | id;
}

// Merge sort of bin[0 .. cnt) (cnt >= 2) by key, in place, through the two
// shared-memory buffers src and dst of at least cnt keys each.  Keys are
// unique (a splat covers a tile once), so an entry's place in a merged run is
// its place in its own run plus the number of the partner run's entries below
// it.  Ends with a block barrier.
template <int THREADS>
__device__ void merge_sort_bin(const uint32_t* __restrict__ depth_bits, int32_t* bin, int cnt,
                               uint64_t* src, uint64_t* dst) {
    constexpr int kW = THREADS / kWarp;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int c = warp; c * 64 < cnt; c += kW) {
        const int i0 = c * 64 + lane, i1 = i0 + 32;
        uint64_t x0 = i0 < cnt ? bin_key(depth_bits, bin, i0) : ~0ull;  // padding sorts last
        uint64_t x1 = i1 < cnt ? bin_key(depth_bits, bin, i1) : ~0ull;
        chunk_stages(x0, x1, 0, 2, 64, lane);  // all levels up to 64, ascending
        if (i0 < cnt) src[i0] = x0;
        if (i1 < cnt) src[i1] = x1;
    }
    __syncthreads();
    for (int L = 64; L < cnt; L <<= 1) {
        for (int i = tid; i < cnt; i += THREADS) {
            const uint64_t x = src[i];
            const int start = i & ~(L - 1);       // this run
            const int pair = start & ~(2 * L - 1);  // the merged run
            const bool left = start == pair;
            const int p0 = left ? start + L : pair;  // the partner run [p0, p1)
            const int p1 = left ? min(start + 2 * L, cnt) : start;
            const int below = p1 > p0 ? count_below(src + p0, p1 - p0, x) : 0;
            dst[pair + (i - start) + below] = x;
        }
        __syncthreads();
        uint64_t* t = src;
        src = dst;
        dst = t;
    }
    for (int k = tid; k < cnt; k += THREADS) bin[k] = (int32_t)(uint32_t)src[k];
    __syncthreads();
}

// Compare-exchange of two registers: a gets the smaller key.
__device__ __forceinline__ void order2(uint64_t& a, uint64_t& b) {
    const uint64_t lo = a < b ? a : b, hi = a < b ? b : a;
    a = lo;
    b = hi;
}

// Batcher's odd-even merge sort of eight keys held in registers (19
// compare-exchanges).
__device__ __forceinline__ void sort8(uint64_t (&v)[8]) {
    order2(v[0], v[1]); order2(v[2], v[3]); order2(v[4], v[5]); order2(v[6], v[7]);
    order2(v[0], v[2]); order2(v[1], v[3]); order2(v[4], v[6]); order2(v[5], v[7]);
    order2(v[1], v[2]); order2(v[5], v[6]);
    order2(v[0], v[4]); order2(v[1], v[5]); order2(v[2], v[6]); order2(v[3], v[7]);
    order2(v[2], v[4]); order2(v[3], v[5]);
    order2(v[1], v[2]); order2(v[3], v[4]); order2(v[5], v[6]);
}

// The same sort for long bins, where a thread has several entries per
// merge: runs of eight are sorted in registers; then runs of 8, 16, ... are
// merged pairwise, each thread writing E consecutive entries of the merged
// runs -- it finds where its first entry's diagonal crosses the two runs by
// binary search (the merge path) and merges sequentially from there.  E is
// odd (so a warp's 8-byte stores spread over the banks) and large enough
// that one pass of the block covers the bin (cnt <= THREADS * E).  Buffers
// of at least cnt keys rounded up to 8.  Ends with a block barrier.
template <int THREADS>
__device__ void merge_path_sort_bin(const uint32_t* __restrict__ depth_bits, int32_t* bin,
                                    int cnt, uint64_t* src, uint64_t* dst) {
    const int tid = threadIdx.x;
    const int E = max(7, (cnt + THREADS - 1) / THREADS) | 1;
    for (int r = tid; r * 8 < cnt; r += THREADS) {
        uint64_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = r * 8 + j < cnt ? bin_key(depth_bits, bin, r * 8 + j) : ~0ull;  // padding last
        sort8(v);
        ulonglong2* out = reinterpret_cast<ulonglong2*>(src + r * 8);
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j] = make_ulonglong2(v[2 * j], v[2 * j + 1]);
    }
    __syncthreads();
    for (int L = 8; L < cnt; L <<= 1) {
        for (int o0 = tid * E; o0 < cnt; o0 += THREADS * E) {
            const int o1 = min(o0 + E, cnt);
            int o = o0;
            while (o < o1) {  // a step may cross into the next pair of runs
                const int pair = o & ~(2 * L - 1);
                const int la = min(L, cnt - pair);             // run A = src[pair, +la)
                const int lb = max(0, min(L, cnt - pair - L));  // run B right after it
                const int seg = min(o1, pair + la + lb);
                const uint64_t* A = src + pair;
                const uint64_t* B = A + la;
                const int d = o - pair;  // entries of the merged run before o
                int lo = max(0, d - lb), hi = min(d, la);
                while (lo < hi) {  // entries of A among those d
                    const int mid = (lo + hi) >> 1;
                    if (A[mid] < B[d - 1 - mid]) lo = mid + 1;
                    else hi = mid;
                }
                int ia = lo, ib = d - lo;
                uint64_t va = ia < la ? A[ia] : ~0ull, vb = ib < lb ? B[ib] : ~0ull;
                for (; o < seg; ++o) {
                    const bool ta = va < vb;
                    dst[o] = ta ? va : vb;
                    ia += ta;
                    ib += !ta;
                    const bool more = ta ? ia < la : ib < lb;
                    const uint64_t x = more ? (ta ? A[ia] : B[ib]) : ~0ull;
                    va = ta ? x : va;
                    vb = ta ? vb : x;
                }
            }
        }
        __syncthreads();
        uint64_t* t = src;
        src = dst;
        dst = t;
    }
    for (int k = tid; k < cnt; k += THREADS) bin[k] = (int32_t)(uint32_t)src[k];
    __syncthreads();
}

// Bitonic sort of bin[0 .. cnt) (cnt >= 2) by key over n2 = the next power
// of two (at least 64) of cnt, padded with all-ones keys that sort last, in
// one shared-memory buffer of n2 keys.  Strides below 64 run in registers
// with warp shuffles on 64-element chunks; only the longer strides go
// through shared memory with a block barrier.  Ends with a block barrier.
template <int THREADS>
__device__ void bitonic_sort_bin(const uint32_t* __restrict__ depth_bits, int32_t* bin, int cnt,
                                 uint64_t* keys) {
    constexpr int kW = THREADS / kWarp;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int n2 = 64;
    while (n2 < cnt) n2 <<= 1;
    for (int k = tid; k < n2; k += THREADS) keys[k] = k < cnt ? bin_key(depth_bits, bin, k) : ~0ull;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride >= 64; stride >>= 1) {
            for (int p = tid; p < (n2 >> 1); p += THREADS) {
                const int lo = ((p / stride) * 2 * stride) + (p % stride);
                const int hi = lo + stride;
                const bool ascending = (lo & size) == 0;
                const uint64_t x = keys[lo], y = keys[hi];
                if ((x > y) == ascending) {
                    keys[lo] = y;
                    keys[hi] = x;
                }
            }
            __syncthreads();
        }
        // the rest in registers: all levels up to 64 at once, then per level
        const int size_lo = size <= 64 ? 2 : size, size_hi = size <= 64 ? 64 : size;
        for (int c = warp; c < n2 / 64; c += kW) {
            uint64_t x0 = keys[c * 64 + lane], x1 = keys[c * 64 + lane + 32];
            chunk_stages(x0, x1, c * 64, size_lo, size_hi, lane);
            keys[c * 64 + lane] = x0;
            keys[c * 64 + lane + 32] = x1;
        }
        __syncthreads();
        if (size < 64) size = 64;  // levels 2..64 are done
    }
    for (int k = tid; k < cnt; k += THREADS) bin[k] = (int32_t)(uint32_t)keys[k];
    __syncthreads();
}

// Bin b's entry count (reporting an overflow) and its -1 tail.
template <int THREADS>
__device__ __forceinline__ int bin_entries(int64_t b, int capacity, const int32_t* counts,
                                           int32_t* d_status) {
    const int total = counts[b];
    if (total > capacity && threadIdx.x == 0) report(d_status, GS_ERR_CAPACITY);
    return total < capacity ? total : capacity;
}

template <int THREADS>
__device__ __forceinline__ void fill_tail(int32_t* bin, int cnt, int capacity) {
    for (int k = cnt + (int)threadIdx.x; k < capacity; k += THREADS) bin[k] = -1;
}

// One block per bin; bins of more than kSmallBin entries are left to
// k_bin_merge_large.  Shared memory: two buffers of min(capacity, kSmallBin)
// keys, rounded up to 64.
__global__ void __launch_bounds__(kBinSortThreads)
    k_bin_merge(const uint32_t* __restrict__ depth_bits, int64_t nbins, int capacity,
                int32_t* __restrict__ bins, const int32_t* __restrict__ counts,
                int32_t* d_status) {
    extern __shared__ __align__(16) uint64_t keys[];
    const int64_t b = blockIdx.x;
    if (b >= nbins) return;
    const int cnt = bin_entries<kBinSortThreads>(b, capacity, counts, d_status);
    if (cnt > kSmallBin) return;
    int32_t* bin = bins + b * capacity;
    const int stride = ((capacity < kSmallBin ? capacity : kSmallBin) + 63) & ~63;
    if (cnt > 1) merge_sort_bin<kBinSortThreads>(depth_bits, bin, cnt, keys, keys + stride);
    fill_tail<kBinSortThreads>(bin, cnt, capacity);
}

// Bins of more than kSmallBin entries, walked in turn by a grid of a few
// blocks per SM.  MERGE: two buffers of capacity keys (rounded up to 64);
// otherwise one power-of-two buffer for the bitonic network.
template <bool MERGE>
__global__ void __launch_bounds__(kLargeBinThreads)
    k_bin_merge_large(const uint32_t* __restrict__ depth_bits, int64_t nbins, int capacity,
                      int32_t* __restrict__ bins, const int32_t* __restrict__ counts,
                      int32_t* d_status) {
    extern __shared__ __align__(16) uint64_t keys[];
    for (int64_t b = blockIdx.x; b < nbins; b += gridDim.x) {
        const int cnt = bin_entries<kLargeBinThreads>(b, capacity, counts, d_status);
        if (cnt <= kSmallBin) continue;
        int32_t* bin = bins + b * capacity;
        if (MERGE)
            merge_path_sort_bin<kLargeBinThreads>(depth_bits, bin, cnt, keys,
                                                  keys + ((capacity + 63) & ~63));
        else
            bitonic_sort_bin<kLargeBinThreads>(depth_bits, bin, cnt, keys);
        fill_tail<kLargeBinThreads>(bin, cnt, capacity);
    }
}

}  // namespace

namespace {

int large_smem_bytes(int capacity) {
    if (capacity <= kMergeMaxCapacity) return 2 * ((capacity + 63) & ~63) * 8;
    int n2 = 64;
    while (n2 < capacity) n2 <<= 1;
    return n2 * 8;
}

template <typename K>
int launch_sized(K kern, unsigned grid, int threads, int smem, cudaStream_t s,
                 const uint32_t* depth_bits, int64_t nbins, int capacity, int32_t* bins,
                 const int32_t* counts, int32_t* d_status) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
        return GS_ERR_CUDA;
    kern<<<grid, threads, smem, s>>>(depth_bits, nbins, capacity, bins, counts, d_status);
    return GS_OK;
}

}  // namespace

int launch_bin_splats(const float* means2d, const float* radii, int elliptical,
                      const float* depths, int C, int N, int tile_size, int tile_width,
                      int tile_height, int capacity, int32_t* bins, int32_t* counts,
                      int32_t* d_status, cudaStream_t s) {
    const int64_t CN = (int64_t)C * N;
    const int64_t nbins = (int64_t)C * tile_width * tile_height;
    if (CN > 0) {
        const int64_t chunks = (CN + kFillSplats - 1) / kFillSplats;
        k_bin_fill<<<(unsigned)chunks, kFillThreads, 0, s>>>(
            means2d, radii, elliptical, CN, N, (float)tile_size, exact_tile_inverse(tile_size),
            tile_width, tile_height, capacity, bins, counts);
    }
    const uint32_t* depth_bits = reinterpret_cast<const uint32_t*>(depths);
    const int small = 2 * (((capacity < kSmallBin ? capacity : kSmallBin) + 63) & ~63) * 8;
    int rc = launch_sized(k_bin_merge, (unsigned)nbins, kBinSortThreads, small, s, depth_bits,
                          nbins, capacity, bins, counts, d_status);
    if (rc != GS_OK || capacity <= kSmallBin) return rc;
    // the larger bins: a grid of as many blocks as fit on the GPU at once
    const int large = large_smem_bytes(capacity);
    const bool merge = capacity <= kMergeMaxCapacity;
    auto* kern = merge ? k_bin_merge_large<true> : k_bin_merge_large<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, large) !=
        cudaSuccess)
        return GS_ERR_CUDA;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLargeBinThreads, large) !=
            cudaSuccess)
        return GS_ERR_CUDA;
    const int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    return launch_sized(kern, (unsigned)(grid < nbins ? grid : nbins), kLargeBinThreads, large,
                        s, depth_bits, nbins, capacity, bins, counts, d_status);
}

}  // namespace gs
