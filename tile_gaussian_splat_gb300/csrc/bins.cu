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
//   k_bin_sort  one block per bin: its entries, keyed (depth bits << 32 |
//               splat index), are sorted by a bitonic network (short strides
//               in registers with warp shuffles, long ones in shared memory),
//               written back in order and followed by -1s.  The result does
//               not depend on the append order.
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kFillThreads = 256;
constexpr int kFillSplats = 2 * kFillThreads;
constexpr int kBinSortThreads = 256;

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
    for (int q = tid; q < total; q += kFillThreads) {
        int lo = 0, hi = kFillSplats - 1;  // owner: first o with incl[o] > q
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sm.incl[mid] > q) hi = mid;
            else lo = mid + 1;
        }
        const int o = lo;
        const int li = q - (o == 0 ? 0 : sm.incl[o - 1]);
        const int dy = li / sm.w[o];
        const int64_t t = sm.tile0[o] + (int64_t)(sm.y0[o] + dy) * tile_width + sm.x0[o] +
                          (li - dy * sm.w[o]);
        const int k = atomicAdd(&counts[t], 1);
        if (k < capacity) bins[t * capacity + k] = sm.sid[o];
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

// Bitonic sort of a bin's keys in shared memory over n2 = the next power of
// two (at least 64) of the bin's entry count, padded with all-ones keys that
// sort last.  Strides below 64 run in registers with warp shuffles on
// 64-element chunks; only the longer strides go through shared memory with
// a block barrier.
__global__ void __launch_bounds__(kBinSortThreads)
    k_bin_sort(const uint32_t* __restrict__ depth_bits, int64_t nbins, int capacity,
               int32_t* __restrict__ bins, const int32_t* __restrict__ counts,
               int32_t* d_status) {
    extern __shared__ uint64_t keys[];
    constexpr int kW = kBinSortThreads / kWarp;
    const int64_t b = blockIdx.x;
    if (b >= nbins) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = counts[b];
    if (total > capacity && tid == 0) report(d_status, GS_ERR_CAPACITY);
    const int cnt = total < capacity ? total : capacity;
    int32_t* bin = bins + b * capacity;
    int n2 = 64;
    while (n2 < cnt) n2 <<= 1;
    if (cnt > 1) {
        for (int k = tid; k < n2; k += kBinSortThreads) {
            uint64_t key = ~0ull;
            if (k < cnt) {
                const uint32_t id = (uint32_t)bin[k];
                key = ((uint64_t)depth_bits[id] << 32) | id;
            }
            keys[k] = key;
        }
        __syncthreads();
        for (int size = 2; size <= n2; size <<= 1) {
            // shared-memory stages of this level (strides >= 64)
            for (int stride = size >> 1; stride >= 64; stride >>= 1) {
                for (int p = tid; p < (n2 >> 1); p += kBinSortThreads) {
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
        for (int k = tid; k < cnt; k += kBinSortThreads) bin[k] = (int32_t)(uint32_t)keys[k];
    }
    for (int k = cnt + tid; k < capacity; k += kBinSortThreads) bin[k] = -1;
}

}  // namespace

int bin_sort_smem_bytes(int capacity) {
    int n2 = 64;
    while (n2 < capacity) n2 <<= 1;
    return n2 * (int)sizeof(uint64_t);
}

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
            tile_width, tile_height,
            capacity, bins, counts);
    }
    const int smem = bin_sort_smem_bytes(capacity);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_bin_sort, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
        return GS_ERR_CUDA;
    k_bin_sort<<<(unsigned)nbins, kBinSortThreads, smem, s>>>(
        reinterpret_cast<const uint32_t*>(depths), nbins, capacity, bins, counts, d_status);
    return GS_OK;
}

}  // namespace gs
