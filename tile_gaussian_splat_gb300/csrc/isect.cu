// Tile intersection (gsplat 1.0.0, intersections.c: gs_bounds,
// gs_isect_tiles) and tile ranges (gs_offset_encode) on sm_103a.
//
//   k_isect_count  one thread per splat: rect, tiles_per_gauss, block sum
//                  added to the total (size query).
//   k_rect_hist    one pass over the splats in index order: each splat's
//                  tile rect into a 16-byte record (so the emission, which
//                  visits splats in depth order, gathers one sector per splat)
//                  and the histograms of the four 8-bit digits of the depth
//                  bits for the depth sort.
//   k_isect_emit   two splats per thread of a 512-splat chunk taken in
//                  ticket order; a block scan of the counts plus a decoupled
//                  look-back over earlier chunks gives each splat's first
//                  output slot; then each warp writes the keys of its 64
//                  splats 32 consecutive keys at a time (a key's splat comes
//                  from the round's splat-start bits), so stores are
//                  coalesced whatever the per-splat counts are.  Optionally
//                  also histograms the 8-bit digits of the key's upper word
//                  for the radix passes that follow.
//                  With 32-bit keys (sorted path) it writes only the camera |
//                  tile word; the depth bits are attached by the last radix
//                  pass (or k_widen), which reads them from the depths array
//                  through L2.
//   k_tile_ranges  four consecutive sorted keys per thread (two 16-byte
//                  loads when the keys are 16-byte aligned; the key before
//                  them comes from the neighbouring lane): where the tile id
//                  changes, the tiles in between get the key's position.
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kThreads = kIsectThreads;

__global__ void __launch_bounds__(kThreads)
    k_isect_count(const float* __restrict__ means2d, const float* __restrict__ radii,
                  int elliptical, int64_t CN, float ts, float inv_ts, int tile_width,
                  int tile_height, int32_t* __restrict__ tiles_per_gauss,
                  unsigned long long* __restrict__ total) {
    __shared__ int64_t scratch[32];
    constexpr int U = 4;  // splats per thread and round, their loads issued together
    int64_t local = 0;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; i0 < CN; i0 += U * stride) {
        float2 m[U], r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + u * stride;
            m[u] = make_float2(0.0f, 0.0f);
            r[u] = make_float2(0.0f, 0.0f);
            if (i < CN) {
                m[u] = reinterpret_cast<const float2*>(means2d)[i];
                if (elliptical) {
                    r[u] = reinterpret_cast<const float2*>(radii)[i];
                } else {
                    r[u].x = r[u].y = radii[i];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + u * stride;
            if (i >= CN) break;
            const Rect rc = splat_rect(m[u].x, m[u].y, r[u].x, r[u].y, ts, inv_ts, tile_width,
                                       tile_height);
            const int cnt = (rc.x1 - rc.x0) * (rc.y1 - rc.y0);
            if (tiles_per_gauss) tiles_per_gauss[i] = cnt;
            local += cnt;
        }
    }
    int64_t sum;
    block_exclusive_scan<kThreads>(local, scratch, &sum);
    if (threadIdx.x == 0 && sum) atomicAdd(total, (unsigned long long)sum);
}

__global__ void __launch_bounds__(kThreads)
    k_rect_hist(const float* __restrict__ means2d, const float* __restrict__ radii,
                int elliptical, const uint32_t* __restrict__ dbits, int64_t CN, float ts,
                float inv_ts, int tile_width, int tile_height, int4* __restrict__ rects,
                uint32_t* __restrict__ hist) {
    constexpr int kW = kThreads / kWarp;
    // one private histogram per warp and digit; a digit shared by the whole
    // warp (common in the high bits) is added once by lane 0
    __shared__ uint32_t sh[kW][4][256];
    for (int i = threadIdx.x; i < kW * 4 * 256; i += kThreads) (&sh[0][0][0])[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t begin = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    constexpr int U = 2;  // splats per thread and round, their loads issued together
    // same trip count in every lane
    const int64_t rounds = (CN + U * stride - 1) / (U * stride);
    for (int64_t r = 0; r < rounds; ++r) {
        float2 m[U], rr[U];
        uint32_t key[U];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = begin + (r * U + u) * stride;
            valid[u] = i < CN;
            m[u] = make_float2(0.0f, 0.0f);
            rr[u] = make_float2(0.0f, 0.0f);
            key[u] = 0;
            if (valid[u]) {
                m[u] = reinterpret_cast<const float2*>(means2d)[i];
                if (elliptical) {
                    rr[u] = reinterpret_cast<const float2*>(radii)[i];
                } else {
                    rr[u].x = rr[u].y = radii[i];
                }
                key[u] = dbits[i];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = begin + (r * U + u) * stride;
            if (valid[u]) {
                const Rect rc = splat_rect(m[u].x, m[u].y, rr[u].x, rr[u].y, ts, inv_ts,
                                           tile_width, tile_height);
                rects[i] = make_int4(rc.x0, rc.y0, rc.x1, rc.y1);
            }
            const bool full = __all_sync(0xffffffffu, valid[u]);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint32_t d = (key[u] >> (8 * p)) & 0xffu;
                const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
                if (full && __all_sync(0xffffffffu, d == d0)) {
                    if (lane == 0) sh[warp][p][d] += 32u;
                } else if (valid[u]) {
                    atomicAdd(&sh[warp][p][d], 1u);
                }
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 256; i += kThreads) {
        uint32_t v = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) v += (&sh[w][0][0])[i];
        if (v) atomicAdd(&hist[i], v);
    }
}

// Widens sorted 32-bit camera|tile keys to the 64-bit keys (depth bits from
// the splat's depth) when no radix pass over them is needed.
__global__ void __launch_bounds__(kThreads)
    k_widen(const uint32_t* __restrict__ k32, const int32_t* __restrict__ v32,
            const uint32_t* __restrict__ dbits, int64_t n, uint64_t* __restrict__ keys,
            int32_t* __restrict__ ids) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
        const int32_t v = v32[i];
        keys[i] = ((uint64_t)k32[i] << 32) | dbits[v];
        ids[i] = v;
    }
}

constexpr int kEmitSplats = kEmitChunk;  // splats per emit block (2 per thread)

struct EmitSmem {
    int32_t incl[kEmitSplats];  // inclusive prefix of counts in the chunk
    int32_t x0[kEmitSplats];    // rect origin in tiles
    int32_t y0[kEmitSplats];
    int32_t w[kEmitSplats];     // rect width in tiles
    uint32_t upper[kEmitSplats];  // camera << tile_bits
    uint32_t dbits[kEmitSplats];
    int32_t sid[kEmitSplats];
    float rw[kEmitSplats];      // 1 / rect width
    int16_t owner[kThreads / kWarp][kWarp];  // per warp: splat slot starting at R + i
    uint32_t hist[4][256];
    int64_t scratch[32];
    int64_t base;
    uint32_t blk;
};

// One count per valid lane into bins[d].  A digit shared by every valid lane
// of the warp (the high digit of neighbouring tiles, mostly) is added once;
// otherwise each lane adds its own (neighbouring tiles' low digits rarely
// collide, so the shared-memory atomics seldom serialise).
__device__ __forceinline__ void hist_inc(uint32_t* bins, uint32_t d, bool valid) {
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    if (act == 0) return;
    const int first = __ffs(act) - 1;
    const uint32_t d0 = __shfl_sync(0xffffffffu, d, first);
    if (__all_sync(0xffffffffu, !valid || d == d0)) {
        if ((int)(threadIdx.x & 31) == first) atomicAdd(&bins[d0], (uint32_t)__popc(act));
    } else if (valid) {
        atomicAdd(&bins[d], 1u);
    }
}

// Exclusive prefix of this chunk's total over earlier chunks, by warp 0: the
// 32 nearest predecessors' words are read at once (each lane waits on one),
// summed up to the nearest inclusive prefix, and the window moves back until
// one is found.  Lane 0 then publishes this chunk's inclusive prefix.
__device__ __forceinline__ int64_t chunk_lookback(uint64_t* lookback, int64_t blk, int64_t total,
                                                  const ErrorSink& err) {
    const int lane = threadIdx.x & 31;
    if (blk == 0) {
        if (lane == 0) st_relaxed_u64(lookback, ((uint64_t)total << 2) | kFlagPrefix);
        return 0;
    }
    if (lane == 0) st_relaxed_u64(lookback + blk, ((uint64_t)total << 2) | kFlagAggregate);
    int64_t prefix = 0;
    for (int64_t top = blk - 1;; top -= kWarp) {
        const int64_t p = top - lane;
        const uint64_t v = p >= 0 ? wait_published(lookback + p, err) : kFlagPrefix;
        const unsigned pre = __ballot_sync(0xffffffffu, (v & kFlagMask) == kFlagPrefix);
        // lanes up to (and including) the nearest inclusive prefix contribute
        const int stop = pre ? __ffs(pre) - 1 : kWarp - 1;
        int64_t c = lane <= stop ? (int64_t)(v >> 2) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        prefix += c;
        if (pre) break;
    }
    if (lane == 0) st_relaxed_u64(lookback + blk, ((uint64_t)(prefix + total) << 2) | kFlagPrefix);
    return prefix;
}

// WIDE: 64-bit keys (camera | tile) << 32 | depth bits; else the 32-bit
// camera | tile word alone (keys32).  rects (may be null): the splats' rects
// from k_rect_hist, else computed here from means2d and radii.
template <bool WIDE>
__global__ void __launch_bounds__(kThreads)
    k_isect_emit(const float* __restrict__ means2d, const float* __restrict__ radii, int elliptical,
                 const float* __restrict__ depths, const int4* __restrict__ rects,
                 const int32_t* __restrict__ order, int64_t CN,
                 float ts, float inv_ts, int tile_width, int tile_height, int N, int tile_bits,
                 uint64_t* __restrict__ keys, uint32_t* __restrict__ keys32,
                 int32_t* __restrict__ ids, int64_t capacity,
                 int32_t* __restrict__ tiles_per_gauss, uint64_t* __restrict__ lookback,
                 uint32_t* __restrict__ ticket, uint32_t* __restrict__ up_hist, int up_passes,
                 ErrorSink err) {
    __shared__ EmitSmem sm;
    const int tid = threadIdx.x;
    if (tid == 0) sm.blk = atomicAdd(ticket, 1u);
    if (up_hist)
        for (int i = tid; i < 4 * 256; i += kThreads) (&sm.hist[0][0])[i] = 0;
    __syncthreads();
    const int64_t blk = sm.blk;
    // splats 2 tid and 2 tid + 1 of the chunk
    int cnt[2];
    int64_t local = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int slot = 2 * tid + u;
        const int64_t k = blk * kEmitSplats + slot;
        cnt[u] = 0;
        if (k < CN) {
            const int64_t s = order ? (int64_t)order[k] : k;
            Rect r;
            if (rects) {
                const int4 rc = rects[s];
                r = Rect{rc.x, rc.y, rc.z, rc.w};
            } else {
                const float2 m = reinterpret_cast<const float2*>(means2d)[s];
                float rx, ry;
                if (elliptical) {
                    const float2 rr = reinterpret_cast<const float2*>(radii)[s];
                    rx = rr.x;
                    ry = rr.y;
                } else {
                    rx = ry = radii[s];
                }
                r = splat_rect(m.x, m.y, rx, ry, ts, inv_ts, tile_width, tile_height);
            }
            cnt[u] = (r.x1 - r.x0) * (r.y1 - r.y0);
            sm.x0[slot] = r.x0;
            sm.y0[slot] = r.y0;
            sm.w[slot] = r.x1 - r.x0;
            sm.rw[slot] = __frcp_rn((float)(r.x1 - r.x0));
            sm.upper[slot] = (uint32_t)((uint64_t)(s / N) << tile_bits);
            if (WIDE) sm.dbits[slot] = __float_as_uint(depths[s]);
            sm.sid[slot] = (int32_t)s;
            if (tiles_per_gauss) tiles_per_gauss[s] = cnt[u];
        }
        local += cnt[u];
    }
    int64_t chunk_total;
    const int64_t excl = block_exclusive_scan<kThreads>(local, sm.scratch, &chunk_total);
    sm.incl[2 * tid] = (int32_t)(excl + cnt[0]);
    sm.incl[2 * tid + 1] = (int32_t)(excl + cnt[0] + cnt[1]);
    if (tid < kWarp) {
        const int64_t prefix = chunk_lookback(lookback, blk, chunk_total, err);
        if (tid == 0) {
            sm.base = prefix;
            const int64_t nchunks = (CN + kEmitSplats - 1) / kEmitSplats;
            if (prefix + chunk_total > capacity) err.raise(GS_ERR_COUNT_MISMATCH);
            if (blk == nchunks - 1 && prefix + chunk_total != capacity)
                err.raise(GS_ERR_COUNT_MISMATCH);
        }
    }
    __syncthreads();
    const int64_t base = sm.base;
    // Each warp writes the keys of its own 64 splats (slots 64 w .. 64 w + 63,
    // two per lane), 32 consecutive keys per round: a key's splat is the last
    // one starting at or before it, found from the round's start bits (each
    // splat starting in the round marks its offset and leaves its slot in
    // the warp's table) and, before the first start, the previous round's
    // last splat.
    const int lane = tid & 31, warp = tid >> 5;
    const int s_first = 2 * kWarp * warp;
    const int wstart = s_first == 0 ? 0 : sm.incl[s_first - 1];
    const int wend = sm.incl[s_first + 2 * kWarp - 1];
    int start[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) start[u] = sm.incl[2 * tid + u] - cnt[u];
    int carry = 0;
    for (int R = wstart; R < wend; R += kWarp) {
        unsigned mine = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int off = start[u] - R;
            if (cnt[u] > 0 && off >= 0 && off < kWarp) {
                mine |= 1u << off;
                sm.owner[warp][off] = (int16_t)(2 * tid + u);
            }
        }
        const unsigned starts = __reduce_or_sync(0xffffffffu, mine);
        __syncwarp();
        const unsigned upto = starts & (0xffffffffu >> (31 - lane));
        const int o = upto ? sm.owner[warp][31 - __clz(upto)] : carry;
        carry = starts ? sm.owner[warp][31 - __clz(starts)] : carry;
        __syncwarp();  // the table is read before the next round writes it
        const int q = R + lane;
        const bool valid = q < wend;
        uint32_t upper = 0;
        if (valid) {
            const int li = q - (o == 0 ? 0 : sm.incl[o - 1]);
            const int w = sm.w[o];
            // li / w from the reciprocal: li < 2^23, so the product is within
            // 1 of the quotient and one step either way corrects it
            int dy = __float2int_rz((float)li * sm.rw[o]);
            int rem = li - dy * w;
            if (rem < 0) {
                --dy;
                rem += w;
            } else if (rem >= w) {
                ++dy;
                rem -= w;
            }
            const int ty = sm.y0[o] + dy;
            const int tx = sm.x0[o] + rem;
            upper = sm.upper[o] | (uint32_t)(ty * tile_width + tx);
            const int64_t pos = base + q;
            if (pos < capacity) {
                if (WIDE) keys[pos] = ((uint64_t)upper << 32) | sm.dbits[o];
                else keys32[pos] = upper;
                ids[pos] = sm.sid[o];
            }
        }
        if (up_hist) {
            for (int p = 0; p < up_passes; ++p) hist_inc(sm.hist[p], (upper >> (8 * p)) & 0xffu, valid);
        }
    }
    if (up_hist) {
        __syncthreads();
        for (int i = tid; i < up_passes * 256; i += kThreads) {
            const uint32_t v = (&sm.hist[0][0])[i];
            if (v) atomicAdd(&up_hist[i], v);
        }
    }
}

__device__ __forceinline__ int64_t flat_tile(uint64_t key, int C, int64_t per_camera,
                                             int tile_bits, bool* ok) {
    const uint64_t upper = key >> 32;
    const uint64_t cam = upper >> tile_bits;
    const uint64_t tile = tile_bits == 0 ? 0 : (upper & ((1ull << tile_bits) - 1));
    *ok = cam < (uint64_t)C && tile < (uint64_t)per_camera;
    return (int64_t)cam * per_camera + (int64_t)tile;
}

// Tile ids of positions i - 1 (prev) and i (cur; position n is the end:
// every tile after the last key starts there) -> offsets of the tiles in
// between.  ok_* say whether the key lies inside the grid.
__device__ __forceinline__ void range_step(int64_t i, int64_t cur, bool ok_cur, int64_t prev,
                                           bool ok_prev, int64_t ntiles,
                                           int32_t* __restrict__ offsets, int32_t* d_status) {
    if (!ok_cur) {
        report(d_status, GS_ERR_KEY_OUT_OF_GRID);
        return;
    }
    if (!ok_prev) return;  // reported by that key's own step
    if (cur < prev) {
        report(d_status, GS_ERR_UNSORTED);
        return;
    }
    for (int64_t t = prev + 1; t <= cur && t < ntiles; ++t) offsets[t] = (int32_t)i;
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    k_tile_ranges(const uint64_t* __restrict__ keys, int64_t n, int C, int tile_width,
                  int tile_height, int tile_bits, int32_t* __restrict__ offsets,
                  int32_t* d_status) {
    const int64_t per_camera = (int64_t)tile_width * tile_height;
    const int lane = threadIdx.x & 31;
    const int64_t groups = (n + 1 + 3) / 4;  // positions 0 .. n, four per thread
    const int64_t warps = (int64_t)gridDim.x * (kThreads / kWarp);
    // whole warps step together, so every lane takes part in the shuffle
    for (int64_t wg = ((int64_t)blockIdx.x * (kThreads / kWarp) + (threadIdx.x >> 5)) * kWarp;
         wg < groups; wg += warps * kWarp) {
        const int64_t g = wg + lane;
        const int64_t p0 = 4 * g;
        uint64_t k[4] = {0, 0, 0, 0};
        if (VEC && p0 + 3 < n) {
            const ulonglong2 a = reinterpret_cast<const ulonglong2*>(keys)[2 * g];
            const ulonglong2 b = reinterpret_cast<const ulonglong2*>(keys)[2 * g + 1];
            k[0] = a.x;
            k[1] = a.y;
            k[2] = b.x;
            k[3] = b.y;
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (p0 + u < n) k[u] = keys[p0 + u];
        }
        // the key at p0 - 1 is the previous lane's last one (its group is
        // complete whenever this one has a position <= n)
        uint64_t before = __shfl_up_sync(0xffffffffu, k[3], 1);
        if (lane == 0 && p0 > 0 && p0 <= n) before = keys[p0 - 1];
        const int64_t ntiles = (int64_t)C * per_camera;
        // each key's tile id is worked out once and serves as the next
        // position's predecessor
        bool ok_prev = true;
        int64_t prev = p0 > 0 ? flat_tile(before, C, per_camera, tile_bits, &ok_prev) : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = p0 + u;
            if (i > n) break;
            bool ok_cur = true;
            const int64_t cur = i < n ? flat_tile(k[u], C, per_camera, tile_bits, &ok_cur) : ntiles;
            range_step(i, cur, ok_cur, prev, ok_prev, ntiles, offsets, d_status);
            prev = cur;
            ok_prev = ok_cur;
        }
    }
}

// Copies the device total to a mapped host word (a plain store over the
// host link, so it does not wait for the copy engines).
__global__ void k_publish_total(const unsigned long long* __restrict__ total,
                                volatile unsigned long long* host_word) {
    *host_word = *total;
    __threadfence_system();
}

int grid_for(int64_t n, int per_thread) {
    int64_t g = (n + (int64_t)kThreads * per_thread - 1) / ((int64_t)kThreads * per_thread);
    if (g < 1) g = 1;
    if (g > 152 * 16) g = 152 * 16;
    return (int)g;
}

}  // namespace

void launch_isect_count(const float* means2d, const float* radii, int elliptical, int64_t CN,
                        int tile_size, int tile_width, int tile_height, int32_t* tiles_per_gauss,
                        unsigned long long* total, cudaStream_t s) {
    if (CN <= 0) return;
    k_isect_count<<<grid_for(CN, 4), kThreads, 0, s>>>(means2d, radii, elliptical, CN,
                                                       (float)tile_size,
                                                       exact_tile_inverse(tile_size), tile_width,
                                                       tile_height, tiles_per_gauss, total);
}

void launch_publish_total(const unsigned long long* total, unsigned long long* host_word,
                          cudaStream_t s) {
    k_publish_total<<<1, 1, 0, s>>>(total, host_word);
}

void launch_rect_hist(const float* means2d, const float* radii, int elliptical,
                      const uint32_t* dbits, int64_t CN, int tile_size, int tile_width,
                      int tile_height, int4* rects, uint32_t* hist, cudaStream_t s) {
    if (CN <= 0) return;
    k_rect_hist<<<grid_for(CN, 4), kThreads, 0, s>>>(means2d, radii, elliptical, dbits, CN,
                                                     (float)tile_size,
                                                     exact_tile_inverse(tile_size), tile_width,
                                                     tile_height, rects, hist);
}

void launch_isect_emit(const float* means2d, const float* radii, int elliptical,
                       const float* depths, const int4* rects, const int32_t* order, int64_t CN,
                       int tile_size, int tile_width, int tile_height, int N, int tile_bits,
                       uint64_t* keys, uint32_t* keys32, int32_t* ids, int64_t capacity,
                       int32_t* tiles_per_gauss, LookbackScratch lb, uint32_t* up_hist,
                       int up_passes, int32_t* abort_flag, int32_t* d_status, cudaStream_t s) {
    if (CN <= 0) return;
    const int64_t chunks = (CN + kEmitSplats - 1) / kEmitSplats;
    const ErrorSink err{abort_flag, d_status};
    if (keys)
        k_isect_emit<true><<<(unsigned)chunks, kThreads, 0, s>>>(
            means2d, radii, elliptical, depths, rects, order, CN, (float)tile_size,
            exact_tile_inverse(tile_size), tile_width,
            tile_height, N, tile_bits, keys, nullptr, ids, capacity, tiles_per_gauss, lb.words,
            lb.ticket, up_hist, up_passes, err);
    else
        k_isect_emit<false><<<(unsigned)chunks, kThreads, 0, s>>>(
            means2d, radii, elliptical, depths, rects, order, CN, (float)tile_size,
            exact_tile_inverse(tile_size), tile_width,
            tile_height, N, tile_bits, nullptr, keys32, ids, capacity, tiles_per_gauss,
            lb.words, lb.ticket, up_hist, up_passes, err);
}

void launch_widen(const uint32_t* k32, const int32_t* v32, const uint32_t* dbits, int64_t n,
                  uint64_t* keys, int32_t* ids, cudaStream_t s) {
    if (n <= 0) return;
    k_widen<<<grid_for(n, 4), kThreads, 0, s>>>(k32, v32, dbits, n, keys, ids);
}

void launch_tile_ranges(const uint64_t* keys, int64_t n, int C, int tile_width, int tile_height,
                        int tile_bits, int32_t* offsets, int32_t* d_status, cudaStream_t s) {
    const int grid = grid_for(n + 1, 4);
    if ((reinterpret_cast<uintptr_t>(keys) & 15) == 0)
        k_tile_ranges<true><<<grid, kThreads, 0, s>>>(keys, n, C, tile_width, tile_height,
                                                       tile_bits, offsets, d_status);
    else
        k_tile_ranges<false><<<grid, kThreads, 0, s>>>(keys, n, C, tile_width, tile_height,
                                                        tile_bits, offsets, d_status);
}

}  // namespace gs
