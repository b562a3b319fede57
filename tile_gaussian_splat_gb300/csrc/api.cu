// C ABI of libgs_splat_gb300 (declared in include/gs_splat.h): argument
// checks, workspace layout and the launch sequence of each call.
//
// gs_isect_tiles with sort != 0 produces the listing's stable sort by the
// 64-bit key (gsplat 1.0.0, intersections.c, gs_radix_sort_without_gvl) in
// fewer bytes moved:
//   1. the splats are sorted by the bits of their depth (four 8-bit passes
//      over C*N 32-bit keys, stable, so equal depths stay in index order);
//      the pass that histograms their digits also caches every splat's tile
//      rect, so step 2 gathers 16 bytes per splat in depth order;
//   2. the intersections are emitted splat by splat in that order, so in
//      every tile they already appear by (depth bits, splat index); only the
//      32-bit camera|tile word is written;
//   3. a stable LSD sort on the camera|tile digits (ceil((tile_bits +
//      camera bits) / 8) passes over the I 32-bit keys with their ids) then
//      yields exactly the order of a stable sort of the full keys; the last
//      pass writes the 64-bit keys, taking each key's low word (the splat's
//      depth bits) from the depths array.
// Every key of a splat carries the same depth bits, so its low 32 bits are
// sorted once per splat instead of once per intersection, and the radix
// passes move 8 bytes per intersection instead of 12.
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/gs_splat.h"
#include "gs_internal.h"

namespace {

using namespace gs;

constexpr int kVersion = 100;  // 0.1.0
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int bitlen(uint64_t v) {
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

// Bump allocator over a caller buffer (or a null base when only sizing).
struct Carver {
    char* base;
    size_t used = 0;
    template <typename T>
    T* take(size_t count) {
        size_t at = used;
        used = align_up(used + count * sizeof(T));
        return base ? reinterpret_cast<T*>(base + at) : nullptr;
    }
};

constexpr int kMaxPasses = 8;

// Limits of the timeout-path test hook (gs_debug_sort_wait_timeout).
constexpr int kMaxDebugTickets = 64;
constexpr int kMaxDebugPolls = 1 << 20;

// Workspace of gs_isect_tiles.  Everything up to `zero_end` is cleared by one
// memset per call; the sort buffers after it are fully overwritten.
struct IsectLayout {
    int32_t* abort_flag;
    unsigned long long* total;
    uint32_t* tickets;       // [2 * kMaxPasses + 1]
    uint32_t* hist_depth;    // [4][256]
    uint32_t* hist_up;       // [4][256]
    uint64_t* lb_emit;       // [chunks]
    uint64_t* lb_depth[4];   // [blocks32 * 256] each
    uint64_t* lb_up[4];      // [blocks32 * 256] each
    size_t zero_end;
    uint32_t* dkeys[2];      // [C*N]
    int32_t* dvals[2];       // [C*N]
    int4* rects;             // [C*N] tile rects (x0, y0, x1, y1), presort only
    uint32_t* k32;           // [I] camera|tile keys (sorted path)
    int32_t* v32;            // [I] their flatten ids
    size_t bytes;
};

struct IsectPlan {
    int64_t CN;
    int tile_bits, cam_bits, up_passes;
    bool sort, presort;
};

IsectPlan make_plan(int C, int N, int tw, int th, int64_t n_isects, int sort) {
    IsectPlan p;
    p.CN = (int64_t)C * N;
    p.tile_bits = gs_tile_bits(tw, th);
    p.cam_bits = bitlen((uint64_t)(C > 0 ? C - 1 : 0));
    p.up_passes = sort ? (p.tile_bits + p.cam_bits + 7) / 8 : 0;
    p.sort = sort != 0;
    p.presort = sort && n_isects > 1 && p.CN > 1;
    if (n_isects <= 1) p.up_passes = 0;
    return p;
}

IsectLayout carve_isect(void* ws, const IsectPlan& p, int64_t n_isects, bool query) {
    Carver cv{static_cast<char*>(ws)};
    IsectLayout L{};
    L.abort_flag = cv.take<int32_t>(1);
    L.total = cv.take<unsigned long long>(1);
    L.tickets = cv.take<uint32_t>(2 * kMaxPasses + 1);
    L.hist_depth = cv.take<uint32_t>(4 * 256);
    L.hist_up = cv.take<uint32_t>(4 * 256);
    if (!query) {
        L.lb_emit = cv.take<uint64_t>((size_t)((p.CN + kEmitChunk - 1) / kEmitChunk));
        if (p.presort)
            for (int i = 0; i < 4; ++i)
                L.lb_depth[i] = cv.take<uint64_t>((size_t)sort_blocks(p.CN, kTile32) * 256);
        for (int i = 0; i < p.up_passes; ++i)
            L.lb_up[i] = cv.take<uint64_t>((size_t)sort_blocks(n_isects, kTile32) * 256);
    }
    L.zero_end = cv.used;
    if (!query) {
        if (p.presort) {
            for (int i = 0; i < 2; ++i) {
                L.dkeys[i] = cv.take<uint32_t>((size_t)p.CN);
                L.dvals[i] = cv.take<int32_t>((size_t)p.CN);
            }
            L.rects = cv.take<int4>((size_t)p.CN);
        }
        if (p.sort) {
            L.k32 = cv.take<uint32_t>((size_t)n_isects);
            L.v32 = cv.take<int32_t>((size_t)n_isects);
        }
    }
    L.bytes = cv.used;
    return L;
}

// One word of mapped pinned host memory per calling thread and device, for
// the size query's count: the device stores it directly, so the query does
// not wait behind large copies queued on the copy engines.  Allocated on
// first use and kept for the thread's lifetime.
struct MappedWord {
    unsigned long long* host = nullptr;
    unsigned long long* dev = nullptr;
};

constexpr int kMaxDevices = 64;

bool mapped_word(MappedWord* out) {
    thread_local MappedWord words[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    MappedWord& w = words[dev];
    if (!w.host) {
        void* h = nullptr;
        void* d = nullptr;
        if (cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
            return false;
        if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
            cudaFreeHost(h);
            return false;
        }
        w.host = static_cast<unsigned long long*>(h);
        w.dev = static_cast<unsigned long long*>(d);
    }
    *out = w;
    return true;
}

int check_launch() {
    return cudaGetLastError() == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}

int isect_args_ok(const float* means2d, const float* radii, int C, int N, int tile_size,
                  int tile_width, int tile_height) {
    if (C < 1 || N < 0 || tile_size < 1 || tile_width < 1 || tile_height < 1) return 0;
    if ((int64_t)C * N >= ((int64_t)1 << 31)) return 0;
    if ((int64_t)tile_width * tile_height > ((int64_t)1 << 23)) return 0;
    if (gs_tile_bits(tile_width, tile_height) + bitlen((uint64_t)(C - 1)) > 32) return 0;
    if ((int64_t)C * N > 0 && (!means2d || !radii)) return 0;
    return 1;
}

int raster_args_ok(const float* means2d, const float* conics, const float* colors,
                   const float* opacities, int C, int N, int channels, int width, int height,
                   int tile_size, const int32_t* offsets, const int32_t* flatten_ids,
                   int64_t n_isects) {
    if (C < 1 || N < 0 || width < 1 || height < 1) return 0;
    if (channels < 1 || channels > GS_MAX_CHANNELS || tile_size != 16) return 0;
    if ((int64_t)C * N >= ((int64_t)1 << 31) || n_isects < 0 || n_isects >= ((int64_t)1 << 31))
        return 0;
    if (!offsets) return 0;
    if (n_isects > 0 && (!flatten_ids || !means2d || !conics || !colors || !opacities)) return 0;
    return 1;
}

}  // namespace

extern "C" {

int gs_version(void) { return kVersion; }

const char* gs_status_string(int status) {
    switch (status) {
        case GS_OK: return "ok";
        case GS_ERR_INVALID_ARG: return "invalid argument";
        case GS_ERR_CAPACITY: return "more intersections than the buffers hold";
        case GS_ERR_KEY_OUT_OF_GRID: return "intersection key is outside the tile grid";
        case GS_ERR_WORKSPACE: return "workspace missing or too small";
        case GS_ERR_TIMEOUT: return "a bounded inter-block wait ran out";
        case GS_ERR_CUDA: return "CUDA runtime error";
        case GS_ERR_UNSORTED: return "keys are not sorted";
        case GS_ERR_COUNT_MISMATCH: return "n_isects differs from the emitted total";
        case GS_ERR_OUT_OF_BOUNDS: return "an index read from the inputs is outside its array";
        default: return "unknown status";
    }
}

int gs_tile_bits(int tile_width, int tile_height) {
    if (tile_width < 1 || tile_height < 1) return 0;
    const uint64_t tiles = (uint64_t)tile_width * (uint64_t)tile_height;
    int b = 0;
    while (((uint64_t)1 << b) < tiles) ++b;
    return b;
}

size_t gs_isect_workspace_size(int C, int N, int tile_width, int tile_height, int64_t n_isects,
                               int sort) {
    if (C < 1 || N < 0 || n_isects < 0) return 0;
    // the emitting layout for n_isects also covers the size query's needs
    IsectPlan p = make_plan(C, N, tile_width, tile_height, n_isects, sort);
    return carve_isect(nullptr, p, n_isects, false).bytes;
}

int gs_isect_tiles(const float* means2d, const float* radii, int elliptical, const float* depths,
                   int C, int N, int tile_size, int tile_width, int tile_height, int sort,
                   int32_t* tiles_per_gauss, int64_t* h_n_isects, uint64_t* keys,
                   int32_t* flatten_ids, int64_t n_isects, void* workspace,
                   size_t workspace_bytes, int32_t* d_status, void* stream) {
    if (!isect_args_ok(means2d, radii, C, N, tile_size, tile_width, tile_height))
        return GS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool query = keys == nullptr;
    if (query) {
        if (!h_n_isects) return GS_ERR_INVALID_ARG;
        IsectPlan p = make_plan(C, N, tile_width, tile_height, 0, sort);
        IsectLayout L = carve_isect(workspace, p, 0, true);
        if (!workspace || workspace_bytes < L.bytes) return GS_ERR_WORKSPACE;
        if (cudaMemsetAsync(workspace, 0, L.zero_end, s) != cudaSuccess) return GS_ERR_CUDA;
        launch_isect_count(means2d, radii, elliptical, p.CN, tile_size, tile_width, tile_height,
                           tiles_per_gauss, L.total, s);
        if (check_launch() != GS_OK) return GS_ERR_CUDA;
        unsigned long long total = 0;
        MappedWord mw;
        if (mapped_word(&mw)) {
            launch_publish_total(L.total, mw.dev, s);
            if (check_launch() != GS_OK) return GS_ERR_CUDA;
            if (cudaStreamSynchronize(s) != cudaSuccess) return GS_ERR_CUDA;
            total = *static_cast<volatile unsigned long long*>(mw.host);
        } else {  // no mapped host memory: a copy
            if (cudaMemcpyAsync(&total, L.total, sizeof(total), cudaMemcpyDeviceToHost, s) !=
                cudaSuccess)
                return GS_ERR_CUDA;
            if (cudaStreamSynchronize(s) != cudaSuccess) return GS_ERR_CUDA;
        }
        *h_n_isects = (int64_t)total;
        return total >= ((unsigned long long)1 << 31) ? GS_ERR_CAPACITY : GS_OK;
    }
    if (n_isects < 0 || n_isects >= ((int64_t)1 << 31)) return GS_ERR_INVALID_ARG;
    if (n_isects > 0 && (!flatten_ids || !depths)) return GS_ERR_INVALID_ARG;
    IsectPlan p = make_plan(C, N, tile_width, tile_height, n_isects, sort);
    IsectLayout L = carve_isect(workspace, p, n_isects, false);
    if (!workspace || workspace_bytes < L.bytes) return GS_ERR_WORKSPACE;
    if (cudaMemsetAsync(workspace, 0, L.zero_end, s) != cudaSuccess) return GS_ERR_CUDA;
    if (p.CN == 0) {
        if (n_isects != 0 && d_status) {
            const int32_t code = GS_ERR_COUNT_MISMATCH;
            if (cudaMemcpyAsync(d_status, &code, 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
                return GS_ERR_CUDA;
            if (cudaStreamSynchronize(s) != cudaSuccess) return GS_ERR_CUDA;
        }
        return GS_OK;
    }
    const uint32_t* dbits = reinterpret_cast<const uint32_t*>(depths);
    if (!p.sort) {
        // emission order, 64-bit keys straight into the outputs
        launch_isect_emit(means2d, radii, elliptical, depths, nullptr, nullptr, p.CN, tile_size,
                          tile_width, tile_height, N, p.tile_bits, keys, nullptr, flatten_ids,
                          n_isects, tiles_per_gauss,
                          LookbackScratch{L.lb_emit, L.tickets + 2 * kMaxPasses}, nullptr, 0,
                          L.abort_flag, d_status, s);
        return check_launch();
    }
    const int32_t* order = nullptr;
    if (p.presort) {
        // 1. tile rects and depth-digit histograms, then the splats by depth
        //    bits in four stable passes (values start as indices)
        launch_rect_hist(means2d, radii, elliptical, dbits, p.CN, tile_size, tile_width,
                         tile_height, L.rects, L.hist_depth, s);
        const uint32_t* kin = dbits;
        const int32_t* vin = nullptr;
        for (int pass = 0; pass < 4; ++pass) {
            uint32_t* kout = L.dkeys[pass & 1];
            int32_t* vout = L.dvals[pass & 1];
            launch_onesweep_u32(kin, vin, kout, vout, p.CN, 8 * pass, 32,
                                L.hist_depth + 256 * pass,
                                LookbackScratch{L.lb_depth[pass], L.tickets + pass},
                                L.abort_flag, d_status, s);
            kin = kout;
            vin = vout;
        }
        order = vin;
    }
    // 2. emission of 32-bit camera|tile keys.  The passes alternate between
    //    the workspace pair (k32, v32) and the caller's keys buffer (8 bytes
    //    per key: 32-bit keys in its first half, ids in its second); the
    //    start is chosen so that the last pass reads the workspace pair and
    //    writes the 64-bit keys and the ids.
    uint32_t* ak = reinterpret_cast<uint32_t*>(keys);
    int32_t* av = reinterpret_cast<int32_t*>(keys) + n_isects;
    const bool start_a = p.up_passes > 0 && (p.up_passes & 1) == 0;
    uint32_t* ck = start_a ? ak : L.k32;
    int32_t* cv = start_a ? av : L.v32;
    launch_isect_emit(means2d, radii, elliptical, depths, p.presort ? L.rects : nullptr, order,
                      p.CN, tile_size, tile_width, tile_height, N, p.tile_bits, nullptr, ck, cv,
                      n_isects, tiles_per_gauss,
                      LookbackScratch{L.lb_emit, L.tickets + 2 * kMaxPasses},
                      p.up_passes ? L.hist_up : nullptr, p.up_passes, L.abort_flag, d_status, s);
    // 3. stable passes over the camera|tile digits; the last one widens
    const int end_bit = p.tile_bits + p.cam_bits;
    for (int pass = 0; pass < p.up_passes; ++pass) {
        const LookbackScratch lb{L.lb_up[pass], L.tickets + 4 + pass};
        if (pass == p.up_passes - 1) {
            launch_onesweep_u32_widen(ck, cv, keys, flatten_ids, n_isects, 8 * pass, end_bit,
                                      L.hist_up + 256 * pass, dbits, lb, L.abort_flag, d_status,
                                      s);
        } else {
            uint32_t* nk = ck == ak ? L.k32 : ak;
            int32_t* nv = cv == av ? L.v32 : av;
            launch_onesweep_u32(ck, cv, nk, nv, n_isects, 8 * pass, end_bit,
                                L.hist_up + 256 * pass, lb, L.abort_flag, d_status, s);
            ck = nk;
            cv = nv;
        }
    }
    if (p.up_passes == 0) launch_widen(ck, cv, dbits, n_isects, keys, flatten_ids, s);
    return check_launch();
}

int gs_tile_offsets(const uint64_t* keys, int64_t n_isects, int C, int tile_width,
                    int tile_height, int32_t* offsets, int32_t* d_status, void* stream) {
    if (C < 1 || tile_width < 1 || tile_height < 1 || !offsets) return GS_ERR_INVALID_ARG;
    if (n_isects < 0 || n_isects >= ((int64_t)1 << 31) || (n_isects > 0 && !keys))
        return GS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t ntiles = (int64_t)C * tile_width * tile_height;
    if (n_isects == 0) {
        if (cudaMemsetAsync(offsets, 0, (size_t)ntiles * sizeof(int32_t), s) != cudaSuccess)
            return GS_ERR_CUDA;
        return GS_OK;
    }
    launch_tile_ranges(keys, n_isects, C, tile_width, tile_height,
                       gs_tile_bits(tile_width, tile_height), offsets, d_status, s);
    return check_launch();
}

}  // extern "C"

namespace {

// The raster calls over either list form: sorted lists (offsets != null,
// flatten_ids of length n_isects) or bin lists (bin_counts != null,
// flatten_ids = the bins, n_isects = tiles * bin_capacity).
int raster_fwd(const float* means2d, const float* conics, const float* colors,
               const float* opacities, const float* backgrounds, const int32_t* masks, int C,
               int N, int channels, int width, int height, const int32_t* offsets,
               const int32_t* bin_counts, int bin_capacity, const int32_t* flatten_ids,
               int64_t n_isects, float alpha_cutoff, float transmittance_threshold,
               float* render_colors, float* render_alphas, int32_t* last_ids,
               int32_t* pair_counts, uint32_t* trace, int32_t* d_status, void* stream,
               const StepArgs* steps = nullptr) {
    if (!render_colors || !render_alphas || !last_ids) return GS_ERR_INVALID_ARG;
    if (trace && (reinterpret_cast<uintptr_t>(trace) & 15u)) return GS_ERR_INVALID_ARG;
    RasterArgs a{means2d, conics, colors, opacities, backgrounds, masks,
                 C, N, width, height, (width + 15) / 16, (height + 15) / 16,
                 offsets, flatten_ids, n_isects, alpha_cutoff, transmittance_threshold,
                 channels, 0, 1, bin_counts, bin_capacity, d_status};
    launch_raster_fwd(a, render_colors, render_alphas, last_ids, pair_counts, trace,
                      static_cast<cudaStream_t>(stream), steps);
    return check_launch();
}

int raster_bwd(const float* means2d, const float* conics, const float* colors,
               const float* opacities, const float* backgrounds, const int32_t* masks, int C,
               int N, int channels, int width, int height, const int32_t* offsets,
               const int32_t* bin_counts, int bin_capacity, const int32_t* flatten_ids,
               int64_t n_isects, float alpha_cutoff, const float* render_alphas,
               const int32_t* last_ids, const float* grad_render_colors,
               const float* grad_render_alphas, float* grad_means2d, float* grad_conics,
               float* grad_colors, float* grad_opacities, float* grad_backgrounds,
               float* grad_means2d_abs, const uint32_t* trace, int32_t* d_status,
               void* stream, const StepArgs* steps = nullptr) {
    if (!render_alphas || !last_ids || !grad_render_colors || !grad_render_alphas)
        return GS_ERR_INVALID_ARG;
    const int64_t CN = (int64_t)C * N;
    if (CN > 0 && (!grad_means2d || !grad_conics || !grad_colors || !grad_opacities))
        return GS_ERR_INVALID_ARG;
    if (grad_backgrounds && !backgrounds) return GS_ERR_INVALID_ARG;
    if (trace && (reinterpret_cast<uintptr_t>(trace) & 15u)) return GS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t f = sizeof(float);
    if (CN > 0) {
        if (cudaMemsetAsync(grad_means2d, 0, CN * 2 * f, s) != cudaSuccess ||
            cudaMemsetAsync(grad_conics, 0, CN * 3 * f, s) != cudaSuccess ||
            cudaMemsetAsync(grad_colors, 0, CN * channels * f, s) != cudaSuccess ||
            cudaMemsetAsync(grad_opacities, 0, CN * f, s) != cudaSuccess)
            return GS_ERR_CUDA;
        if (grad_means2d_abs && cudaMemsetAsync(grad_means2d_abs, 0, CN * 2 * f, s) != cudaSuccess)
            return GS_ERR_CUDA;
    }
    if (grad_backgrounds && cudaMemsetAsync(grad_backgrounds, 0, (size_t)C * channels * f, s) != cudaSuccess)
        return GS_ERR_CUDA;
    RasterArgs a{means2d, conics, colors, opacities, backgrounds, masks,
                 C, N, width, height, (width + 15) / 16, (height + 15) / 16,
                 offsets, flatten_ids, n_isects, alpha_cutoff, 0.0f, channels, 0, 1,
                 bin_counts, bin_capacity, d_status};
    RasterGrads g{render_alphas, last_ids, grad_render_colors, grad_render_alphas,
                  grad_means2d, grad_conics, grad_colors, grad_opacities, grad_backgrounds,
                  grad_means2d_abs};
    if (steps)
        launch_raster_bwd_steps(a, g, *steps, s);
    else
        launch_raster_bwd(a, g, trace, s);
    return check_launch();
}

// Bin form: capacity in [1, kMaxBinCapacity], positions tiles * capacity
// below 2^31 (last_ids are positions into the bins).
int bin_args_ok(int C, int width, int height, int tile_size, int capacity, const int32_t* bins,
                const int32_t* counts, int64_t* n_slots) {
    if (C < 1 || width < 1 || height < 1 || tile_size < 1) return 0;
    if (capacity < 1 || capacity > kMaxBinCapacity || !bins || !counts) return 0;
    const int64_t tw = (width + tile_size - 1) / tile_size, th = (height + tile_size - 1) / tile_size;
    *n_slots = (int64_t)C * tw * th * capacity;
    return *n_slots < ((int64_t)1 << 31);
}

}  // namespace

extern "C" {

int gs_rasterize_fwd(const float* means2d, const float* conics, const float* colors,
                     const float* opacities, const float* backgrounds, const int32_t* masks,
                     int C, int N, int channels, int width, int height, int tile_size,
                     const int32_t* offsets, const int32_t* flatten_ids, int64_t n_isects,
                     float alpha_cutoff, float transmittance_threshold, float* render_colors,
                     float* render_alphas, int32_t* last_ids, int32_t* pair_counts,
                     uint32_t* trace, int32_t* d_status, void* stream) {
    if (!raster_args_ok(means2d, conics, colors, opacities, C, N, channels, width, height,
                        tile_size, offsets, flatten_ids, n_isects))
        return GS_ERR_INVALID_ARG;
    return raster_fwd(means2d, conics, colors, opacities, backgrounds, masks, C, N, channels,
                      width, height, offsets, nullptr, 0, flatten_ids, n_isects, alpha_cutoff,
                      transmittance_threshold, render_colors, render_alphas, last_ids,
                      pair_counts, trace, d_status, stream);
}

int gs_rasterize_bwd(const float* means2d, const float* conics, const float* colors,
                     const float* opacities, const float* backgrounds, const int32_t* masks,
                     int C, int N, int channels, int width, int height, int tile_size,
                     const int32_t* offsets, const int32_t* flatten_ids, int64_t n_isects,
                     float alpha_cutoff, const float* render_alphas, const int32_t* last_ids,
                     const float* grad_render_colors, const float* grad_render_alphas,
                     float* grad_means2d, float* grad_conics, float* grad_colors,
                     float* grad_opacities, float* grad_backgrounds, float* grad_means2d_abs,
                     const uint32_t* trace, int32_t* d_status, void* stream) {
    if (!raster_args_ok(means2d, conics, colors, opacities, C, N, channels, width, height,
                        tile_size, offsets, flatten_ids, n_isects))
        return GS_ERR_INVALID_ARG;
    return raster_bwd(means2d, conics, colors, opacities, backgrounds, masks, C, N, channels,
                      width, height, offsets, nullptr, 0, flatten_ids, n_isects, alpha_cutoff,
                      render_alphas, last_ids, grad_render_colors, grad_render_alphas,
                      grad_means2d, grad_conics, grad_colors, grad_opacities, grad_backgrounds,
                      grad_means2d_abs, trace, d_status, stream);
}

// The step-trace arrays: max_steps >= 1, pos/T of max_steps * C*H*W elements.
static int steps_ok(int max_steps, int C, int width, int height, const void* pos, const void* T,
                    const void* count) {
    if (max_steps < 1 || !pos || !T || !count) return 0;
    return (int64_t)max_steps * C * width * height < ((int64_t)1 << 40);
}

int gs_rasterize_fwd_steps(const float* means2d, const float* conics, const float* colors,
                           const float* opacities, const float* backgrounds,
                           const int32_t* masks, int C, int N, int channels, int width,
                           int height, int tile_size, const int32_t* offsets,
                           const int32_t* flatten_ids, int64_t n_isects, float alpha_cutoff,
                           float transmittance_threshold, int max_steps, float* render_colors,
                           float* render_alphas, int32_t* last_ids, int32_t* step_pos,
                           float* step_T, int32_t* step_count, int32_t* d_status, void* stream) {
    if (!raster_args_ok(means2d, conics, colors, opacities, C, N, channels, width, height,
                        tile_size, offsets, flatten_ids, n_isects) ||
        !steps_ok(max_steps, C, width, height, step_pos, step_T, step_count))
        return GS_ERR_INVALID_ARG;
    const StepArgs sa{step_pos, step_T, step_count, max_steps};
    return raster_fwd(means2d, conics, colors, opacities, backgrounds, masks, C, N, channels,
                      width, height, offsets, nullptr, 0, flatten_ids, n_isects, alpha_cutoff,
                      transmittance_threshold, render_colors, render_alphas, last_ids, nullptr,
                      nullptr, d_status, stream, &sa);
}

int gs_rasterize_bwd_steps(const float* means2d, const float* conics, const float* colors,
                           const float* opacities, const float* backgrounds,
                           const int32_t* masks, int C, int N, int channels, int width,
                           int height, int tile_size, const int32_t* offsets,
                           const int32_t* flatten_ids, int64_t n_isects, float alpha_cutoff,
                           const float* render_alphas, const int32_t* last_ids, int max_steps,
                           const int32_t* step_pos, const float* step_T,
                           const int32_t* step_count, const float* grad_render_colors,
                           const float* grad_render_alphas, float* grad_means2d,
                           float* grad_conics, float* grad_colors, float* grad_opacities,
                           float* grad_backgrounds, float* grad_means2d_abs, int32_t* d_status,
                           void* stream) {
    if (!raster_args_ok(means2d, conics, colors, opacities, C, N, channels, width, height,
                        tile_size, offsets, flatten_ids, n_isects) ||
        !steps_ok(max_steps, C, width, height, step_pos, step_T, step_count))
        return GS_ERR_INVALID_ARG;
    const StepArgs sa{const_cast<int32_t*>(step_pos), const_cast<float*>(step_T),
                      const_cast<int32_t*>(step_count), max_steps};
    return raster_bwd(means2d, conics, colors, opacities, backgrounds, masks, C, N, channels,
                      width, height, offsets, nullptr, 0, flatten_ids, n_isects, alpha_cutoff,
                      render_alphas, last_ids, grad_render_colors, grad_render_alphas,
                      grad_means2d, grad_conics, grad_colors, grad_opacities, grad_backgrounds,
                      grad_means2d_abs, nullptr, d_status, stream, &sa);
}

int gs_bin_splats(const float* means2d, const float* radii, int elliptical, const float* depths,
                  int C, int N, int tile_size, int tile_width, int tile_height, int capacity,
                  int32_t* bins, int32_t* bin_counts, int32_t* d_status, void* stream) {
    if (!isect_args_ok(means2d, radii, C, N, tile_size, tile_width, tile_height))
        return GS_ERR_INVALID_ARG;
    if (capacity < 1 || capacity > kMaxBinCapacity || !bins || !bin_counts) return GS_ERR_INVALID_ARG;
    const int64_t nbins = (int64_t)C * tile_width * tile_height;
    if (nbins * capacity >= ((int64_t)1 << 31)) return GS_ERR_INVALID_ARG;
    if ((int64_t)C * N > 0 && !depths) return GS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(bin_counts, 0, (size_t)nbins * sizeof(int32_t), s) != cudaSuccess)
        return GS_ERR_CUDA;
    const int rc = launch_bin_splats(means2d, radii, elliptical, depths, C, N, tile_size,
                                     tile_width, tile_height, capacity, bins, bin_counts,
                                     d_status, s);
    if (rc != GS_OK) return rc;
    return check_launch();
}

int gs_rasterize_fwd_bins(const float* means2d, const float* conics, const float* colors,
                          const float* opacities, const float* backgrounds, const int32_t* masks,
                          int C, int N, int channels, int width, int height, int tile_size,
                          const int32_t* bins, const int32_t* bin_counts, int capacity,
                          float alpha_cutoff, float transmittance_threshold,
                          float* render_colors, float* render_alphas, int32_t* last_ids,
                          int32_t* pair_counts, uint32_t* trace, int32_t* d_status,
                          void* stream) {
    (void)d_status;
    int64_t n_slots = 0;
    if (!bin_args_ok(C, width, height, tile_size, capacity, bins, bin_counts, &n_slots) ||
        !raster_args_ok(means2d, conics, colors, opacities, C, N, channels, width, height,
                        tile_size, bin_counts, bins, n_slots))
        return GS_ERR_INVALID_ARG;
    return raster_fwd(means2d, conics, colors, opacities, backgrounds, masks, C, N, channels,
                      width, height, nullptr, bin_counts, capacity, bins, n_slots, alpha_cutoff,
                      transmittance_threshold, render_colors, render_alphas, last_ids,
                      pair_counts, trace, d_status, stream);
}

int gs_rasterize_bwd_bins(const float* means2d, const float* conics, const float* colors,
                          const float* opacities, const float* backgrounds, const int32_t* masks,
                          int C, int N, int channels, int width, int height, int tile_size,
                          const int32_t* bins, const int32_t* bin_counts, int capacity,
                          float alpha_cutoff, const float* render_alphas,
                          const int32_t* last_ids, const float* grad_render_colors,
                          const float* grad_render_alphas, float* grad_means2d,
                          float* grad_conics, float* grad_colors, float* grad_opacities,
                          float* grad_backgrounds, float* grad_means2d_abs,
                          const uint32_t* trace, int32_t* d_status, void* stream) {
    (void)d_status;
    int64_t n_slots = 0;
    if (!bin_args_ok(C, width, height, tile_size, capacity, bins, bin_counts, &n_slots) ||
        !raster_args_ok(means2d, conics, colors, opacities, C, N, channels, width, height,
                        tile_size, bin_counts, bins, n_slots))
        return GS_ERR_INVALID_ARG;
    return raster_bwd(means2d, conics, colors, opacities, backgrounds, masks, C, N, channels,
                      width, height, nullptr, bin_counts, capacity, bins, n_slots, alpha_cutoff,
                      render_alphas, last_ids, grad_render_colors, grad_render_alphas,
                      grad_means2d, grad_conics, grad_colors, grad_opacities, grad_backgrounds,
                      grad_means2d_abs, trace, d_status, stream);
}

int gs_project(const float* means, const float* covars, const float* viewmats,
               const float* intrinsics, int C, int N, int width, int height, float eps2d,
               float near_plane, float far_plane, float radius_clip, int orthographic,
               int32_t* radii, float* means2d, float* depths, float* conics,
               float* compensations, float* radii_float, int32_t* d_status, void* stream) {
    (void)d_status;
    if (C < 1 || N < 0 || width < 1 || height < 1) return GS_ERR_INVALID_ARG;
    if ((int64_t)C * N >= ((int64_t)1 << 31)) return GS_ERR_INVALID_ARG;
    if (N == 0) return GS_OK;
    if (!means || !covars || !viewmats || !intrinsics || !radii || !means2d || !depths || !conics)
        return GS_ERR_INVALID_ARG;
    // radii, means2d and radii_float are stored as 8-byte pairs
    if ((reinterpret_cast<uintptr_t>(radii) | reinterpret_cast<uintptr_t>(means2d) |
         reinterpret_cast<uintptr_t>(radii_float)) & 7u)
        return GS_ERR_INVALID_ARG;
    const ProjectArgs pa{width, height, orthographic ? 1 : 0, eps2d, near_plane, far_plane,
                         radius_clip};
    launch_project(means, covars, viewmats, intrinsics, C, N, pa, radii, means2d, depths, conics,
                   compensations, radii_float, static_cast<cudaStream_t>(stream));
    return check_launch();
}

size_t gs_sort_workspace_size(int64_t n) {
    if (n < 0) return 0;
    Carver cv{nullptr};
    cv.take<int32_t>(1);
    cv.take<uint32_t>(kMaxPasses);
    cv.take<uint32_t>(kMaxPasses * 256);
    for (int i = 0; i < kMaxPasses; ++i) cv.take<uint64_t>((size_t)sort_blocks(n, kTile64) * 256);
    cv.take<uint64_t>((size_t)n);
    cv.take<int32_t>((size_t)n);
    return cv.used;
}

int gs_sort_pairs(uint64_t* keys, int32_t* values, int64_t n, int begin_bit, int end_bit,
                  void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
    if (n < 0 || n >= ((int64_t)1 << 31) || begin_bit < 0 || end_bit > 64 ||
        begin_bit > end_bit || (n > 0 && (!keys || !values)))
        return GS_ERR_INVALID_ARG;
    if (n <= 1 || begin_bit == end_bit) return GS_OK;
    if (!workspace || workspace_bytes < gs_sort_workspace_size(n)) return GS_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int passes = (end_bit - begin_bit + 7) / 8;
    Carver cv{static_cast<char*>(workspace)};
    int32_t* abort_flag = cv.take<int32_t>(1);
    uint32_t* tickets = cv.take<uint32_t>(kMaxPasses);
    uint32_t* hist = cv.take<uint32_t>(kMaxPasses * 256);
    uint64_t* lb[kMaxPasses];
    for (int i = 0; i < kMaxPasses; ++i)
        lb[i] = cv.take<uint64_t>((size_t)sort_blocks(n, kTile64) * 256);
    const size_t zero_end = cv.used;
    uint64_t* alt_k = cv.take<uint64_t>((size_t)n);
    int32_t* alt_v = cv.take<int32_t>((size_t)n);
    if (cudaMemsetAsync(workspace, 0, zero_end, s) != cudaSuccess) return GS_ERR_CUDA;
    launch_digit_hist_u64(keys, n, begin_bit, end_bit, hist, s);
    uint64_t* sk = keys;
    int32_t* sv = values;
    for (int pass = 0; pass < passes; ++pass) {
        uint64_t* dk = sk == keys ? alt_k : keys;
        int32_t* dv = sv == values ? alt_v : values;
        launch_onesweep_u64(sk, sv, dk, dv, n, begin_bit + 8 * pass, end_bit, hist + 256 * pass,
                            LookbackScratch{lb[pass], tickets + pass}, abort_flag, d_status, s);
        sk = dk;
        sv = dv;
    }
    if (sk != keys) {
        if (cudaMemcpyAsync(keys, sk, (size_t)n * 8, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(values, sv, (size_t)n * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return GS_ERR_CUDA;
    }
    return check_launch();
}

int gs_debug_sort_wait_timeout(uint64_t* keys, int32_t* values, int64_t n, int ticket_start,
                               int wait_polls, void* workspace, size_t workspace_bytes,
                               int32_t* d_status, void* stream) {
    if (n < 1 || n >= ((int64_t)1 << 30) || !keys || !values || !d_status ||
        ticket_start < 1 || ticket_start > kMaxDebugTickets || wait_polls < 1 ||
        wait_polls > kMaxDebugPolls)
        return GS_ERR_INVALID_ARG;
    const int64_t n_virtual = n + (int64_t)ticket_start * kTile64;
    if (!workspace || workspace_bytes < gs_sort_workspace_size(n_virtual)) return GS_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the layout of gs_sort_pairs for n_virtual pairs: its first look-back
    // region has a word per digit for every virtual block the pass can name
    // (tickets ticket_start .. ticket_start + blocks(n) - 1)
    Carver cv{static_cast<char*>(workspace)};
    int32_t* abort_flag = cv.take<int32_t>(1);
    uint32_t* tickets = cv.take<uint32_t>(kMaxPasses);
    uint32_t* hist = cv.take<uint32_t>(kMaxPasses * 256);
    uint64_t* lb0 = cv.take<uint64_t>((size_t)sort_blocks(n_virtual, kTile64) * 256);
    for (int i = 1; i < kMaxPasses; ++i)
        cv.take<uint64_t>((size_t)sort_blocks(n_virtual, kTile64) * 256);
    const size_t zero_end = cv.used;
    uint64_t* alt_k = cv.take<uint64_t>((size_t)n);
    int32_t* alt_v = cv.take<int32_t>((size_t)n);
    if (cudaMemsetAsync(workspace, 0, zero_end, s) != cudaSuccess) return GS_ERR_CUDA;
    const uint32_t first = (uint32_t)ticket_start;
    // from a host variable: the copy has been staged when the call returns
    if (cudaMemcpyAsync(tickets, &first, sizeof(first), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GS_ERR_CUDA;
    launch_digit_hist_u64(keys, n, 0, 8, hist, s);
    launch_onesweep_u64(keys, values, alt_k, alt_v, n, 0, 8, hist, LookbackScratch{lb0, tickets},
                        abort_flag, d_status, s, wait_polls);
    return check_launch();
}

int gs_peak_probe(int kind, int iters, int blocks, float* out, int64_t* h_ops, void* stream) {
    if (kind < 0 || kind > 2 || iters < 1 || blocks < 1 || !out || !h_ops)
        return GS_ERR_INVALID_ARG;
    *h_ops = launch_peak_probe(kind, iters, blocks, out, static_cast<cudaStream_t>(stream));
    return check_launch();
}

}  // extern "C"
