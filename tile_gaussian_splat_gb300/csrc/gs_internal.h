// Host-side launchers shared between the translation units of
// libgs_splat_gb300.  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gs {

// Scratch carved from the caller's workspace (all pointers device).
struct LookbackScratch {
    uint64_t* words;   // per-block (per-digit) look-back words, zeroed per call
    uint32_t* ticket;  // virtual block counter, zeroed per call
};

// ---- sort.cu
constexpr int kSortThreads = 256;
constexpr int kItems64 = 8;   // keys per thread, 64-bit keys
constexpr int kItems32 = 12;  // keys per thread, 32-bit keys
constexpr int kTile64 = kSortThreads * kItems64;
constexpr int kTile32 = kSortThreads * kItems32;

inline int64_t sort_blocks(int64_t n, int tile) { return (n + tile - 1) / tile; }

// Digit histograms of the 8-bit digits covering bits [shift0, end_bit),
// accumulated into hist[pass][256] (zeroed by the caller).
void launch_digit_hist_u64(const uint64_t* keys, int64_t n, int shift0, int end_bit,
                           uint32_t* hist, cudaStream_t s);
void launch_digit_hist_u32(const uint32_t* keys, int64_t n, int shift0, int end_bit,
                           uint32_t* hist, cudaStream_t s);

// One stable onesweep pass over digit bits [shift, min(shift+8, end_bit)).
// vals_in ==
// nullptr means values are the element indices.  lookback needs
// sort_blocks(n, tile) * 256 words, ticket one word, both zeroed.
// spin_limit > 0 replaces the default bound on the polls of one look-back
// word (a test of the timeout path uses a small one).
void launch_onesweep_u64(const uint64_t* keys_in, const int32_t* vals_in, uint64_t* keys_out,
                         int32_t* vals_out, int64_t n, int shift, int end_bit,
                         const uint32_t* hist,
                         LookbackScratch lb, int32_t* abort_flag, int32_t* d_status,
                         cudaStream_t s, int spin_limit = 0);
void launch_onesweep_u32(const uint32_t* keys_in, const int32_t* vals_in, uint32_t* keys_out,
                         int32_t* vals_out, int64_t n, int shift, int end_bit,
                         const uint32_t* hist,
                         LookbackScratch lb, int32_t* abort_flag, int32_t* d_status,
                         cudaStream_t s);

// The same pass over 32-bit keys (with values) whose output keys are the
// 64-bit key << 32 | wide_low[value].
void launch_onesweep_u32_widen(const uint32_t* keys_in, const int32_t* vals_in,
                               uint64_t* keys_out, int32_t* vals_out, int64_t n, int shift,
                               int end_bit, const uint32_t* hist, const uint32_t* wide_low,
                               LookbackScratch lb, int32_t* abort_flag, int32_t* d_status,
                               cudaStream_t s);

// 1 / tile_size when tile_size is a power of two (then exact, and the tile
// bounds may multiply by it instead of dividing), else 0.
inline float exact_tile_inverse(int tile_size) {
    return tile_size > 0 && (tile_size & (tile_size - 1)) == 0 ? 1.0f / (float)tile_size : 0.0f;
}

// ---- isect.cu
constexpr int kIsectThreads = 256;
constexpr int kEmitChunk = 2 * kIsectThreads;  // splats per emit block

void launch_isect_count(const float* means2d, const float* radii, int elliptical, int64_t CN,
                        int tile_size, int tile_width, int tile_height, int32_t* tiles_per_gauss,
                        unsigned long long* total, cudaStream_t s);

// Emits keys/ids for splats in `order` (nullptr = index order) with a
// decoupled look-back scan of their counts.  up_hist (may be null) receives
// histograms of the up_passes 8-bit digits of the key's upper word.
// *host_word (mapped pinned host memory, device address) = *total.
void launch_publish_total(const unsigned long long* total, unsigned long long* host_word,
                          cudaStream_t s);
// Tile rects (x0, y0, x1, y1) of every splat, in index order, plus the
// histograms of the four 8-bit digits of the depth bits (hist [4][256]).
void launch_rect_hist(const float* means2d, const float* radii, int elliptical,
                      const uint32_t* dbits, int64_t CN, int tile_size, int tile_width,
                      int tile_height, int4* rects, uint32_t* hist, cudaStream_t s);
// keys != null: 64-bit keys; else 32-bit camera|tile keys into keys32.
// rects may be null (then computed from means2d and radii).
void launch_isect_emit(const float* means2d, const float* radii, int elliptical,
                       const float* depths, const int4* rects, const int32_t* order, int64_t CN,
                       int tile_size, int tile_width, int tile_height, int N, int tile_bits,
                       uint64_t* keys, uint32_t* keys32, int32_t* ids, int64_t capacity,
                       int32_t* tiles_per_gauss, LookbackScratch lb, uint32_t* up_hist,
                       int up_passes, int32_t* abort_flag, int32_t* d_status, cudaStream_t s);
// keys[i] = k32[i] << 32 | dbits[v32[i]], ids[i] = v32[i].
void launch_widen(const uint32_t* k32, const int32_t* v32, const uint32_t* dbits, int64_t n,
                  uint64_t* keys, int32_t* ids, cudaStream_t s);

void launch_tile_ranges(const uint64_t* keys, int64_t n, int C, int tile_width, int tile_height,
                        int tile_bits, int32_t* offsets, int32_t* d_status, cudaStream_t s);

// ---- raster.cu
struct RasterArgs {
    const float* means2d;
    const float* conics;
    const float* colors;
    const float* opacities;
    const float* backgrounds;
    const int32_t* masks;
    int C, N, width, height, tile_width, tile_height;
    const int32_t* offsets;
    const int32_t* flatten_ids;
    int64_t n_isects;
    float alpha_cutoff, transmittance_threshold;
    // channel chunk of this launch: colours, backgrounds, render_colors and
    // their gradients have `channels` per splat / pixel; the launch handles
    // channels [ch_off, ch_off + chunk width)
    int channels, ch_off;
    int first_chunk;  // forward: writes alphas, last ids, counts, trace;
                      // backward: adds the render_alpha gradient's terms
    // bin lists instead of offsets (offsets == nullptr): tile t's list is
    // flatten_ids[t * bin_capacity, + min(bin_counts[t], bin_capacity))
    const int32_t* bin_counts;
    int bin_capacity;
    int32_t* d_status;  // caller's status word or null
};

// Per-pixel step trace: pos int32 and T float32 (max_steps, C*H*W), count
// int32 (C*H*W).
struct StepArgs {
    int32_t* pos;
    float* T;
    int32_t* count;
    int max_steps;
};

// trace (may be null): per list entry 8 words, the tile pixels that composited it.
// steps (may be null): the per-pixel step trace to record (then no trace or
// pair counts).  Runs one launch per chunk of up to 4 channels.
void launch_raster_fwd(RasterArgs a, float* render_colors, float* render_alphas,
                       int32_t* last_ids, int32_t* pair_counts, uint32_t* trace,
                       cudaStream_t s, const StepArgs* steps = nullptr);

struct RasterGrads {
    const float* render_alphas;
    const int32_t* last_ids;
    const float* grad_render_colors;
    const float* grad_render_alphas;
    float* grad_means2d;
    float* grad_conics;
    float* grad_colors;
    float* grad_opacities;
    float* grad_backgrounds;
    float* grad_means2d_abs;
};

void launch_raster_bwd(RasterArgs a, const RasterGrads& g, const uint32_t* trace,
                       cudaStream_t s);
// The backward over a per-pixel step trace (one thread per pixel, all channels).
void launch_raster_bwd_steps(RasterArgs a, const RasterGrads& g, const StepArgs& steps,
                             cudaStream_t s);

// ---- projection (project.cu)
struct ProjectArgs {
    int width, height, orthographic;
    float eps2d, near_plane, far_plane, radius_clip;
};
// means (N,3), covars (N,3,3), viewmats (C,4,4), intrinsics (C,3,3); outputs
// indexed c*N + n; compensations and radii_float may be null.
void launch_project(const float* means, const float* covars, const float* viewmats,
                    const float* intrinsics, int C, int N, const ProjectArgs& pa, int32_t* radii,
                    float* means2d, float* depths, float* conics, float* compensations,
                    float* radii_float, cudaStream_t s);

// ---- peaks.cu
// Throughput probe: kind 0 scalar FP32 FMA, 1 packed f32x2 FMA, 2 ex2.approx;
// blocks x 256 threads, iters rounds; out gets blocks * 256 floats.  Returns
// the operations performed (an FMA is one operation, a packed FMA two).
int64_t launch_peak_probe(int kind, int iters, int blocks, float* out, cudaStream_t s);

// ---- bins.cu
// Largest bin capacity (the bin sort holds a bin's keys in shared memory).
constexpr int kMaxBinCapacity = 16384;
// Fills bins (C*TH*TW, capacity) and counts (zeroed by the caller); reports
// GS_ERR_CAPACITY to d_status for a bin with more splats than capacity.
int launch_bin_splats(const float* means2d, const float* radii, int elliptical,
                      const float* depths, int C, int N, int tile_size, int tile_width,
                      int tile_height, int capacity, int32_t* bins, int32_t* counts,
                      int32_t* d_status, cudaStream_t s);

}  // namespace gs
