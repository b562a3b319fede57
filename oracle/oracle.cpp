// CPU oracle for tile-binned Gaussian-splat rasterization.
//
// TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
// restatement of what the raster path computes.  It exists to check the CUDA
// library; only the tests, the smoke check and the bench's CPU-baseline leg
// may load it.  It shares no code, header, table or helper with the CUDA
// library (tile_gaussian_splat_gb300/csrc), and the library never calls it.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared (oracle/build.py).
// Floating point: single precision where the listings use `float`, with no
// contraction into FMA, so each expression rounds exactly as written.
// Gradient accumulators are double and rounded to float once at the end.
//
// Sources (page title, file, function):
//   [G-isect]  gsplat 1.0.0, data/ext/gsplat_native/intersections.c:
//              gs_tile_bits, gs_clamp_tile, gs_bounds, gs_isect_tiles,
//              gs_radix_sort_without_gvl, gs_offset_encode.
//   [G-bwd]    gsplat 1.0.0, data/ext/gsplat_native/raster_backward.c:
//              gs_raster_backward_pixel, gs_raster_backward_without_gvl.
//   [G-bridge] gsplat 1.0.0, data/ext/gsplat_native/raster_backward_bridge.c:
//              gs_raster_backward (argument set, zeroed outputs).
//   [P3D-fine] pytorch3d rasterize_meshes.cu, RasterizeMeshesFineCudaKernel:
//              fixed-capacity bin lists with a -1 sentinel (layout only).
//   [R-train]  rlx-metal 0.2.9, src/splat_training.rs:
//              training_forward_metal_traced (alpha_cutoff,
//              transmittance_threshold), alpha_cutoff = 1/255.
// The forward compositing source is not on the pages.  It is restated as the
// recurrence whose reverse walk is [G-bwd]: alpha = min(0.99, o*exp(-s)),
// skip alpha < cutoff, T <- T(1-alpha), stop once T < threshold, then blend
// the background with the remaining T.  Readings taken where the pages are
// silent are listed next to the code that takes them.
//
// Parity status of every function here is pinned by tests/test_oracle_*.py.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// Largest channel count (the library's limit; per-pixel channel arrays are
// sized for it).
constexpr int kMaxChannels = 1024;

constexpr float kAlphaClamp = 0.99f;

// Accumulation into shared sums.  The plain build (liboracle.so, the one the
// tests load) is single-threaded and adds in pixel order.  The OpenMP build
// (liboracle_omp.so, compiled from this same file with -fopenmp, used only to
// time the oracle on all host cores) runs pixels on several threads, so its
// adds and flag stores are atomic.
// FNV-1a (64-bit) parameters of the composite-position hash.
constexpr uint64_t kHashBasis = 14695981039346656037ull;
constexpr uint64_t kHashPrime = 1099511628211ull;

inline void acc(double& dst, double v) {
#ifdef _OPENMP
#pragma omp atomic
#endif
    dst += v;
}

inline void acc_i64(int64_t& dst, int64_t v) {
#ifdef _OPENMP
#pragma omp atomic
#endif
    dst += v;
}

inline void set_flag(uint8_t& f) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
    f = 1;
}  // upper clamp of alpha (the 0.99 in the
                                      // path's statement; GS_ALPHA_CLAMP's header
                                      // is not on the pages)

// [G-isect] gs_tile_bits: the fewest bits b with 2^b >= tiles.
int tile_bits_for(int tile_width, int tile_height) {
    uint64_t tiles = (uint64_t)tile_width * (uint64_t)tile_height;
    int b = 0;
    while (((uint64_t)1 << b) < tiles) ++b;
    return b;
}

// [G-isect] gs_clamp_tile + the (int) conversion of floorf/ceilf.
// Reading: the clamp is taken on the float before conversion, which equals
// the listing whenever its conversion is defined and extends it to values
// outside the int range (they land on the grid edge).
int clamp_to_grid(float v, int maximum) {
    if (!(v > 0.0f)) return 0;  // also catches -inf
    if (v >= (float)maximum) return maximum;
    return (int)v;
}

struct Rect {
    int x0, y0, x1, y1;
};

// [G-isect] gs_bounds.  The rect is [x0,x1) x [y0,y1) in tile units.
// Reading: a non-finite mean or radius gives an empty rect (the listing's
// conversion is undefined there).
Rect bounds_of(const float* mean, const float* radius, int elliptical, int tile_size,
               int tile_width, int tile_height) {
    Rect r = {0, 0, 0, 0};
    float rx = radius[0];
    float ry = elliptical ? radius[1] : rx;
    if (!std::isfinite(mean[0]) || !std::isfinite(mean[1]) || !std::isfinite(rx) ||
        !std::isfinite(ry))
        return r;
    if (rx <= 0.0f || ry <= 0.0f) return r;
    float ts = (float)tile_size;
    r.x0 = clamp_to_grid(std::floor((mean[0] - rx) / ts), tile_width);
    r.y0 = clamp_to_grid(std::floor((mean[1] - ry) / ts), tile_height);
    r.x1 = clamp_to_grid(std::ceil((mean[0] + rx) / ts), tile_width);
    r.y1 = clamp_to_grid(std::ceil((mean[1] + ry) / ts), tile_height);
    return r;
}

uint32_t float_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

struct Pair {
    uint64_t key;
    int32_t id;
};

}  // namespace

extern "C" {

int orc_tile_bits(int tile_width, int tile_height) {
    return tile_bits_for(tile_width, tile_height);
}

// Tile rect of every splat: rects (C*N, 4) as x0, y0, x1, y1.
void orc_bounds(const float* means2d, const float* radii, int elliptical, int64_t C, int64_t N,
                int tile_size, int tile_width, int tile_height, int32_t* rects) {
    for (int64_t i = 0; i < C * N; ++i) {
        Rect r = bounds_of(means2d + 2 * i, radii + (elliptical ? 2 : 1) * i, elliptical,
                           tile_size, tile_width, tile_height);
        rects[4 * i + 0] = r.x0;
        rects[4 * i + 1] = r.y0;
        rects[4 * i + 2] = r.x1;
        rects[4 * i + 3] = r.y1;
    }
}

// [G-isect] gs_isect_tiles, first loop: tiles per splat and their total.
int64_t orc_isect_count(const float* means2d, const float* radii, int elliptical, int64_t C,
                        int64_t N, int tile_size, int tile_width, int tile_height,
                        int32_t* tiles_per_gauss) {
    int64_t total = 0;
    for (int64_t i = 0; i < C * N; ++i) {
        Rect r = bounds_of(means2d + 2 * i, radii + (elliptical ? 2 : 1) * i, elliptical,
                           tile_size, tile_width, tile_height);
        int count = (r.x1 - r.x0) * (r.y1 - r.y0);
        if (tiles_per_gauss) tiles_per_gauss[i] = count;
        total += count;
    }
    return total;
}

// [G-isect] gs_isect_tiles, second loop: one key per (splat, covered tile),
// emitted camera by camera, splat by splat, tile row by tile row.
//   key = ((camera << tile_bits | (ty * tile_width + tx)) << 32) | bits(depth)
//   id  = camera * N + splat
// `capacity` bounds the writes; the return value is the number emitted.
int64_t orc_isect_emit(const float* means2d, const float* radii, int elliptical,
                       const float* depths, int64_t C, int64_t N, int tile_size, int tile_width,
                       int tile_height, uint64_t* keys, int32_t* ids, int64_t capacity) {
    int tile_bits = tile_bits_for(tile_width, tile_height);
    int64_t w = 0;
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t i = c * N + n;
            Rect r = bounds_of(means2d + 2 * i, radii + (elliptical ? 2 : 1) * i, elliptical,
                               tile_size, tile_width, tile_height);
            if ((r.x1 - r.x0) * (r.y1 - r.y0) == 0) continue;
            uint64_t upper_camera = (uint64_t)c << tile_bits;
            uint64_t depth_bits = float_bits(depths[i]);
            for (int ty = r.y0; ty < r.y1; ++ty) {
                for (int tx = r.x0; tx < r.x1; ++tx) {
                    uint64_t tile = (uint64_t)ty * (uint64_t)tile_width + (uint64_t)tx;
                    if (w < capacity) {
                        keys[w] = ((upper_camera | tile) << 32) | depth_bits;
                        ids[w] = (int32_t)i;
                    }
                    ++w;
                }
            }
        }
    }
    return w;
}

// Stable ascending sort of (key, id) by key: the library's stable sort.
void orc_sort_stable(uint64_t* keys, int32_t* ids, int64_t n) {
    std::vector<Pair> v((size_t)n);
    for (int64_t i = 0; i < n; ++i) v[i] = Pair{keys[i], ids[i]};
    std::stable_sort(v.begin(), v.end(),
                     [](const Pair& a, const Pair& b) { return a.key < b.key; });
    for (int64_t i = 0; i < n; ++i) {
        keys[i] = v[i].key;
        ids[i] = v[i].id;
    }
}

// [G-isect] gs_radix_sort_without_gvl: least-significant-digit radix sort,
// eight passes of 8-bit digits, each a counting pass, an exclusive scan of
// the 256 counts and a stable scatter into the other buffer.  Returns 0, or
// 1 when the temporary buffers cannot be had.
int orc_sort_lsd(uint64_t* keys, int32_t* ids, int64_t n) {
    std::vector<uint64_t> k2;
    std::vector<int32_t> i2;
    try {
        k2.resize((size_t)n);
        i2.resize((size_t)n);
    } catch (...) {
        return 1;
    }
    uint64_t* src_k = keys;
    int32_t* src_i = ids;
    uint64_t* dst_k = k2.data();
    int32_t* dst_i = i2.data();
    for (int pass = 0; pass < 8; ++pass) {
        int shift = 8 * pass;
        int64_t start[256] = {0};
        for (int64_t j = 0; j < n; ++j) start[(src_k[j] >> shift) & 0xff] += 1;
        int64_t run = 0;
        for (int d = 0; d < 256; ++d) {
            int64_t cnt = start[d];
            start[d] = run;
            run += cnt;
        }
        for (int64_t j = 0; j < n; ++j) {
            int d = (int)((src_k[j] >> shift) & 0xff);
            int64_t o = start[d]++;
            dst_k[o] = src_k[j];
            dst_i[o] = src_i[j];
        }
        std::swap(src_k, dst_k);
        std::swap(src_i, dst_i);
    }
    // eight passes: the result is back in the caller's arrays
    return 0;
}

// [G-isect] gs_offset_encode: per-tile key counts, then their exclusive
// prefix sum, giving offsets (C, tile_height, tile_width).  Counting, not
// boundary detection, so unsorted keys are fine.  Returns 0, or 3 when a key
// names a camera >= C or a tile >= tile_width * tile_height (the listing
// raises an ArgError there).
int orc_tile_offsets(const uint64_t* keys, int64_t n, int C, int tile_width, int tile_height,
                     int32_t* offsets) {
    int tile_bits = tile_bits_for(tile_width, tile_height);
    uint64_t mask = tile_bits == 0 ? 0 : (((uint64_t)1 << tile_bits) - 1);
    uint64_t per_camera = (uint64_t)tile_width * (uint64_t)tile_height;
    std::vector<int64_t> counts((size_t)(C * per_camera), 0);
    for (int64_t j = 0; j < n; ++j) {
        uint64_t upper = keys[j] >> 32;
        uint64_t camera = upper >> tile_bits;
        uint64_t tile = upper & mask;
        if (camera >= (uint64_t)C || tile >= per_camera) return 3;
        counts[camera * per_camera + tile] += 1;
    }
    int64_t run = 0;
    for (size_t t = 0; t < counts.size(); ++t) {
        offsets[t] = (int32_t)run;
        run += counts[t];
    }
    return 0;
}

// Fixed-capacity bin lists (the bin_faces layout of the pytorch3d fine
// rasterizer, "pytorch3d rasterize_meshes.cu", RasterizeMeshesFineCudaKernel:
// (N, BH, BW, M) int32 with -1 as sentinel) holding, per tile, the splats
// whose rect covers it in compositing order: ascending depth bits, ties by
// splat index (the order of the stable sort of the 64-bit keys restricted
// to the tile).  counts[t] = number of covering splats (may exceed M);
// bins[t][k] for k < min(count, M), -1 after.  Reading: on overflow the bin
// keeps the first M in that order.  Returns the largest count.
int64_t orc_bin_splats(const float* means2d, const float* radii, int elliptical,
                       const float* depths, int64_t C, int64_t N, int tile_size,
                       int tile_width, int tile_height, int64_t M, int32_t* bins,
                       int32_t* counts) {
    const int64_t per_camera = (int64_t)tile_width * tile_height;
    std::vector<std::vector<int32_t>> lists((size_t)(C * per_camera));
    for (int64_t c = 0; c < C; ++c)
        for (int64_t n = 0; n < N; ++n) {
            const int64_t i = c * N + n;
            Rect r = bounds_of(means2d + 2 * i, radii + (elliptical ? 2 : 1) * i, elliptical,
                               tile_size, tile_width, tile_height);
            for (int ty = r.y0; ty < r.y1; ++ty)
                for (int tx = r.x0; tx < r.x1; ++tx)
                    lists[(size_t)(c * per_camera + (int64_t)ty * tile_width + tx)].push_back(
                        (int32_t)i);
        }
    int64_t largest = 0;
    for (size_t t = 0; t < lists.size(); ++t) {
        std::vector<int32_t>& v = lists[t];
        // splats were appended in index order; a stable sort by depth bits
        // keeps equal depths in that order
        std::stable_sort(v.begin(), v.end(), [&](int32_t x, int32_t y) {
            return float_bits(depths[x]) < float_bits(depths[y]);
        });
        counts[t] = (int32_t)v.size();
        largest = std::max<int64_t>(largest, (int64_t)v.size());
        for (int64_t k = 0; k < M; ++k)
            bins[(int64_t)t * M + k] = k < (int64_t)v.size() ? v[(size_t)k] : -1;
    }
    return largest;
}

// Forward compositing of one pixel (float, as the listings).
//   px = x + 0.5, py = y + 0.5; d = mean - pixel                 [G-bwd]
//   s = 0.5 (a dx^2 + c dy^2) + b dx dy                           [G-bwd]
//   skip unless s >= 0; alpha = min(0.99, o exp(-s));             [G-bwd]
//   skip alpha < cutoff                                            [G-bwd], [R-train]
//   rgb += T alpha color; T <- T (1 - alpha); last = j
//   stop once T < threshold (reading: the splat that crosses the threshold is
//   composited and becomes last_id, which the reverse walk's last_id >= j
//   test then includes)
//   out = rgb + T bg; out_alpha = 1 - T; last_id = -1 if nothing composited.
// Masked tiles (masks[tile] == 0) composite nothing (reading: the reverse
// walk returns before the list there).
//
// Optional outputs:
//   stats[0] += pairs evaluated (entries visited, until the pixel stops)
//   stats[1] += pairs composited
//   stats[2] += pixels flagged near-tie (below)
//   near_tie[pixel] = the number of decisions (saturating at 255) taken
//     within a relative margin:
//     |alpha - cutoff| <= tie_rel * cutoff, 0 < |s| <= tie_rel, or
//     |T - threshold| <= tie_rel_T * threshold after a composite.  At such
//     pixels an exp or rounding-order difference of a few ulp can flip the
//     decision (T carries the accumulated error of every 1 - alpha, which is
//     large relative to itself for alpha near 0.99, hence its own margin).
//   tie_splats[g] = 1 for every splat g that took part in such a decision.
//   step_pos / step_T (max_steps, C, H, W) and step_count (C, H, W), when
//     step_pos is not null: the per-pixel step trace of rlx-metal's traced
//     forward (splat_training.rs, training_forward_metal_traced): for the
//     pixel's s-th composited pair (front to back, s < max_steps) its list
//     position and the transmittance before it; step_count = the pairs the
//     pixel composited (the records stop at max_steps).
//   comp_hash[pixel] = a 64-bit FNV-1a hash of the list positions j the pixel
//     composited, in order (h = (h ^ j) * 1099511628211 from 14695981039346656037):
//     another implementation's decisions at a pixel can be compared with these
//     without listing them.
struct FwdArgs {
    const float* means2d;
    const float* conics;
    const float* colors;
    const float* opacities;
    const float* backgrounds;
    const int32_t* masks;
    int64_t C, N;
    int channels, width, height, tile_size, tile_width, tile_height;
    const int32_t* offsets;
    const int32_t* flatten_ids;
    int64_t n_isects;
    float alpha_cutoff, transmittance_threshold;
    // optional step records (see orc_rasterize_fwd)
    int max_steps;
    int32_t* step_pos;
    float* step_T;
    int32_t* step_count;
};

static void fwd_pixel(const FwdArgs& a, int64_t c, int x, int y, float* out_rgb,
                      float* out_alpha, int32_t* out_last, int64_t* stats, uint8_t* near_tie,
                      float tie_rel, float tie_rel_T, uint8_t* tie_splats, uint64_t* comp_hash) {
    int64_t tiles = (int64_t)a.C * a.tile_height * a.tile_width;
    int64_t t = (c * a.tile_height + y / a.tile_size) * a.tile_width + x / a.tile_size;
    int64_t start = a.offsets[t];
    int64_t end = t + 1 < tiles ? a.offsets[t + 1] : a.n_isects;
    float T = 1.0f;
    float rgb[kMaxChannels];
    for (int ch = 0; ch < a.channels; ++ch) rgb[ch] = 0.0f;
    int32_t last = -1;
    int64_t evaluated = 0, composited = 0;
    int n_tie = 0;  // decisions taken within the margins
    uint64_t hash = kHashBasis;  // of the composited list positions, in order
    bool masked = a.masks != nullptr && a.masks[t] == 0;
    if (!masked) {
        float px = (float)x + 0.5f, py = (float)y + 0.5f;
        for (int64_t j = start; j < end; ++j) {
            ++evaluated;
            int32_t g = a.flatten_ids[j];
            float dx = a.means2d[2 * g] - px;
            float dy = a.means2d[2 * g + 1] - py;
            const float* q = a.conics + 3 * (int64_t)g;
            float s = 0.5f * (q[0] * dx * dx + q[2] * dy * dy) + q[1] * dx * dy;
            bool pair_tie = s != 0.0f && std::fabs(s) <= tie_rel;
            if (!(s >= 0.0f)) {
                if (pair_tie && tie_splats) set_flag(tie_splats[g]);
                n_tie += pair_tie ? 1 : 0;
                continue;
            }
            float raw = a.opacities[g] * std::exp(-s);
            float alpha = raw > kAlphaClamp ? kAlphaClamp : raw;
            // a cutoff <= 0 cannot be crossed by an alpha >= 0: no tie there
            pair_tie |= a.alpha_cutoff > 0.0f &&
                        std::fabs(alpha - a.alpha_cutoff) <= tie_rel * a.alpha_cutoff;
            if (pair_tie && tie_splats) set_flag(tie_splats[g]);
            n_tie += pair_tie ? 1 : 0;
            if (alpha < a.alpha_cutoff) continue;
            float w = T * alpha;
            const float* col = a.colors + (int64_t)a.channels * g;
            for (int ch = 0; ch < a.channels; ++ch) rgb[ch] += w * col[ch];
            if (a.step_pos != nullptr && composited < a.max_steps) {
                int64_t o = composited * (a.C * a.height * (int64_t)a.width) +
                            (c * a.height + y) * (int64_t)a.width + x;
                a.step_pos[o] = (int32_t)j;
                a.step_T[o] = T;  // before this pair
            }
            T = T * (1.0f - alpha);
            last = (int32_t)j;
            ++composited;
            hash = (hash ^ (uint64_t)(uint32_t)j) * kHashPrime;
            if (std::fabs(T - a.transmittance_threshold) <=
                tie_rel_T * a.transmittance_threshold) {
                ++n_tie;
                if (tie_splats) set_flag(tie_splats[g]);
            }
            if (T < a.transmittance_threshold) break;
        }
    }
    int64_t p = (c * a.height + y) * (int64_t)a.width + x;
    for (int ch = 0; ch < a.channels; ++ch) {
        float bg = a.backgrounds ? a.backgrounds[c * a.channels + ch] : 0.0f;
        out_rgb[p * a.channels + ch] = rgb[ch] + T * bg;
    }
    out_alpha[p] = 1.0f - T;
    out_last[p] = last;
    if (stats) {
        acc_i64(stats[0], evaluated);
        acc_i64(stats[1], composited);
        acc_i64(stats[2], n_tie > 0 ? 1 : 0);
    }
    if (near_tie) near_tie[p] = (uint8_t)std::min(n_tie, 255);
    if (comp_hash) comp_hash[p] = hash;
    if (a.step_count) a.step_count[p] = (int32_t)composited;
}

// Renders every pixel (pixels == nullptr) or only the listed flat pixel
// indices p = (c*H + y)*W + x.  Outputs are full-size arrays
// render_colors (C,H,W,ch), render_alphas (C,H,W), last_ids (C,H,W); pixels
// not listed are left untouched.  Returns 0, or 1 on bad arguments.
int orc_rasterize_fwd(const float* means2d, const float* conics, const float* colors,
                      const float* opacities, const float* backgrounds, const int32_t* masks,
                      int64_t C, int64_t N, int channels, int width, int height, int tile_size,
                      int tile_width, int tile_height, const int32_t* offsets,
                      const int32_t* flatten_ids, int64_t n_isects, float alpha_cutoff,
                      float transmittance_threshold, const int64_t* pixels, int64_t n_pixels,
                      float* render_colors, float* render_alphas, int32_t* last_ids,
                      int64_t* stats, uint8_t* near_tie, float tie_rel, float tie_rel_T,
                      uint8_t* tie_splats, uint64_t* comp_hash, int max_steps,
                      int32_t* step_pos, float* step_T, int32_t* step_count) {
    if (channels < 1 || channels > kMaxChannels) return 1;
    FwdArgs a = {means2d,   conics,     colors,      opacities, backgrounds,
                 masks,     C,          N,           channels,  width,
                 height,    tile_size,  tile_width,  tile_height, offsets,
                 flatten_ids, n_isects, alpha_cutoff, transmittance_threshold,
                 max_steps, step_pos, step_T, step_count};
    if (pixels == nullptr) {
        // OpenMP build: rows of pixels handed out dynamically (list lengths,
        // and so the work per row, vary a lot)
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
#endif
        for (int64_t c = 0; c < C; ++c)
            for (int y = 0; y < height; ++y)
                for (int x = 0; x < width; ++x)
                    fwd_pixel(a, c, x, y, render_colors, render_alphas, last_ids, stats,
                              near_tie, tie_rel, tie_rel_T, tie_splats, comp_hash);
    } else {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
        for (int64_t k = 0; k < n_pixels; ++k) {
            int64_t p = pixels[k];
            int64_t c = p / ((int64_t)width * height);
            int64_t r = p % ((int64_t)width * height);
            fwd_pixel(a, c, (int)(r % width), (int)(r / width), render_colors, render_alphas,
                      last_ids, stats, near_tie, tie_rel, tie_rel_T, tie_splats, comp_hash);
        }
    }
    return 0;
}

// Double-precision twin of the forward, used only to take finite differences
// of the loss in the backward's tests.  Same recurrence, every quantity in
// double, inputs in double.  margins[0..2] receive the smallest relative
// distance seen of alpha to the cutoff, raw alpha to the 0.99 clamp and T to
// the threshold (a finite difference across one of them is meaningless).
int orc_rasterize_fwd_f64(const double* means2d, const double* conics, const double* colors,
                          const double* opacities, const double* backgrounds, int64_t C,
                          int64_t N, int channels, int width, int height, int tile_size,
                          int tile_width, int tile_height, const int32_t* offsets,
                          const int32_t* flatten_ids, int64_t n_isects, double alpha_cutoff,
                          double transmittance_threshold, double* render_colors,
                          double* render_alphas, double* margins) {
    if (channels < 1 || channels > kMaxChannels) return 1;
    (void)N;
    int64_t tiles = C * tile_height * tile_width;
    double m_cut = 1e30, m_clamp = 1e30, m_thr = 1e30;
    for (int64_t c = 0; c < C; ++c) {
        for (int y = 0; y < height; ++y) {
            for (int x = 0; x < width; ++x) {
                int64_t t = (c * tile_height + y / tile_size) * tile_width + x / tile_size;
                int64_t start = offsets[t];
                int64_t end = t + 1 < tiles ? offsets[t + 1] : n_isects;
                double T = 1.0, rgb[kMaxChannels];
                for (int ch = 0; ch < channels; ++ch) rgb[ch] = 0.0;
                double px = x + 0.5, py = y + 0.5;
                for (int64_t j = start; j < end; ++j) {
                    int32_t g = flatten_ids[j];
                    double dx = means2d[2 * g] - px, dy = means2d[2 * g + 1] - py;
                    const double* q = conics + 3 * (int64_t)g;
                    double s = 0.5 * (q[0] * dx * dx + q[2] * dy * dy) + q[1] * dx * dy;
                    if (!(s >= 0.0)) continue;
                    double raw = opacities[g] * std::exp(-s);
                    double alpha = raw > 0.99 ? 0.99 : raw;
                    m_cut = std::min(m_cut, std::fabs(alpha - alpha_cutoff) / alpha_cutoff);
                    m_clamp = std::min(m_clamp, std::fabs(raw - 0.99) / 0.99);
                    if (alpha < alpha_cutoff) continue;
                    for (int ch = 0; ch < channels; ++ch)
                        rgb[ch] += T * alpha * colors[(int64_t)channels * g + ch];
                    T = T * (1.0 - alpha);
                    m_thr = std::min(m_thr,
                                     std::fabs(T - transmittance_threshold) /
                                         transmittance_threshold);
                    if (T < transmittance_threshold) break;
                }
                int64_t p = (c * height + y) * (int64_t)width + x;
                for (int ch = 0; ch < channels; ++ch)
                    render_colors[p * channels + ch] =
                        rgb[ch] + T * (backgrounds ? backgrounds[c * channels + ch] : 0.0);
                render_alphas[p] = 1.0 - T;
            }
        }
    }
    if (margins) {
        margins[0] = m_cut;
        margins[1] = m_clamp;
        margins[2] = m_thr;
    }
    return 0;
}

// [G-bwd] gs_raster_backward_pixel / gs_raster_backward_without_gvl,
// [G-bridge] gs_raster_backward.  Per pixel, the tile's list is walked from
// its end back to its start; transmittance before each valid pair is
// recovered as T_before = T / (1 - alpha).  A pair is valid when
//   render_alpha > 0, s >= 0, alpha >= cutoff, last_id >= j, T < 1, alpha < 1.
// For a valid pair (float, as the listing):
//   vis = T_before alpha; dL/dcolor += g_rgb vis
//   dot = sum_ch g_rgb (color - rem); g_alpha = T_before (dot + g_a T_after)
//   g_raw = raw < 0.99 ? g_alpha : 0; dL/dopacity += g_raw exp(-s)
//   g_s = -g_raw raw
//   dL/dmean += g_s (a dx + b dy, c dy + b dx)   (|.| summed for absgrad)
//   dL/dconic += g_s (dx^2 / 2, dx dy, dy^2 / 2)
//   rem <- alpha color + (1 - alpha) rem; T_after *= 1 - alpha; T <- T_before
// dL/dbackground += g_rgb (1 - render_alpha) per pixel.
// Every gradient output is zeroed first (the bridge allocates them zeroed).
// Per-pair terms are float as listed; they are summed in double and rounded
// to float once.  pixels/n_pixels restricts the walk to listed pixels.
// near_tie (optional, per pixel) counts the pairs whose alpha was within
// tie_rel of the cutoff (low 4 bits) and those whose raw alpha was within
// tie_rel of the clamp (high 4 bits), each saturating at 15; tie_splats
// (optional, per splat) marks the splats of those pairs.
// step_pos / step_T / step_count (optional, the forward's step records for
// max_steps): a pixel whose records hold all its pairs visits just those and
// reads T before each instead of dividing (the trace-buffer backward of
// rlx-metal's training step); other pixels walk their list as above.
// magnitudes (optional, double) receives, per gradient element, the sum of
// the absolute values of its per-pair terms, laid out as grad_means2d (2CN),
// grad_conics (3CN), grad_colors (channels*CN), grad_opacities (CN): the
// scale of the rounding error any other summation order makes.
int orc_rasterize_bwd(const float* means2d, const float* conics, const float* colors,
                      const float* opacities, const float* backgrounds, const int32_t* masks,
                      int64_t C, int64_t N, int channels, int width, int height, int tile_size,
                      int tile_width, int tile_height, const int32_t* offsets,
                      const int32_t* flatten_ids, int64_t n_isects, float alpha_cutoff,
                      const float* render_alphas, const int32_t* last_ids,
                      const float* grad_render_colors, const float* grad_render_alphas,
                      const int64_t* pixels, int64_t n_pixels, float* grad_means2d,
                      float* grad_conics, float* grad_colors, float* grad_opacities,
                      float* grad_backgrounds, float* grad_means2d_abs, uint8_t* near_tie,
                      float tie_rel, double* magnitudes, uint8_t* tie_splats, int max_steps,
                      const int32_t* step_pos, const float* step_T,
                      const int32_t* step_count) {
    if (channels < 1 || channels > kMaxChannels) return 1;
    int64_t CN = C * N;
    std::vector<double> gm(2 * CN, 0.0), gq(3 * CN, 0.0), gc((size_t)channels * CN, 0.0),
        go(CN, 0.0), gb((size_t)channels * C, 0.0), gma(2 * CN, 0.0);
    double* mag_m = magnitudes;
    double* mag_q = magnitudes ? magnitudes + 2 * CN : nullptr;
    double* mag_c = magnitudes ? magnitudes + 5 * CN : nullptr;
    double* mag_o = magnitudes ? magnitudes + (5 + channels) * CN : nullptr;
    if (magnitudes)
        for (int64_t i = 0; i < (6 + (int64_t)channels) * CN; ++i) magnitudes[i] = 0.0;
    int64_t tiles = C * tile_height * tile_width;
    int64_t HW = (int64_t)width * height;
    int64_t count = pixels ? n_pixels : C * HW;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (int64_t k = 0; k < count; ++k) {
        int64_t p = pixels ? pixels[k] : k;
        int64_t c = p / HW;
        int x = (int)((p % HW) % width), y = (int)((p % HW) / width);
        int64_t t = (c * tile_height + y / tile_size) * tile_width + x / tile_size;
        int64_t start = offsets[t];
        int64_t end = t + 1 < tiles ? offsets[t + 1] : n_isects;
        const float* g_rgb = grad_render_colors + p * channels;
        float g_a = grad_render_alphas[p];
        float ra = render_alphas[p];
        int32_t last = last_ids[p];
        float Tc = 1.0f - ra;
        float Ta = 1.0f;
        float rem[kMaxChannels];
        int n_tie = 0, n_clamp_tie = 0;
        for (int ch = 0; ch < channels; ++ch) {
            rem[ch] = backgrounds ? backgrounds[c * channels + ch] : 0.0f;
            if (grad_backgrounds) acc(gb[c * channels + ch], (double)(g_rgb[ch] * Tc));
        }
        if (masks != nullptr && masks[t] == 0) continue;
        float px = (float)x + 0.5f, py = (float)y + 0.5f;
        // with a step trace holding all of this pixel's pairs, the recorded
        // pairs are visited (last to first) and T before each is read;
        // otherwise the list is walked and T before is recovered by division
        const int32_t n_rec = step_count ? step_count[p] : -1;
        const bool use_steps = step_count != nullptr && n_rec <= max_steps;
        const int64_t iters = use_steps ? n_rec : end - start;
        for (int64_t it = 0; it < iters; ++it) {
            int64_t j;
            float t_rec = 0.0f;
            if (use_steps) {
                int64_t o = (n_rec - 1 - it) * (C * HW) + p;
                j = step_pos[o];
                t_rec = step_T[o];
            } else {
                j = end - 1 - it;
            }
            int32_t g = flatten_ids[j];
            float dx = means2d[2 * g] - px;
            float dy = means2d[2 * g + 1] - py;
            const float* q = conics + 3 * (int64_t)g;
            float s = 0.5f * (q[0] * dx * dx + q[2] * dy * dy) + q[1] * dx * dy;
            float resp = std::exp(-s);
            float raw = opacities[g] * resp;
            float alpha = raw > kAlphaClamp ? kAlphaClamp : raw;
            bool valid = ra > 0.0f && s >= 0.0f && alpha >= alpha_cutoff && last >= j &&
                         Tc < 1.0f && alpha < 1.0f;
            if (last >= j && s >= 0.0f) {
                bool cut_tie = alpha_cutoff > 0.0f &&
                               std::fabs(alpha - alpha_cutoff) <= tie_rel * alpha_cutoff;
                bool clamp_tie = std::fabs(raw - kAlphaClamp) <= tie_rel * kAlphaClamp;
                if ((cut_tie || clamp_tie) && tie_splats) set_flag(tie_splats[g]);
                n_tie += cut_tie ? 1 : 0;
                n_clamp_tie += clamp_tie ? 1 : 0;
            }
            if (!valid) continue;
            float Tb = use_steps ? t_rec : Tc / (1.0f - alpha);
            float vis = Tb * alpha;
            const float* col = colors + (int64_t)channels * g;
            float dot = 0.0f;
            for (int ch = 0; ch < channels; ++ch) {
                acc(gc[(int64_t)channels * g + ch], (double)(g_rgb[ch] * vis));
                if (mag_c) acc(mag_c[(int64_t)channels * g + ch], std::fabs((double)(g_rgb[ch] * vis)));
                dot += g_rgb[ch] * (col[ch] - rem[ch]);
            }
            float g_alpha = Tb * (dot + g_a * Ta);
            float g_raw = raw < kAlphaClamp ? g_alpha : 0.0f;
            acc(go[g], (double)(g_raw * resp));
            float g_s = -g_raw * raw;
            float gmx = g_s * (q[0] * dx + q[1] * dy);
            float gmy = g_s * (q[2] * dy + q[1] * dx);
            acc(gm[2 * g], (double)gmx);
            acc(gm[2 * g + 1], (double)gmy);
            acc(gma[2 * g], (double)std::fabs(gmx));
            acc(gma[2 * g + 1], (double)std::fabs(gmy));
            acc(gq[3 * g], (double)(g_s * 0.5f * dx * dx));
            acc(gq[3 * g + 1], (double)(g_s * dx * dy));
            acc(gq[3 * g + 2], (double)(g_s * 0.5f * dy * dy));
            if (magnitudes) {
                acc(mag_m[2 * g], std::fabs((double)gmx));
                acc(mag_m[2 * g + 1], std::fabs((double)gmy));
                acc(mag_q[3 * g], std::fabs((double)(g_s * 0.5f * dx * dx)));
                acc(mag_q[3 * g + 1], std::fabs((double)(g_s * dx * dy)));
                acc(mag_q[3 * g + 2], std::fabs((double)(g_s * 0.5f * dy * dy)));
                acc(mag_o[g], std::fabs((double)(g_raw * resp)));
            }
            for (int ch = 0; ch < channels; ++ch)
                rem[ch] = alpha * col[ch] + (1.0f - alpha) * rem[ch];
            Ta *= 1.0f - alpha;
            Tc = Tb;
        }
        if (near_tie)
            near_tie[p] = (uint8_t)(std::min(n_tie, 15) | (std::min(n_clamp_tie, 15) << 4));
    }
    for (int64_t i = 0; i < 2 * CN; ++i) grad_means2d[i] = (float)gm[i];
    for (int64_t i = 0; i < 3 * CN; ++i) grad_conics[i] = (float)gq[i];
    for (int64_t i = 0; i < (int64_t)channels * CN; ++i) grad_colors[i] = (float)gc[i];
    for (int64_t i = 0; i < CN; ++i) grad_opacities[i] = (float)go[i];
    if (grad_backgrounds)
        for (int64_t i = 0; i < (int64_t)channels * C; ++i) grad_backgrounds[i] = (float)gb[i];
    if (grad_means2d_abs)
        for (int64_t i = 0; i < 2 * CN; ++i) grad_means2d_abs[i] = (float)gma[i];
    return 0;
}

}  // extern "C"
