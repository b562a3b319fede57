/*
 * gs_splat.h -- C ABI of the GB300 (sm_103a) tile-binned Gaussian-splat
 * raster library (libgs_splat_gb300.so).
 *
 * The path has four calls, in order (gs_project, before them, makes their
 * 2D inputs from 3D Gaussians):
 *   gs_isect_tiles    tile rect of every splat, 64-bit intersection keys
 *                     (camera | tile | depth bits) with flatten ids, sorted
 *   gs_tile_offsets   first list position of every tile
 *   gs_rasterize_fwd  front-to-back compositing of each tile's sorted list
 *   gs_rasterize_bwd  reverse walk giving per-splat gradients
 *
 * Sources (page title, file, function):
 *   gsplat 1.0.0, data/ext/gsplat_native/intersections.c:
 *       gs_tile_bits, gs_bounds, gs_isect_tiles, gs_radix_sort_without_gvl,
 *       gs_offset_encode
 *   gsplat 1.0.0, data/ext/gsplat_native/projection.c: gs_project_one,
 *       gs_projection_forward
 *   pytorch3d rasterize_meshes.cu, RasterizeMeshesFineCudaKernel: the
 *       fixed-capacity bin layout of gs_bin_splats
 *   gsplat 1.0.0, data/ext/gsplat_native/raster_backward.c and
 *       raster_backward_bridge.c: gs_raster_backward_pixel,
 *       gs_raster_backward_without_gvl, gs_raster_backward
 *   rlx-metal 0.2.9, src/splat_training.rs: training_forward_metal_traced
 *       (alpha_cutoff, transmittance_threshold)
 *
 * Conventions for every call:
 *   - Array arguments are DEVICE pointers owned by the caller, C-contiguous,
 *     row-major, in the dtype named.  Host pointers are marked "host".
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it; no call synchronises it except the
 *     size query of gs_isect_tiles (documented there).
 *   - The library never allocates device memory.  Scratch space is the
 *     caller's `workspace` (size from the matching *_workspace_size call).
 *   - Every call returns a gs_status.  Argument errors are found on the host
 *     before anything is enqueued, and nothing is written then.  Errors only
 *     the GPU can see (a key outside the grid, a total that differs from the
 *     caller's, a wait that ran out) are written to `d_status`, an optional
 *     device int32 that the caller zeroes beforehand; the library only ever
 *     stores a nonzero code there (the first error wins).  NULL = not reported.
 *   - No call traps, asserts or aborts.
 */
#ifndef GS_SPLAT_H
#define GS_SPLAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gs_status {
    GS_OK = 0,
    GS_ERR_INVALID_ARG = 1,    /* bad pointer, size, shape or option          */
    GS_ERR_CAPACITY = 2,       /* more intersections than the buffers hold   */
    GS_ERR_KEY_OUT_OF_GRID = 3,/* key names camera >= C or tile >= TW*TH     */
    GS_ERR_WORKSPACE = 4,      /* workspace missing or smaller than needed   */
    GS_ERR_TIMEOUT = 5,        /* a bounded inter-block wait ran out         */
    GS_ERR_CUDA = 6,           /* a CUDA runtime call failed                 */
    GS_ERR_UNSORTED = 7,       /* gs_tile_offsets was given unsorted keys    */
    GS_ERR_COUNT_MISMATCH = 8, /* n_isects differs from the emitted total    */
    GS_ERR_OUT_OF_BOUNDS = 9   /* an index read from the inputs (a list range,
                                  a flatten id) lies outside its array; only the
                                  range-checking build (GS_DEBUG_BOUNDS) reports
                                  it -- every build skips such an access */
} gs_status;

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gs_version(void);

/* Static English text for a status code. */
const char* gs_status_string(int status);

/* gsplat 1.0.0, intersections.c, gs_tile_bits: the fewest bits b with
 * 2^b >= tile_width * tile_height (0 for a single tile). */
int gs_tile_bits(int tile_width, int tile_height);

/* Bytes of workspace gs_isect_tiles needs.  n_isects = 0 gives the size of
 * the size-query call; the emitting call needs the size for its n_isects. */
size_t gs_isect_workspace_size(int C, int N, int tile_width, int tile_height,
                               int64_t n_isects, int sort);

/*
 * gs_isect_tiles -- gsplat 1.0.0, intersections.c, gs_bounds and
 * gs_isect_tiles (+ gs_radix_sort_without_gvl when sort != 0).
 *
 * Inputs (device):
 *   means2d  float32 (C, N, 2)   splat centres in pixels
 *   radii    float32 (C, N) if elliptical == 0 (isotropic, ry = rx),
 *            float32 (C, N, 2) if elliptical != 0 (rx, ry)
 *   depths   float32 (C, N)
 * Per splat i = c*N + n the tile rect is
 *   x0 = clamp(floor((mx - rx) / tile_size), 0, tile_width)
 *   x1 = clamp(ceil ((mx + rx) / tile_size), 0, tile_width)   (y likewise)
 * in IEEE single precision; rx <= 0 or ry <= 0, or a non-finite mean or
 * radius, gives an empty rect; a finite value beyond the grid clamps to
 * its edge.  tiles_per_gauss[i] = (x1 - x0) * (y1 - y0).
 * For every covered tile (ty, tx) one intersection is emitted:
 *   key = ((c << tile_bits | (ty * tile_width + tx)) << 32) | bits(depth_i)
 *   flatten_id = c*N + n
 * With sort == 0 they are in emission order (camera, splat, ty, tx); with
 * sort != 0 they are sorted ascending by key, equal keys in emission order
 * (a stable sort).  Both orders match the CPU listing bit for bit.
 *
 * Two calls:
 *   1. Size query: keys == NULL.  Writes tiles_per_gauss (if not NULL) and
 *      the total count I to *h_n_isects (host).  This call synchronises
 *      `stream`, because the caller must size keys/flatten_ids from I.  The
 *      count reaches the host through one word of mapped pinned host memory
 *      that the library allocates once per calling thread and device (kept
 *      for the thread's lifetime), so the query does not wait behind large
 *      host<->device copies queued on other streams.
 *      workspace needs gs_isect_workspace_size(C, N, TW, TH, 0, sort).
 *   2. Emit: keys != NULL, n_isects = I from the query.  Writes keys
 *      uint64 (I), flatten_ids int32 (I) and, if not NULL, tiles_per_gauss
 *      int32 (C, N).  Asynchronous.  If the emitted total differs from
 *      n_isects, GS_ERR_COUNT_MISMATCH goes to d_status and at most
 *      n_isects entries are written.
 * Limits: C >= 1, N >= 0, C*N < 2^31, tile_size >= 1, tile dims >= 1,
 * tile_bits + bitlen(C-1) <= 32, I < 2^31.
 */
int gs_isect_tiles(const float* means2d, const float* radii, int elliptical,
                   const float* depths, int C, int N, int tile_size,
                   int tile_width, int tile_height, int sort,
                   int32_t* tiles_per_gauss, int64_t* h_n_isects,
                   uint64_t* keys, int32_t* flatten_ids, int64_t n_isects,
                   void* workspace, size_t workspace_bytes,
                   int32_t* d_status, void* stream);

/*
 * gs_tile_offsets -- gsplat 1.0.0, intersections.c, gs_offset_encode.
 * offsets int32 (C, tile_height, tile_width): offsets[t] = number of keys
 * whose tile (camera * tile_width * tile_height + tile) is below t, i.e. the
 * first list position of tile t; an empty tile gets the next tile's start.
 * A tile's list ends at offsets[t + 1], or at n_isects for the last tile.
 * keys must be sorted ascending (as gs_isect_tiles with sort != 0 leaves
 * them): the start of each tile is found where the tile id changes.
 * Out-of-grid keys (camera >= C or tile >= TW*TH) report
 * GS_ERR_KEY_OUT_OF_GRID and unsorted keys GS_ERR_UNSORTED in d_status;
 * offsets are then unspecified.
 */
int gs_tile_offsets(const uint64_t* keys, int64_t n_isects, int C,
                    int tile_width, int tile_height, int32_t* offsets,
                    int32_t* d_status, void* stream);

/*
 * gs_project -- gsplat 1.0.0, data/ext/gsplat_native/projection.c,
 * gs_project_one (per camera c and Gaussian n) and gs_projection_forward
 * (argument and output set).  Produces the 2D inputs of gs_isect_tiles and
 * gs_rasterize_fwd from 3D Gaussians.
 *   p = R mean + t, depth = p.z, S = (R Sigma) R^T   (R, t from viewmats[c])
 *   z = depth, or 1 when depth <= near_plane or depth >= far_plane
 *   perspective: J = [[fx/z, 0, -fx tx/z^2], [0, fy/z, -fy ty/z^2]] with
 *     tx/z, ty/z clamped to the image extent widened by 0.15 of the image
 *     size on each side; means2d = (K row 0, K row 1) . (p.x, p.y, z) / z
 *   orthographic (orthographic != 0): J = [[fx, 0, 0], [0, fy, 0]],
 *     means2d = (fx p.x + cx, fy p.y + cy)
 *   cov = J S J^T; det0 = det(cov); cov += eps2d I; det = det(cov)
 *   r_i = ceil(3.33 sqrt(max(cov_ii, 0))) (saturating at 2^31 - 1)
 *   visible = det > 0, near < depth < far, r_x or r_y above radius_clip,
 *     and the box means2d +- r overlapping [0, W] x [0, H]
 *   radii = visible ? r : 0; conics = (cov_11, -(cov_01 + cov_10) / 2,
 *     cov_00) / det' with det' = det, or 1e-10 when det <= 0;
 *   compensations = sqrt(max(det0 / det', 0)).
 * Every operation is one IEEE single-precision operation in the order
 * above (no fused multiply-add), so results are reproducible bit for bit.
 * Inputs (device, float32): means (N,3), covars (N,3,3) (symmetric),
 *   viewmats (C,4,4) world-to-camera row-major [R | t], intrinsics (C,3,3)
 *   [[fx, skew, cx], [k10, fy, cy], [0, 0, 1]].
 * Outputs, indexed c*N + n: radii int32 (C,N,2), means2d float32 (C,N,2),
 *   depths (C,N), conics (C,N,3) (written for every pair, visible or not);
 *   compensations (C,N) or NULL; radii_float float32 (C,N,2) or NULL: the
 *   radii as floats, the form gs_isect_tiles takes (elliptical).
 *   radii, means2d and radii_float must be 8-byte aligned.
 * Limits: C >= 1, N >= 0, C*N < 2^31, width, height >= 1.
 */
int gs_project(const float* means, const float* covars, const float* viewmats,
               const float* intrinsics, int C, int N, int width, int height,
               float eps2d, float near_plane, float far_plane, float radius_clip,
               int orthographic, int32_t* radii, float* means2d, float* depths,
               float* conics, float* compensations, float* radii_float,
               int32_t* d_status, void* stream);

/* Largest capacity (slots per bin) of the bin-list calls. */
#define GS_BIN_MAX_CAPACITY 16384

/*
 * gs_bin_splats -- fixed-capacity per-tile bin lists, the bin_faces layout
 * of the pytorch3d fine rasterizer (rasterize_meshes.cu,
 * RasterizeMeshesFineCudaKernel: (N, BH, BW, M) int32, -1 as sentinel),
 * holding for every tile the splats whose rect covers it (the rect of
 * gs_isect_tiles) in compositing order: ascending depth bits, ties by splat
 * index -- exactly the tile's slice of gs_isect_tiles' sorted flatten_ids,
 * without a global sort.
 * Inputs: as gs_isect_tiles (means2d, radii, elliptical, depths, C, N,
 *   tile_size, tile grid); capacity M in [1, GS_BIN_MAX_CAPACITY] with
 *   C * TH * TW * M < 2^31.
 * Outputs (device): bins int32 (C, TH, TW, M): bin t's splats (flatten ids
 *   c*N + n) in slots [0, min(count, M)), -1 after; bin_counts int32
 *   (C, TH, TW): the number of splats covering each tile (zeroed by this
 *   call; may exceed M).  A bin with more than M splats reports
 *   GS_ERR_CAPACITY to d_status and then holds M of them, which ones being
 *   unspecified; retry with M >= the largest count.
 * Asynchronous; needs no workspace.
 */
int gs_bin_splats(const float* means2d, const float* radii, int elliptical,
                  const float* depths, int C, int N, int tile_size,
                  int tile_width, int tile_height, int capacity, int32_t* bins,
                  int32_t* bin_counts, int32_t* d_status, void* stream);

/*
 * gs_rasterize_fwd_bins / gs_rasterize_bwd_bins -- gs_rasterize_fwd and
 * gs_rasterize_bwd over bin lists instead of (offsets, flatten_ids): tile
 * t's list is bins[t, 0 .. min(bin_counts[t], capacity)).  List positions
 * (last_ids, trace rows) are positions in the bins array, t * capacity + k;
 * the optional trace has C * TH * TW * capacity rows of 8 words.  Everything
 * else (arguments, outputs, errors) as the sorted-list calls.
 */
int gs_rasterize_fwd_bins(const float* means2d, const float* conics,
                          const float* colors, const float* opacities,
                          const float* backgrounds, const int32_t* masks,
                          int C, int N, int channels, int width, int height,
                          int tile_size, const int32_t* bins,
                          const int32_t* bin_counts, int capacity,
                          float alpha_cutoff, float transmittance_threshold,
                          float* render_colors, float* render_alphas,
                          int32_t* last_ids, int32_t* pair_counts,
                          uint32_t* trace, int32_t* d_status, void* stream);
int gs_rasterize_bwd_bins(const float* means2d, const float* conics,
                          const float* colors, const float* opacities,
                          const float* backgrounds, const int32_t* masks,
                          int C, int N, int channels, int width, int height,
                          int tile_size, const int32_t* bins,
                          const int32_t* bin_counts, int capacity,
                          float alpha_cutoff, const float* render_alphas,
                          const int32_t* last_ids,
                          const float* grad_render_colors,
                          const float* grad_render_alphas, float* grad_means2d,
                          float* grad_conics, float* grad_colors,
                          float* grad_opacities, float* grad_backgrounds,
                          float* grad_means2d_abs, const uint32_t* trace,
                          int32_t* d_status, void* stream);

/* Largest channel count the rasterizer accepts. */
#define GS_MAX_CHANNELS 1024

/*
 * gs_rasterize_fwd -- front-to-back compositing (the recurrence whose
 * reverse walk is gsplat 1.0.0, raster_backward.c, gs_raster_backward_pixel;
 * parameters of rlx-metal 0.2.9, splat_training.rs).
 * For pixel (x, y) of camera c in tile t, over list positions
 * j = offsets[t] .. end(t)-1, g = flatten_ids[j]:
 *   d = means2d[g] - (x + 0.5, y + 0.5)
 *   s = 0.5 (a dx^2 + c dy^2) + b dx dy      conics[g] = (a, b, c)
 *   skip unless s >= 0;  alpha = min(0.99, opacities[g] exp(-s))
 *   skip if alpha < alpha_cutoff
 *   rgb += T alpha colors[g];  T *= 1 - alpha;  last = j
 *   stop once T < transmittance_threshold (after compositing that splat)
 * render_colors = rgb + T * backgrounds[c] (0 if backgrounds == NULL),
 * render_alphas = 1 - T, last_ids = last (-1 if none).  A tile with
 * masks[t] == 0 composites nothing.
 * Inputs: means2d (C,N,2), conics (C,N,3), colors (C,N,channels),
 *   opacities (C,N), backgrounds (C,channels) or NULL, masks int32
 *   (C,TH,TW) or NULL, offsets int32 (C,TH,TW), flatten_ids int32
 *   (n_isects) -- flatten ids index the (C*N) splat arrays.
 * Outputs: render_colors float32 (C,H,W,channels), render_alphas float32
 *   (C,H,W,1), last_ids int32 (C,H,W); pair_counts int32 (C,H,W,3) or NULL:
 *   a work measure per pixel -- the list entries evaluated before the pixel
 *   stopped, the entries composited, and the entries evaluated up to and
 *   including the last composited one (entries whose splat provably cannot
 *   reach the cutoff at the pixel -- anywhere in its 8-row half of the tile --
 *   are skipped unevaluated and not counted).
 *   trace uint32 (n_isects, 8) or NULL, 16-byte aligned: per list entry, a
 *   256-bit mask of the tile's pixels that composited it (the forward's
 *   decisions, for gs_rasterize_bwd).  Words 4h .. 4h + 3 (tile rows
 *   8h .. 8h + 7) of entries past the point where every pixel of those rows
 *   had stopped are not written.  Bit layout: word
 *   w (0..7), bit l covers tile pixel column (32 (w / 4) + l) % 16, row
 *   4 ((32 (w / 4) + l) / 16) + w % 4.
 * Supported: 1 <= channels <= GS_MAX_CHANNELS, tile_size == 16;
 *   TH = ceil(H/16), TW = ceil(W/16).  Channels are composited in chunks of
 *   up to 4 per kernel launch (the walk is repeated per chunk).
 */
int gs_rasterize_fwd(const float* means2d, const float* conics,
                     const float* colors, const float* opacities,
                     const float* backgrounds, const int32_t* masks,
                     int C, int N, int channels, int width, int height,
                     int tile_size, const int32_t* offsets,
                     const int32_t* flatten_ids, int64_t n_isects,
                     float alpha_cutoff, float transmittance_threshold,
                     float* render_colors, float* render_alphas,
                     int32_t* last_ids, int32_t* pair_counts, uint32_t* trace,
                     int32_t* d_status, void* stream);

/*
 * gs_rasterize_bwd -- gsplat 1.0.0, raster_backward.c,
 * gs_raster_backward_pixel / gs_raster_backward_without_gvl, and
 * raster_backward_bridge.c, gs_raster_backward (argument and output sets).
 * Per pixel the list is walked from its end to its start.  With
 * T = 1 - render_alpha, T_after = 1, rem = background (or 0), a pair j is
 * valid when render_alpha > 0, s >= 0, alpha >= alpha_cutoff,
 * last_ids >= j, T < 1 and alpha < 1; then
 *   T_before = T / (1 - alpha), vis = T_before alpha
 *   dL/dcolors += g_rgb vis
 *   g_alpha = T_before (sum_ch g_rgb (color - rem) + g_a T_after)
 *   g_raw = raw < 0.99 ? g_alpha : 0;  dL/dopacities += g_raw exp(-s)
 *   g_s = -g_raw raw
 *   dL/dmeans2d += g_s (a dx + b dy, c dy + b dx)
 *   dL/dconics  += g_s (dx^2 / 2, dx dy, dy^2 / 2)
 *   rem = alpha color + (1 - alpha) rem; T_after *= 1 - alpha; T = T_before
 * dL/dbackgrounds += g_rgb (1 - render_alpha) per pixel.
 * grad_means2d_abs (absgrad, optional) sums |dL/dmeans2d| per pixel term.
 * trace (optional): the mask table gs_rasterize_fwd wrote for the same
 * inputs.  With it, only the pairs the forward composited are revisited;
 * without it, alpha is re-evaluated for every entry up to each pixel's
 * last_id.  Both give the same result (each pair is re-tested either way).
 * Inputs: the forward's inputs (means2d ... n_isects, alpha_cutoff),
 *   render_alphas float32 (C,H,W,1), last_ids int32 (C,H,W),
 *   grad_render_colors float32 (C,H,W,channels),
 *   grad_render_alphas float32 (C,H,W,1).
 * Outputs (zeroed by this call, then accumulated with atomics, so the sum
 * order and the last bits vary from run to run):
 *   grad_means2d (C,N,2), grad_conics (C,N,3), grad_colors (C,N,channels),
 *   grad_opacities (C,N); grad_backgrounds (C,channels) or NULL;
 *   grad_means2d_abs (C,N,2) or NULL.
 * Supported: 1 <= channels <= GS_MAX_CHANNELS, tile_size == 16.  More than
 *   4 channels run as chunks of up to 4, whose contributions add up: every
 *   term above is linear in the per-channel products.  grad_means2d_abs is
 *   not (|.| of a sum over all channels cannot be formed from per-chunk
 *   parts), so above 4 channels it comes from one more walk of the lists
 *   with the full channel sums, read from global memory for every pair.
 */
int gs_rasterize_bwd(const float* means2d, const float* conics,
                     const float* colors, const float* opacities,
                     const float* backgrounds, const int32_t* masks,
                     int C, int N, int channels, int width, int height,
                     int tile_size, const int32_t* offsets,
                     const int32_t* flatten_ids, int64_t n_isects,
                     float alpha_cutoff, const float* render_alphas,
                     const int32_t* last_ids, const float* grad_render_colors,
                     const float* grad_render_alphas, float* grad_means2d,
                     float* grad_conics, float* grad_colors,
                     float* grad_opacities, float* grad_backgrounds,
                     float* grad_means2d_abs, const uint32_t* trace,
                     int32_t* d_status, void* stream);

/*
 * gs_rasterize_fwd_steps / gs_rasterize_bwd_steps -- the forward and
 * backward over a per-pixel step trace, the trace buffers of rlx-metal 0.2.9,
 * src/splat_training.rs, training_forward_metal_traced (per-pixel splat ids up
 * to max_splat_steps), in place of gs_rasterize_fwd's per-entry masks.
 *
 * gs_rasterize_fwd_steps: gs_rasterize_fwd (same arguments, results and
 * errors; no pair counts or mask trace) that also records, for every pixel
 * p = (c * H + y) * W + x and its s-th composited pair front to back
 * (s < max_steps):
 *   step_pos int32 (max_steps, C, H, W): the pair's list position j
 *   step_T float32 (max_steps, C, H, W): the transmittance T before it
 *   step_count int32 (C, H, W): the pairs the pixel composited; it may exceed
 *     max_steps, and then only the first max_steps are recorded.
 * Records past step_count[p] are not written.
 *
 * gs_rasterize_bwd_steps: gs_rasterize_bwd's result (same gradients, same
 * zeroing, any channel count, absgrad optional) from the step trace of
 * gs_rasterize_fwd_steps on the same inputs: one thread per pixel walks the
 * pixel's records from its last to its first, so no other list entry is
 * revisited and T before each pair is read instead of recovered by a
 * division; a pixel whose step_count exceeds max_steps walks its tile's list
 * from its last id down instead, recovering T_before = T / (1 - alpha) as
 * gsplat 1.0.0, raster_backward.c, gs_raster_backward_pixel does.  The
 * pixels of a warp walk in step by list position, and each pair's terms are
 * summed over the warp before one global atomic per field (an alternative
 * to the mask-trace backward, which is cheaper; both are measured).
 * Limits: max_steps >= 1 and max_steps * C * H * W < 2^40; otherwise as the
 * forward and backward above.
 */
int gs_rasterize_fwd_steps(const float* means2d, const float* conics, const float* colors,
                           const float* opacities, const float* backgrounds,
                           const int32_t* masks, int C, int N, int channels, int width,
                           int height, int tile_size, const int32_t* offsets,
                           const int32_t* flatten_ids, int64_t n_isects, float alpha_cutoff,
                           float transmittance_threshold, int max_steps, float* render_colors,
                           float* render_alphas, int32_t* last_ids, int32_t* step_pos,
                           float* step_T, int32_t* step_count, int32_t* d_status, void* stream);
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
                           void* stream);

/* Bytes of workspace gs_sort_pairs needs for n pairs. */
size_t gs_sort_workspace_size(int64_t n);

/*
 * gs_sort_pairs -- the stable LSD radix sort of gsplat 1.0.0,
 * intersections.c, gs_radix_sort_without_gvl, restricted to the bits that
 * can differ: sorts (keys uint64 (n), values int32 (n)) in place, ascending
 * by bits [begin_bit, end_bit) of the key, equal digits keeping their input
 * order.  With begin_bit = 0, end_bit = 64 this is the listing's sort; when
 * the key bits outside the range are equal across all keys the result is
 * the full stable sort.  0 <= begin_bit <= end_bit <= 64, n < 2^31.
 */
int gs_sort_pairs(uint64_t* keys, int32_t* values, int64_t n, int begin_bit,
                  int end_bit, void* workspace, size_t workspace_bytes,
                  int32_t* d_status, void* stream);

/* Largest n gs_sort_pairs_noalloc accepts. */
#define GS_SORT_NOALLOC_MAX_PAIRS (1 << 20)

/*
 * gs_sort_pairs_noalloc -- no counterpart on the pages: a convenience for
 * callers of this library that cannot allocate device memory, such as code
 * running inside a host framework that owns every device allocation and
 * forbids others, or a loop that must never pay for an allocation, and
 * therefore cannot hand gs_sort_pairs its workspace.
 * Same result as gs_sort_pairs (stable, ascending by key bits
 * [begin_bit, end_bit), in place), but it allocates nothing and takes no
 * workspace: its scratch space is one fixed device array inside the library
 * (20,980,224 bytes, about 21.0 MB, held on every GPU that loads the library
 * until the process exits), sized for n <= GS_SORT_NOALLOC_MAX_PAIRS.
 *   - n > GS_SORT_NOALLOC_MAX_PAIRS returns GS_ERR_CAPACITY, nothing enqueued.
 *   - It runs on the current device.  Its first call on a device looks up the
 *     array's device address there (cudaGetSymbolAddress); make that first
 *     call before any stream capture.
 *   - Every call shares the one array and clears what must start at zero, so
 *     calls whose GPU work overlaps (other streams, other host threads on the
 *     same device) race: order them on one stream or synchronise between them.
 *   - keys, values: caller-owned device arrays; d_status, stream: as for every
 *     call of this library.
 */
int gs_sort_pairs_noalloc(uint64_t* keys, int32_t* values, int64_t n,
                          int begin_bit, int end_bit, int32_t* d_status,
                          void* stream);

/*
 * gs_peak_probe -- a measurement helper, not part of the path (the pages give
 * no peak figures): a kernel of blocks x 256 threads, each running 8
 * independent chains of `iters` x 4 operations of one kind:
 *   kind 0: scalar FP32 fused multiply-add (x <- 0.999 x + 0.001)
 *   kind 1: packed f32x2 fused multiply-add (the same on both halves)
 *   kind 2: the ex2.approx special-function instruction (x <- 2^-x)
 * out float32 (blocks * 256) receives each thread's sum of its chains (so no
 * work is dead); *h_ops (host) the number of operations enqueued (an FMA is
 * one operation, a packed FMA two).  Timing it with events on `stream` gives
 * the GPU's FP32-pipe and special-function throughput, the denominators of
 * the raster kernels' roofline fractions.  Asynchronous.
 */
int gs_peak_probe(int kind, int iters, int blocks, float* out, int64_t* h_ops, void* stream);

/*
 * gs_debug_sort_wait_timeout -- test hook for the failure path of the
 * bounded inter-block waits (the pages' sort, gsplat 1.0.0, intersections.c,
 * gs_radix_sort_without_gvl, returns an error instead of aborting; this makes
 * the library's equivalent error happen on purpose, without a fault).
 * Runs the histogram and ONE sorting pass of gs_sort_pairs (digit bits 0..7)
 * over keys uint64 (n), values int32 (n), with two changes:
 *   - the pass's block ticket starts at ticket_start (1 .. 64) instead of 0,
 *     so the look-back words of virtual blocks 0 .. ticket_start - 1 are
 *     never published;
 *   - a look-back wait polls a word at most wait_polls (1 .. 2^20) times,
 *     instead of 2^22, before it gives up.
 * The first block then waits on a word that nobody writes, gives up after
 * wait_polls polls and stores GS_ERR_TIMEOUT in *d_status (required, device)
 * and in the workspace's abort flag; every other waiting block sees that flag
 * within 256 polls; every block returns.  Nothing hangs and nothing faults:
 * the pass writes only inside keys/values' [0, n) ranges and the workspace,
 * but what it writes there is unspecified (callers keep a copy).
 * workspace: at least gs_sort_workspace_size(n + ticket_start * 2048) bytes.
 * Returns GS_OK once enqueued (errors of the arguments as usual); the status
 * word shows the timeout after the stream is synchronised.  1 <= n < 2^30.
 */
int gs_debug_sort_wait_timeout(uint64_t* keys, int32_t* values, int64_t n, int ticket_start,
                               int wait_polls, void* workspace, size_t workspace_bytes,
                               int32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GS_SPLAT_H */
