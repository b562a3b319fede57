// Forward compositing and its reverse-walk backward, one block per 16x16
// tile, PPT pixels per thread in a vertical strip (thread t owns column
// t % 16 and rows (t / 16) * PPT .. + PPT - 1 of the tile).
//
// Why strips: a splat record read from shared memory serves PPT pixels, and
// the terms of the quadratic form that depend only on dx (a dx dx, b dx) are
// computed once per thread and entry -- in the same rounding order as the
// per-pixel formula, so results do not change.  In the backward a warp covers
// 32 * PPT pixels, so the shuffle reduction of a splat's terms (and its
// atomics) is paid once per 32 * PPT pixels.
//
// Forward: the tile's sorted list is streamed through shared memory in
// batches (records gathered through flatten_ids); a warp skips a batch when
// all its pixels have stopped, and the block ends when every pixel has
// (__syncthreads_count vote).
//
// Backward (gsplat 1.0.0, raster_backward.c, gs_raster_backward_pixel): the
// list is walked from the largest last_id of the tile down to the tile's
// start; a warp skips entries beyond the largest last_id of its own pixels.
// Each thread sums its pixels' terms in registers, the warp sums them with
// shuffles, and lane 0 adds them to the gradients with one atomic per field
// (the shuffle-then-atomic pattern of the mxnet depthwise backward-filter
// kernel).  Warps with no valid pair for an entry skip both.
//
// alpha is computed by the same inline code in both kernels, so the backward
// makes exactly the forward's skip/composite decisions.
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kTile = 16;
constexpr int kPPT = 4;                          // pixels per thread
constexpr int kThreads = kTile * kTile / kPPT;   // 64
constexpr int kBatch = 2 * kThreads;             // records staged per batch
constexpr float kAlphaClamp = 0.99f;

// Per-entry terms shared by the PPT pixels of one column.
struct ColumnTerms {
    float dx, qa, bdx;  // dx = mx - px, qa = (a dx) dx, bdx = b dx
};

__device__ __forceinline__ ColumnTerms column_terms(float mx, float a, float b, float px) {
    ColumnTerms t;
    t.dx = __fsub_rn(mx, px);
    t.qa = __fmul_rn(__fmul_rn(a, t.dx), t.dx);
    t.bdx = __fmul_rn(b, t.dx);
    return t;
}

struct PairEval {
    float dy, s, resp, raw, alpha;
};

// s = 0.5 (a dx^2 + c dy^2) + b dx dy rounded exactly as written (no FMA
// contraction), alpha = min(0.99, o exp(-s)).
__device__ __forceinline__ PairEval eval_pair(const ColumnTerms& ct, float my, float c, float op,
                                              float py) {
    PairEval e;
    e.dy = __fsub_rn(my, py);
    const float qc = __fmul_rn(__fmul_rn(c, e.dy), e.dy);
    const float qb = __fmul_rn(ct.bdx, e.dy);
    e.s = __fadd_rn(__fmul_rn(0.5f, __fadd_rn(ct.qa, qc)), qb);
    e.resp = __expf(-e.s);
    e.raw = __fmul_rn(op, e.resp);
    e.alpha = e.raw > kAlphaClamp ? kAlphaClamp : e.raw;
    return e;
}

struct TileRange {
    int64_t tile, start, end;
    int c, ty, tx;
    bool masked;
};

__device__ __forceinline__ TileRange tile_range(const RasterArgs& a) {
    TileRange r;
    r.tile = blockIdx.x;
    const int per_camera = a.tile_width * a.tile_height;
    r.c = (int)(r.tile / per_camera);
    const int local = (int)(r.tile - (int64_t)r.c * per_camera);
    r.ty = local / a.tile_width;
    r.tx = local - r.ty * a.tile_width;
    const int64_t ntiles = (int64_t)a.C * per_camera;
    r.start = a.offsets[r.tile];
    r.end = r.tile + 1 < ntiles ? (int64_t)a.offsets[r.tile + 1] : a.n_isects;
    // offsets from gs_tile_offsets are always inside [0, n_isects]; clamping
    // keeps a corrupted table from reading outside flatten_ids
    r.end = r.end < 0 ? 0 : (r.end > a.n_isects ? a.n_isects : r.end);
    r.start = r.start < 0 ? 0 : (r.start > r.end ? r.end : r.start);
    r.masked = a.masks != nullptr && a.masks[r.tile] == 0;
    if (r.masked) r.end = r.start;
    return r;
}

// Stages the record of list entry j into shared slot k.  A flatten id outside
// [0, C*N) (only from corrupted input) becomes a record with opacity 0, which
// never passes the cutoff.
__device__ __forceinline__ int32_t stage_record(const RasterArgs& a, int64_t j, float4* s_mo,
                                                float4* s_q, float4* s_col, int k) {
    const int64_t g = a.flatten_ids[j];
    if ((uint64_t)g >= (uint64_t)((int64_t)a.C * a.N)) {
        s_mo[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        s_q[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        s_col[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        return -1;
    }
    const float2 m = reinterpret_cast<const float2*>(a.means2d)[g];
    const float* q = a.conics + 3 * g;
    const float* col = a.colors + 3 * g;
    s_mo[k] = make_float4(m.x, m.y, a.opacities[g], 0.0f);
    s_q[k] = make_float4(q[0], q[1], q[2], 0.0f);
    s_col[k] = make_float4(col[0], col[1], col[2], 0.0f);
    return (int32_t)g;
}

struct PixelSlot {
    int x, y0;  // column and first row of the thread's strip
};

__device__ __forceinline__ PixelSlot pixel_slot(const TileRange& tr) {
    PixelSlot p;
    p.x = tr.tx * kTile + (threadIdx.x & (kTile - 1));
    p.y0 = tr.ty * kTile + (threadIdx.x / kTile) * kPPT;
    return p;
}

template <bool COUNT>
__global__ void __launch_bounds__(kThreads)
    k_raster_fwd(RasterArgs a, float* __restrict__ out_rgb, float* __restrict__ out_alpha,
                 int32_t* __restrict__ out_last, int32_t* __restrict__ out_counts) {
    __shared__ float4 s_mo[kBatch];   // mx, my, opacity, -
    __shared__ float4 s_q[kBatch];    // a, b, c, -
    __shared__ float4 s_col[kBatch];  // r, g, b, -
    const TileRange tr = tile_range(a);
    const int tid = threadIdx.x;
    const PixelSlot ps = pixel_slot(tr);
    const float px = (float)ps.x + 0.5f;
    float T[kPPT], cr[kPPT], cg[kPPT], cb[kPPT], py[kPPT];
    int32_t last[kPPT], n_eval[kPPT], n_comp[kPPT];
    bool done[kPPT];
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        T[k] = 1.0f;
        cr[k] = cg[k] = cb[k] = 0.0f;
        last[k] = -1;
        n_eval[k] = n_comp[k] = 0;
        done[k] = !(ps.x < a.width && ps.y0 + k < a.height);
        py[k] = (float)(ps.y0 + k) + 0.5f;
    }
    for (int64_t b0 = tr.start; b0 < tr.end; b0 += kBatch) {
        bool all_done = true;
#pragma unroll
        for (int k = 0; k < kPPT; ++k) all_done &= done[k];
        if (__syncthreads_count(all_done) == kThreads) break;
        const int nb = (int)min((int64_t)kBatch, tr.end - b0);
        for (int i = tid; i < nb; i += kThreads) stage_record(a, b0 + i, s_mo, s_q, s_col, i);
        __syncthreads();
        if (__all_sync(0xffffffffu, all_done)) continue;
        for (int i = 0; i < nb; ++i) {
            const float4 mo = s_mo[i];
            const float4 q = s_q[i];
            const ColumnTerms ct = column_terms(mo.x, q.x, q.y, px);
#pragma unroll
            for (int k = 0; k < kPPT; ++k) {
                if (done[k]) continue;
                const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, py[k]);
                if (COUNT) ++n_eval[k];
                if (!(e.s >= 0.0f) || e.alpha < a.alpha_cutoff) continue;
                if (COUNT) ++n_comp[k];
                const float4 col = s_col[i];
                const float w = T[k] * e.alpha;
                cr[k] += w * col.x;
                cg[k] += w * col.y;
                cb[k] += w * col.z;
                T[k] = T[k] * (1.0f - e.alpha);
                last[k] = (int32_t)(b0 + i);
                if (T[k] < a.transmittance_threshold) done[k] = true;
            }
        }
    }
    float br = 0.0f, bgc = 0.0f, bb = 0.0f;
    if (a.backgrounds) {
        br = a.backgrounds[3 * tr.c];
        bgc = a.backgrounds[3 * tr.c + 1];
        bb = a.backgrounds[3 * tr.c + 2];
    }
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        const int y = ps.y0 + k;
        if (ps.x < a.width && y < a.height) {
            const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + ps.x;
            out_rgb[3 * p] = cr[k] + T[k] * br;
            out_rgb[3 * p + 1] = cg[k] + T[k] * bgc;
            out_rgb[3 * p + 2] = cb[k] + T[k] * bb;
            out_alpha[p] = 1.0f - T[k];
            out_last[p] = last[k];
            if (COUNT) {
                out_counts[2 * p] = n_eval[k];
                out_counts[2 * p + 1] = n_comp[k];
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <bool ABS>
__global__ void __launch_bounds__(kThreads) k_raster_bwd(RasterArgs a, RasterGrads gr) {
    __shared__ float4 s_mo[kBatch];
    __shared__ float4 s_q[kBatch];
    __shared__ float4 s_col[kBatch];
    __shared__ int32_t s_gid[kBatch];
    __shared__ float s_bg[kThreads / kWarp][3];
    __shared__ int s_jmax;
    const TileRange tr = tile_range(a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const PixelSlot ps = pixel_slot(tr);
    const float px = (float)ps.x + 0.5f;

    float ra[kPPT], g0[kPPT], g1[kPPT], g2[kPPT], ga[kPPT], py[kPPT];
    float Tc[kPPT], Ta[kPPT], r0[kPPT], r1[kPPT], r2[kPPT];
    int32_t last[kPPT];
    float bg0 = 0.0f, bg1 = 0.0f, bg2 = 0.0f;
    if (a.backgrounds) {
        bg0 = a.backgrounds[3 * tr.c];
        bg1 = a.backgrounds[3 * tr.c + 1];
        bg2 = a.backgrounds[3 * tr.c + 2];
    }
    int my_max = -1;
    float sb0 = 0.0f, sb1 = 0.0f, sb2 = 0.0f;
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        const int y = ps.y0 + k;
        py[k] = (float)y + 0.5f;
        ra[k] = g0[k] = g1[k] = g2[k] = ga[k] = 0.0f;
        last[k] = -1;
        if (ps.x < a.width && y < a.height) {
            const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + ps.x;
            ra[k] = gr.render_alphas[p];
            last[k] = gr.last_ids[p];
            g0[k] = gr.grad_render_colors[3 * p];
            g1[k] = gr.grad_render_colors[3 * p + 1];
            g2[k] = gr.grad_render_colors[3 * p + 2];
            ga[k] = gr.grad_render_alphas[p];
        }
        Tc[k] = 1.0f - ra[k];
        Ta[k] = 1.0f;
        r0[k] = bg0;
        r1[k] = bg1;
        r2[k] = bg2;
        sb0 += g0[k] * Tc[k];
        sb1 += g1[k] * Tc[k];
        sb2 += g2[k] * Tc[k];
        if (ra[k] > 0.0f && last[k] > my_max) my_max = last[k];
    }
    if (tid == 0) s_jmax = -1;
    if (gr.grad_backgrounds) {
        sb0 = warp_sum(sb0);
        sb1 = warp_sum(sb1);
        sb2 = warp_sum(sb2);
        if (lane == 0) {
            s_bg[warp][0] = sb0;
            s_bg[warp][1] = sb1;
            s_bg[warp][2] = sb2;
        }
    }
    __syncthreads();
    if (gr.grad_backgrounds && tid < 3) {
        float v = 0.0f;
        for (int w = 0; w < kThreads / kWarp; ++w) v += s_bg[w][tid];
        atomicAdd(&gr.grad_backgrounds[3 * tr.c + tid], v);
    }
    if (tr.masked || tr.start == tr.end) return;
    const int warp_max = __reduce_max_sync(0xffffffffu, my_max);
    if (lane == 0) atomicMax(&s_jmax, warp_max);
    __syncthreads();
    const int64_t walk_end = min(tr.end, (int64_t)s_jmax + 1);
    for (int64_t b1 = walk_end; b1 > tr.start; b1 -= kBatch) {
        const int64_t b0 = max(tr.start, b1 - kBatch);
        const int nb = (int)(b1 - b0);
        __syncthreads();
        for (int i = tid; i < nb; i += kThreads)
            s_gid[i] = stage_record(a, b1 - 1 - i, s_mo, s_q, s_col, i);
        __syncthreads();
        // entries of this batch beyond the warp's largest last_id are skipped
        const int first = (int)max((int64_t)0, b1 - 1 - (int64_t)warp_max);
        for (int i = first; i < nb; ++i) {
            const int64_t j = b1 - 1 - i;
            const float4 mo = s_mo[i];
            const float4 q = s_q[i];
            const float4 col = s_col[i];
            const ColumnTerms ct = column_terms(mo.x, q.x, q.y, px);
            const float hdx2 = 0.5f * ct.dx * ct.dx;
            float v_c0 = 0.f, v_c1 = 0.f, v_c2 = 0.f, v_op = 0.f, v_mx = 0.f, v_my = 0.f;
            float v_qa = 0.f, v_qb = 0.f, v_qc = 0.f, v_ax = 0.f, v_ay = 0.f;
            bool any = false;
#pragma unroll
            for (int k = 0; k < kPPT; ++k) {
                const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, py[k]);
                const bool valid = ra[k] > 0.0f && e.s >= 0.0f && e.alpha >= a.alpha_cutoff &&
                                   (int64_t)last[k] >= j && Tc[k] < 1.0f && e.alpha < 1.0f;
                if (!valid) continue;
                any = true;
                const float one_m = 1.0f - e.alpha;
                const float Tb = __fdividef(Tc[k], one_m);
                const float vis = Tb * e.alpha;
                v_c0 += g0[k] * vis;
                v_c1 += g1[k] * vis;
                v_c2 += g2[k] * vis;
                const float dot = g0[k] * (col.x - r0[k]) + g1[k] * (col.y - r1[k]) +
                                  g2[k] * (col.z - r2[k]);
                const float g_alpha = Tb * (dot + ga[k] * Ta[k]);
                const float g_raw = e.raw < kAlphaClamp ? g_alpha : 0.0f;
                v_op += g_raw * e.resp;
                const float g_s = -g_raw * e.raw;
                const float mx = g_s * (q.x * ct.dx + q.y * e.dy);
                const float my = g_s * (q.z * e.dy + q.y * ct.dx);
                v_mx += mx;
                v_my += my;
                if (ABS) {
                    v_ax += fabsf(mx);
                    v_ay += fabsf(my);
                }
                v_qa += g_s * hdx2;
                v_qb += g_s * (ct.dx * e.dy);
                v_qc += g_s * (0.5f * e.dy * e.dy);
                r0[k] = e.alpha * col.x + one_m * r0[k];
                r1[k] = e.alpha * col.y + one_m * r1[k];
                r2[k] = e.alpha * col.z + one_m * r2[k];
                Ta[k] *= one_m;
                Tc[k] = Tb;
            }
            if (!__any_sync(0xffffffffu, any)) continue;
            v_c0 = warp_sum(v_c0);
            v_c1 = warp_sum(v_c1);
            v_c2 = warp_sum(v_c2);
            v_op = warp_sum(v_op);
            v_mx = warp_sum(v_mx);
            v_my = warp_sum(v_my);
            v_qa = warp_sum(v_qa);
            v_qb = warp_sum(v_qb);
            v_qc = warp_sum(v_qc);
            if (ABS) {
                v_ax = warp_sum(v_ax);
                v_ay = warp_sum(v_ay);
            }
            if (lane == 0 && s_gid[i] >= 0) {
                const int64_t g = s_gid[i];
                atomicAdd(&gr.grad_colors[3 * g], v_c0);
                atomicAdd(&gr.grad_colors[3 * g + 1], v_c1);
                atomicAdd(&gr.grad_colors[3 * g + 2], v_c2);
                atomicAdd(&gr.grad_opacities[g], v_op);
                atomicAdd(&gr.grad_means2d[2 * g], v_mx);
                atomicAdd(&gr.grad_means2d[2 * g + 1], v_my);
                atomicAdd(&gr.grad_conics[3 * g], v_qa);
                atomicAdd(&gr.grad_conics[3 * g + 1], v_qb);
                atomicAdd(&gr.grad_conics[3 * g + 2], v_qc);
                if (ABS) {
                    atomicAdd(&gr.grad_means2d_abs[2 * g], v_ax);
                    atomicAdd(&gr.grad_means2d_abs[2 * g + 1], v_ay);
                }
            }
        }
    }
}

}  // namespace

void launch_raster_fwd(const RasterArgs& a, float* render_colors, float* render_alphas,
                       int32_t* last_ids, int32_t* pair_counts, cudaStream_t s) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    if (tiles <= 0) return;
    if (pair_counts)
        k_raster_fwd<true><<<(unsigned)tiles, kThreads, 0, s>>>(a, render_colors, render_alphas,
                                                                last_ids, pair_counts);
    else
        k_raster_fwd<false><<<(unsigned)tiles, kThreads, 0, s>>>(a, render_colors, render_alphas,
                                                                 last_ids, nullptr);
}

void launch_raster_bwd(const RasterArgs& a, const RasterGrads& g, cudaStream_t s) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    if (tiles <= 0) return;
    if (g.grad_means2d_abs)
        k_raster_bwd<true><<<(unsigned)tiles, kThreads, 0, s>>>(a, g);
    else
        k_raster_bwd<false><<<(unsigned)tiles, kThreads, 0, s>>>(a, g);
}

}  // namespace gs
