// Forward compositing and its reverse-walk backward, one 256-thread block per
// 16x16 tile, one pixel per thread.
//
// Forward: the tile's sorted list is streamed through shared memory in
// batches of 256 splat records (gathered through flatten_ids, one record per
// thread); every thread walks the batch for its pixel.  A block stops as soon
// as every pixel has T < threshold (__syncthreads_count vote).
//
// Backward (gsplat 1.0.0, raster_backward.c, gs_raster_backward_pixel): the
// list is walked from the last position any pixel of the tile used down to
// the tile's start, in batches staged the same way.  Each warp sums the
// per-splat terms of its 32 pixels with shuffles before one atomic per
// gradient field (the shuffle-then-atomic pattern of the mxnet depthwise
// backward-filter kernel), and skips the sum when none of its pixels had a
// valid pair.
//
// alpha is computed by the same inline function in both kernels, so the
// backward makes exactly the forward's skip/composite decisions.
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kTile = 16;
constexpr int kThreads = kTile * kTile;
constexpr float kAlphaClamp = 0.99f;

struct PairEval {
    float dx, dy, s, resp, raw, alpha;
};

// s = 0.5 (a dx^2 + c dy^2) + b dx dy, rounded as written (no FMA
// contraction), alpha = min(0.99, o exp(-s)).
__device__ __forceinline__ PairEval eval_pair(float mx, float my, float a, float b, float c,
                                              float op, float px, float py) {
    PairEval e;
    e.dx = __fsub_rn(mx, px);
    e.dy = __fsub_rn(my, py);
    const float qa = __fmul_rn(__fmul_rn(a, e.dx), e.dx);
    const float qc = __fmul_rn(__fmul_rn(c, e.dy), e.dy);
    const float qb = __fmul_rn(__fmul_rn(b, e.dx), e.dy);
    e.s = __fadd_rn(__fmul_rn(0.5f, __fadd_rn(qa, qc)), qb);
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

template <bool COUNT>
__global__ void __launch_bounds__(kThreads)
    k_raster_fwd(RasterArgs a, float* __restrict__ out_rgb, float* __restrict__ out_alpha,
                 int32_t* __restrict__ out_last, int32_t* __restrict__ out_counts) {
    __shared__ float4 s_mo[kThreads];  // mx, my, opacity, -
    __shared__ float4 s_q[kThreads];   // a, b, c, -
    __shared__ float4 s_col[kThreads]; // r, g, b, -
    const TileRange tr = tile_range(a);
    const int tid = threadIdx.x;
    const int x = tr.tx * kTile + (tid & (kTile - 1));
    const int y = tr.ty * kTile + (tid / kTile);
    const bool inside = x < a.width && y < a.height;
    const float px = (float)x + 0.5f, py = (float)y + 0.5f;
    float T = 1.0f, cr = 0.0f, cg = 0.0f, cb = 0.0f;
    int32_t last = -1;
    int32_t n_eval = 0, n_comp = 0;
    bool done = !inside;
    for (int64_t b0 = tr.start; b0 < tr.end; b0 += kThreads) {
        if (__syncthreads_count(done) == kThreads) break;
        const int64_t j = b0 + tid;
        if (j < tr.end) stage_record(a, j, s_mo, s_q, s_col, tid);
        __syncthreads();
        const int nb = (int)min((int64_t)kThreads, tr.end - b0);
        if (!done) {
            for (int k = 0; k < nb; ++k) {
                const float4 mo = s_mo[k];
                const float4 q = s_q[k];
                const PairEval e = eval_pair(mo.x, mo.y, q.x, q.y, q.z, mo.z, px, py);
                if (COUNT) ++n_eval;
                if (!(e.s >= 0.0f) || e.alpha < a.alpha_cutoff) continue;
                if (COUNT) ++n_comp;
                const float4 col = s_col[k];
                const float w = T * e.alpha;
                cr += w * col.x;
                cg += w * col.y;
                cb += w * col.z;
                T = T * (1.0f - e.alpha);
                last = (int32_t)(b0 + k);
                if (T < a.transmittance_threshold) {
                    done = true;
                    break;
                }
            }
        }
    }
    if (inside) {
        const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + x;
        float br = 0.0f, bgc = 0.0f, bb = 0.0f;
        if (a.backgrounds) {
            br = a.backgrounds[3 * tr.c];
            bgc = a.backgrounds[3 * tr.c + 1];
            bb = a.backgrounds[3 * tr.c + 2];
        }
        out_rgb[3 * p] = cr + T * br;
        out_rgb[3 * p + 1] = cg + T * bgc;
        out_rgb[3 * p + 2] = cb + T * bb;
        out_alpha[p] = 1.0f - T;
        out_last[p] = last;
        if (COUNT) {
            out_counts[2 * p] = n_eval;
            out_counts[2 * p + 1] = n_comp;
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kThreads)
    k_raster_bwd(RasterArgs a, RasterGrads gr) {
    __shared__ float4 s_mo[kThreads];
    __shared__ float4 s_q[kThreads];
    __shared__ float4 s_col[kThreads];
    __shared__ int32_t s_gid[kThreads];
    __shared__ float s_bg[kThreads / kWarp][3];
    __shared__ int s_jmax;
    const TileRange tr = tile_range(a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int x = tr.tx * kTile + (tid & (kTile - 1));
    const int y = tr.ty * kTile + (tid / kTile);
    const bool inside = x < a.width && y < a.height;
    const float px = (float)x + 0.5f, py = (float)y + 0.5f;
    const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + x;
    float ra = 0.0f, ga = 0.0f, g0 = 0.0f, g1 = 0.0f, g2 = 0.0f;
    int32_t last = -1;
    if (inside) {
        ra = gr.render_alphas[p];
        last = gr.last_ids[p];
        g0 = gr.grad_render_colors[3 * p];
        g1 = gr.grad_render_colors[3 * p + 1];
        g2 = gr.grad_render_colors[3 * p + 2];
        ga = gr.grad_render_alphas[p];
    }
    float Tc = 1.0f - ra;
    float Ta = 1.0f;
    float rem0 = 0.0f, rem1 = 0.0f, rem2 = 0.0f;
    if (a.backgrounds) {
        rem0 = a.backgrounds[3 * tr.c];
        rem1 = a.backgrounds[3 * tr.c + 1];
        rem2 = a.backgrounds[3 * tr.c + 2];
    }
    if (tid == 0) s_jmax = -1;
    if (gr.grad_backgrounds) {
        const float t = inside ? Tc : 0.0f;
        const float b0 = warp_sum(g0 * t), b1 = warp_sum(g1 * t), b2 = warp_sum(g2 * t);
        if (lane == 0) {
            s_bg[warp][0] = b0;
            s_bg[warp][1] = b1;
            s_bg[warp][2] = b2;
        }
    }
    __syncthreads();
    if (gr.grad_backgrounds && tid < 3) {
        float v = 0.0f;
        for (int w = 0; w < kThreads / kWarp; ++w) v += s_bg[w][tid];
        atomicAdd(&gr.grad_backgrounds[3 * tr.c + tid], v);
    }
    if (tr.masked || tr.start == tr.end) return;
    if (inside && ra > 0.0f && last >= 0) atomicMax(&s_jmax, last);
    __syncthreads();
    const int64_t walk_end = min(tr.end, (int64_t)s_jmax + 1);
    for (int64_t b1 = walk_end; b1 > tr.start; b1 -= kThreads) {
        const int64_t b0 = max(tr.start, b1 - kThreads);
        const int nb = (int)(b1 - b0);
        __syncthreads();
        if (tid < nb) s_gid[tid] = stage_record(a, b1 - 1 - tid, s_mo, s_q, s_col, tid);
        __syncthreads();
        for (int k = 0; k < nb; ++k) {
            const int64_t j = b1 - 1 - k;
            const float4 mo = s_mo[k];
            const float4 q = s_q[k];
            const PairEval e = eval_pair(mo.x, mo.y, q.x, q.y, q.z, mo.z, px, py);
            const bool valid = ra > 0.0f && e.s >= 0.0f && e.alpha >= a.alpha_cutoff &&
                               (int64_t)last >= j && Tc < 1.0f && e.alpha < 1.0f;
            if (!__any_sync(0xffffffffu, valid)) continue;
            float v_c0 = 0.f, v_c1 = 0.f, v_c2 = 0.f, v_op = 0.f, v_mx = 0.f, v_my = 0.f;
            float v_qa = 0.f, v_qb = 0.f, v_qc = 0.f, v_ax = 0.f, v_ay = 0.f;
            if (valid) {
                const float4 col = s_col[k];
                const float one_m = 1.0f - e.alpha;
                const float Tb = __fdividef(Tc, one_m);
                const float vis = Tb * e.alpha;
                v_c0 = g0 * vis;
                v_c1 = g1 * vis;
                v_c2 = g2 * vis;
                const float dot = g0 * (col.x - rem0) + g1 * (col.y - rem1) + g2 * (col.z - rem2);
                const float g_alpha = Tb * (dot + ga * Ta);
                const float g_raw = e.raw < kAlphaClamp ? g_alpha : 0.0f;
                v_op = g_raw * e.resp;
                const float g_s = -g_raw * e.raw;
                v_mx = g_s * (q.x * e.dx + q.y * e.dy);
                v_my = g_s * (q.z * e.dy + q.y * e.dx);
                v_ax = fabsf(v_mx);
                v_ay = fabsf(v_my);
                v_qa = g_s * 0.5f * e.dx * e.dx;
                v_qb = g_s * e.dx * e.dy;
                v_qc = g_s * 0.5f * e.dy * e.dy;
                rem0 = e.alpha * col.x + one_m * rem0;
                rem1 = e.alpha * col.y + one_m * rem1;
                rem2 = e.alpha * col.z + one_m * rem2;
                Ta *= one_m;
                Tc = Tb;
            }
            v_c0 = warp_sum(v_c0);
            v_c1 = warp_sum(v_c1);
            v_c2 = warp_sum(v_c2);
            v_op = warp_sum(v_op);
            v_mx = warp_sum(v_mx);
            v_my = warp_sum(v_my);
            v_qa = warp_sum(v_qa);
            v_qb = warp_sum(v_qb);
            v_qc = warp_sum(v_qc);
            if (gr.grad_means2d_abs) {
                v_ax = warp_sum(v_ax);
                v_ay = warp_sum(v_ay);
            }
            if (lane == 0 && s_gid[k] >= 0) {
                const int64_t g = s_gid[k];
                atomicAdd(&gr.grad_colors[3 * g], v_c0);
                atomicAdd(&gr.grad_colors[3 * g + 1], v_c1);
                atomicAdd(&gr.grad_colors[3 * g + 2], v_c2);
                atomicAdd(&gr.grad_opacities[g], v_op);
                atomicAdd(&gr.grad_means2d[2 * g], v_mx);
                atomicAdd(&gr.grad_means2d[2 * g + 1], v_my);
                atomicAdd(&gr.grad_conics[3 * g], v_qa);
                atomicAdd(&gr.grad_conics[3 * g + 1], v_qb);
                atomicAdd(&gr.grad_conics[3 * g + 2], v_qc);
                if (gr.grad_means2d_abs) {
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
    k_raster_bwd<<<(unsigned)tiles, kThreads, 0, s>>>(a, g);
}

}  // namespace gs
