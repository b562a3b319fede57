// Forward compositing and its reverse-walk backward, one 64-thread block per
// 16x16 tile, 4 pixels per thread in a vertical strip (thread t owns column
// t % 16 and rows 4 (t / 16) .. 4 (t / 16) + 3 of the tile).
//
// Each warp of a tile's block walks the tile's list on its own, 32 entries
// at a time, with no block barrier, so the tile's two warps never wait for
// each other:
//  * The entries are gathered through flatten_ids into a shared buffer of the
//    warp's own.  An entry whose splat cannot reach the alpha cutoff at any
//    pixel centre of the warp's 8 rows is dropped while gathering (exact
//    minimum of the quadratic form over the pixel-centre rectangle, with a
//    margin that covers the rounding of the per-pixel evaluation and of
//    exp); such an entry is skipped by every pixel of the warp anyway, so
//    results are unchanged.
//  * A staged entry serves the thread's 4 pixels, and the dx-only terms of
//    the quadratic form (a dx dx, b dx) are computed once per entry in the
//    per-pixel formula's own rounding order.
//  * alpha comes from the same inline code in both kernels, so the backward
//    makes exactly the forward's skip/composite decisions.
//
// Forward: front to back, per-pixel state in registers; a warp ends once all
// its pixels have stopped.  With a trace, the warp records for every entry it
// gathered which of its pixels composited it.
//
// Backward (gsplat 1.0.0, raster_backward.c, gs_raster_backward_pixel): back
// to front, each warp from its own pixels' largest last_id.  With the
// forward's trace only the entries the warp composited are staged; without,
// every thread re-evaluates alpha for its 4 pixels.  For each entry the
// valid (pixel, entry) pairs of the warp are packed onto consecutive lanes,
// which run the gradient recurrence for them with the per-pixel state (T, Q,
// upstream gradients) kept in shared memory.  Each lane's terms for the
// entry go to a per-warp shared buffer; every 32 / fields entries the warp
// sums the buffer column-wise (one lane per (entry, field)) and adds the
// sums to the gradients with one atomic each.
#include <cstdint>
#include <type_traits>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

// Blocks per SM each kernel is compiled to fit (register budget).
#ifndef GS_FWD_MIN_BLOCKS
#define GS_FWD_MIN_BLOCKS 14
#endif
#ifndef GS_BWD_MIN_BLOCKS
#define GS_BWD_MIN_BLOCKS 12
#endif

constexpr int kTile = 16;
constexpr int kPPT = 4;                          // pixels per thread
constexpr int kThreads = kTile * kTile / kPPT;   // 64
constexpr int kWarps = kThreads / kWarp;         // 2
constexpr int kWarpPix = kWarp * kPPT;           // pixels per warp (128)
constexpr float kAlphaClamp = 0.99f;

// ---------------------------------------------------------------- per pair

// Per-entry terms shared by the 4 pixels of one column.
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

// exp(-s) as 2^(-s log2 e): one rounded multiply and the PTX ex2.approx.ftz
// instruction (relative error below 2^-22; results below 2^-126 flush to 0,
// where alpha is far below any cutoff).  Relative to exp(-s) the error is
// at most about 2.4e-7 + |s| 1e-7.
__device__ __forceinline__ float exp_neg(float s) {
    constexpr float kMinusLog2e = -1.44269504088896341f;  // -1 / ln 2
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmul_rn(s, kMinusLog2e)));
    return y;
}

// exp(-s) for a pair of pixels: the scaling as one packed multiply (each
// component rounded as the scalar multiply), then ex2.approx per pixel.
__device__ __forceinline__ float2 exp_neg2(float2 s) {
    constexpr float kMinusLog2e = -1.44269504088896341f;  // -1 / ln 2
    const float2 t = __fmul2_rn(s, make_float2(kMinusLog2e, kMinusLog2e));
    float y0, y1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(t.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y1) : "f"(t.y));
    return make_float2(y0, y1);
}

// Packed f32x2 add as a PTX instruction with an explicit round-to-nearest
// mode.  Products from the __fmul2_rn intrinsic feeding it stay unfused, so
// each component rounds exactly as the scalar __fmul_rn / __fadd_rn sequence
// (measured bit for bit on 4 M random quadratic forms; the packed add
// intrinsic, and a PTX multiply feeding a PTX add, were fused into packed
// FMAs by the code generator and rounded differently).
__device__ __forceinline__ uint64_t pack2(float2 v) {
    return (uint64_t)__float_as_uint(v.x) | ((uint64_t)__float_as_uint(v.y) << 32);
}
__device__ __forceinline__ float2 unpack2(uint64_t r) {
    return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pack2(a)), "l"(pack2(b)));
    return unpack2(r);
}

// s = 0.5 (a dx^2 + c dy^2) + b dx dy rounded exactly as written (no FMA
// contraction), alpha = min(0.99, o exp(-s)).
__device__ __forceinline__ PairEval eval_pair(const ColumnTerms& ct, float my, float c, float op,
                                              float py) {
    PairEval e;
    e.dy = __fsub_rn(my, py);
    const float qc = __fmul_rn(__fmul_rn(c, e.dy), e.dy);
    const float qb = __fmul_rn(ct.bdx, e.dy);
    e.s = __fadd_rn(__fmul_rn(0.5f, __fadd_rn(ct.qa, qc)), qb);
    e.resp = exp_neg(e.s);
    e.raw = __fmul_rn(op, e.resp);
    e.alpha = e.raw > kAlphaClamp ? kAlphaClamp : e.raw;
    return e;
}

// Fast form of the same evaluation, for entries whose conic is safely
// positive definite (ac - b^2 > 1e-4 ac with a, c in [1e-18, 1e18] and
// |b| <= 1e18), whose mean lies within 1e6 of the origin (so no term
// overflows and no NaN arises) and whose opacity and colours are finite.
//   * s >= 0 needs no test there: s is at least 5e-5 of 0.5 (a dx^2 + c dy^2)
//     while the rounding of the exact-order form is below 5e-7 of it.
//   * With a/2 and c/2 staged, 0.5 ((a dx) dx + (c dy) dy) becomes
//     (a/2 dx) dx + (c/2 dy) dy: halving is exact and commutes with
//     rounding while no value is subnormal, which the ranges above and
//     |dx|, |dy| >= 6e-8 (or 0, for pixel centres at or beyond 0.5) ensure.
// So s, and with it alpha, is bit for bit the exact-order result, in one
// multiply less per pixel, and the compositing that follows can be
// branch-free.
struct FastColumn {
    float dx, qa2, bdx;  // dx = mx - px, qa2 = (a/2 dx) dx, bdx = b dx
};

// h = (a/2, b, c/2, -)
__device__ __forceinline__ FastColumn fast_column(float mx, const float4& h, float px) {
    FastColumn t;
    t.dx = __fsub_rn(mx, px);
    t.qa2 = __fmul_rn(__fmul_rn(h.x, t.dx), t.dx);
    t.bdx = __fmul_rn(h.y, t.dx);
    return t;
}

// Per-entry staging of the fast form; returns whether it applies.
__device__ __forceinline__ bool fast_terms(float mx, float my, float a, float b, float c,
                                           float op, float4& h) {
    h = make_float4(0.5f * a, b, 0.5f * c, 0.0f);
    const float ac = a * c;
    return fabsf(mx) <= 1e6f && fabsf(my) <= 1e6f && fabsf(op) <= 3.0e38f && a >= 1e-18f &&
           a <= 1e18f && c >= 1e-18f && c <= 1e18f && fabsf(b) <= 1e18f &&
           ac - b * b > 1e-4f * ac;
}

// ---------------------------------------------------------------- per tile

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
    if (a.bin_counts) {
        const int n = a.bin_counts[r.tile];
        if (n < 0 && threadIdx.x == 0) GS_BOUNDS_REPORT(a.d_status);
        r.start = r.tile * a.bin_capacity;
        r.end = r.start + (n < 0 ? 0 : (n > a.bin_capacity ? a.bin_capacity : n));
    } else {
        r.start = a.offsets[r.tile];
        r.end = r.tile + 1 < ntiles ? (int64_t)a.offsets[r.tile + 1] : a.n_isects;
    }
    // offsets from gs_tile_offsets are always inside [0, n_isects]; clamping
    // keeps a corrupted table from reading outside flatten_ids
    if ((r.end < 0 || r.end > a.n_isects || r.start < 0 || r.start > r.end) && threadIdx.x == 0)
        GS_BOUNDS_REPORT(a.d_status);
    r.end = r.end < 0 ? 0 : (r.end > a.n_isects ? a.n_isects : r.end);
    r.start = r.start < 0 ? 0 : (r.start > r.end ? r.end : r.start);
    r.masked = a.masks != nullptr && a.masks[r.tile] == 0;
    if (r.masked) r.end = r.start;
    return r;
}

// Pixel-centre rectangle of one warp's pixels (the tile's columns, 8 of its
// rows; clipped to the image) for the cannot-reach test.
struct TileBox {
    float xlo, xhi, ylo, yhi, log_cut;
    bool cull, empty;
};

__device__ __forceinline__ TileBox warp_box(const RasterArgs& a, const TileRange& tr, int warp) {
    constexpr int kRows = kTile / kWarps;  // rows per warp
    TileBox b;
    const int y0 = tr.ty * kTile + warp * kRows;
    b.xlo = (float)(tr.tx * kTile) + 0.5f;
    b.xhi = (float)min(tr.tx * kTile + kTile, a.width) - 0.5f;
    b.ylo = (float)y0 + 0.5f;
    b.yhi = (float)min(y0 + kRows, a.height) - 0.5f;
    b.empty = y0 >= a.height;  // the warp has no pixel inside the image
    b.cull = a.alpha_cutoff > 0.0f && isfinite(a.alpha_cutoff);
    b.log_cut = b.cull ? logf(a.alpha_cutoff) : 0.0f;
    return b;
}

// True when o exp(-s) < cutoff at every pixel centre of the box, with room
// to spare: s is at least its minimum over the (continuous) pixel-centre
// rectangle, which for a positive-definite form is 0 inside and otherwise
// the smallest of the four edge minima (a 1-D quadratic each).  The margin
// (1e-3 + 1e-5 of the form's magnitude over the rectangle) is far above the
// rounding of the per-pixel float evaluation and of exp_neg, so an entry
// dropped here fails the per-pixel alpha test at every pixel.
__device__ __forceinline__ bool cannot_reach(const TileBox& t, float mx, float my, float a,
                                             float b, float c, float op) {
    if (t.empty) return true;          // no pixel to reach
    if (!t.cull) return false;
    if (op <= 0.0f) return true;       // raw <= 0 < cutoff everywhere
    if (!(op > 0.0f)) return false;    // NaN: leave it to the per-pixel path
    if (!(a > 0.0f && c > 0.0f)) return false;
    if (!(a * c - b * b > 1e-6f * (a * c))) return false;  // not clearly positive definite
    float smin = 0.0f;
    const bool inside = mx >= t.xlo && mx <= t.xhi && my >= t.ylo && my <= t.yhi;
    if (!inside) {
        smin = INFINITY;
        const float xe[2] = {t.xlo, t.xhi};
        const float ye[2] = {t.ylo, t.yhi};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float dx = mx - xe[k];
            const float dy = fminf(fmaxf(__fdividef(-b * dx, c), my - t.yhi), my - t.ylo);
            smin = fminf(smin, 0.5f * (a * dx * dx + c * dy * dy) + b * dx * dy);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float dy = my - ye[k];
            const float dx = fminf(fmaxf(__fdividef(-b * dy, a), mx - t.xhi), mx - t.xlo);
            smin = fminf(smin, 0.5f * (a * dx * dx + c * dy * dy) + b * dx * dy);
        }
    }
    const float DX = fmaxf(fabsf(mx - t.xlo), fabsf(mx - t.xhi));
    const float DY = fmaxf(fabsf(my - t.ylo), fabsf(my - t.yhi));
    const float M = 0.5f * (a * DX * DX + c * DY * DY) + fabsf(b) * DX * DY;
    return smin > __logf(op) - t.log_cut + 1e-3f + 1e-5f * M;
}


// Trace words per list entry: one 32-bit mask per (warp, pixel slot) of the
// tile, bit = lane.  Word w = warp * kPPT + k covers the pixels of slot k of
// the threads of warp `warp`.
constexpr int kTraceWords = kWarps * kPPT;  // 8 -> 256 pixels
static_assert(kPPT == 4, "a warp's trace words of one entry are one uint4");

struct PixelSlot {
    int x, y0;  // column and first row of the thread's strip
};

__device__ __forceinline__ PixelSlot pixel_slot(const TileRange& tr) {
    PixelSlot p;
    p.x = tr.tx * kTile + (threadIdx.x & (kTile - 1));
    p.y0 = tr.ty * kTile + (threadIdx.x / kTile) * kPPT;
    return p;
}

// ------------------------------------------------------------------ forward

// Per-pixel step trace (optional forward output, read by the per-pixel
// backward): for pixel p and its s-th composited pair (front to back, s <
// max_steps) the pair's list position pos[s * npix + p] and the
// transmittance before it T[s * npix + p] (step-major, so neighbouring
// pixels' records of one step are neighbours); count[p] = the pairs the
// pixel composited, which may exceed max_steps (then the records stop at
// max_steps and the backward re-walks that pixel's list).
struct StepTrace {
    int32_t* pos;
    float* T;
    int32_t* count;
    int max_steps;
    int64_t npix;
};

// One warp's staged entries (forward).
struct FwdStage {
    float4 mo[kWarp];   // mx, my, opacity, list position (int bits)
    float4 q[kWarp];    // a, b, c
    float4 qf[kWarp];   // a/2, b, c/2, fast form (0 no, 1 yes, 2 yes without clamp)
    float4 col[kWarp];  // up to 4 channels of the launch's chunk
    uint4 tr[kWarp];    // the warp's trace words
};

// *dst = v by lane 0 only, as one predicated store (written as a branch
// around the store, the per-entry trace store made the forward 4 % slower).
__device__ __forceinline__ void st_shared_lane0(uint32_t* dst, uint4 v, int lane) {
    const uint32_t addr = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %0, 0;\n\t"
        "@p st.shared.v4.u32 [%1], {%2, %3, %4, %5};\n\t}"
        :
        : "r"(lane), "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
        : "memory");
}

// Component i (0 or 1, a compile-time constant after unrolling) of a pair.
__device__ __forceinline__ float& comp(float2& v, int i) { return i ? v.y : v.x; }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// At most 72 registers, so 14 blocks (28 warps) fit on an SM: measured
// faster than 12 blocks at 80 registers and than 16 at 64.  With the pair
// counters (a diagnostic) 80 registers, 12 blocks.
//
// A thread's 4 pixels are handled as two pairs (rows 0-1 and 2-3 of its
// strip) with the packed f32x2 operations, whose per-component rounding is
// that of the scalar operation, so results are bit for bit those of the
// scalar code.
template <int CH, bool COUNT, bool TRACE, bool STEPS = false>
__global__ void __launch_bounds__(kThreads, COUNT || STEPS ? 12 : GS_FWD_MIN_BLOCKS)
    k_raster_fwd(RasterArgs a, float* __restrict__ out_rgb, float* __restrict__ out_alpha,
                 int32_t* __restrict__ out_last, int32_t* __restrict__ out_counts,
                 uint32_t* __restrict__ trace, StepTrace stp = StepTrace{}) {
    constexpr int kPairs = kPPT / 2;
    __shared__ FwdStage fst[kWarps];
    const TileRange tr = tile_range(a);
    const PixelSlot ps = pixel_slot(tr);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float px = (float)ps.x + 0.5f;
    float2 T[kPairs], acc[kPairs][4], npy[kPairs];
    float py[kPPT];
    int32_t last[kPPT], n_eval[kPPT], n_comp[kPPT], n_last[kPPT];
    // A pixel that has stopped (outside the image, or its transmittance fell
    // below the threshold) takes no further entry: its cutoff becomes +inf,
    // so "not stopped and alpha >= cutoff" is one comparison and no flag
    // stays live across entries.  The pair counters keep an explicit flag.
    float cut[kPPT];
    bool done_c[COUNT ? kPPT : 1];
    // step trace: records written per pixel, and the pixel's index
    int32_t n_rec[STEPS ? kPPT : 1];
    int64_t pix[STEPS ? kPPT : 1];
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        last[k] = -1;
        n_eval[k] = n_comp[k] = n_last[k] = 0;
        const bool outside = !(ps.x < a.width && ps.y0 + k < a.height);
        cut[k] = outside ? INFINITY : a.alpha_cutoff;
        if (STEPS) {
            n_rec[k] = 0;
            pix[k] = ((int64_t)tr.c * a.height + ps.y0 + k) * a.width + ps.x;
        }
        if (COUNT) done_c[k] = outside;
        py[k] = (float)(ps.y0 + k) + 0.5f;
    }
    auto record = [&](int k, int32_t j, float t_before) {
        if (STEPS) {
            if (n_rec[k] < stp.max_steps) {
                const int64_t o = (int64_t)n_rec[k] * stp.npix + pix[k];
                stp.pos[o] = j;
                stp.T[o] = t_before;
            }
            ++n_rec[k];
        }
    };
    auto stopped = [&](int k) { return COUNT ? done_c[k] : cut[k] == INFINITY; };
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
        T[p] = splat2(1.0f);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[p][c] = splat2(0.0f);
        npy[p] = make_float2(-py[2 * p], -py[2 * p + 1]);
    }
    const float2 one = splat2(1.0f), minus_one = splat2(-1.0f);
    // Each warp walks the tile's list on its own, 32 entries at a time: lane
    // l gathers entry b0 + l and tests it against the warp's own pixel box;
    // the entries that can reach one of the warp's pixels are staged, in
    // order, in the warp's own buffer.  No block barrier: a warp whose
    // pixels have all stopped ends without waiting for the other.
    FwdStage& sw = fst[warp];
    const TileBox wb = warp_box(a, tr, warp);
    const int64_t CN = (int64_t)a.C * a.N;
    const unsigned lt = lanemask_lt();
    for (int64_t b0 = tr.start; b0 < tr.end; b0 += kWarp) {
        bool all_done = true;
#pragma unroll
        for (int k = 0; k < kPPT; ++k) all_done &= stopped(k);
        if (__all_sync(0xffffffffu, all_done)) break;
        const int n_raw = (int)min((int64_t)kWarp, tr.end - b0);
        const int32_t b0_32 = (int32_t)b0;  // list positions are below 2^31
        const int64_t jl = b0 + lane;
        bool reach = false;
        float2 m = make_float2(0.0f, 0.0f);
        float op = 0.0f, qa = 0.0f, qb = 0.0f, qc = 0.0f;
        int64_t g = 0;
        if (lane < n_raw) {
            g = a.flatten_ids[jl];
            if ((uint64_t)g < (uint64_t)CN) {
                m = reinterpret_cast<const float2*>(a.means2d)[g];
                const float* qq = a.conics + 3 * g;
                qa = qq[0];
                qb = qq[1];
                qc = qq[2];
                op = a.opacities[g];
                reach = !cannot_reach(wb, m.x, m.y, qa, qb, qc, op);
            } else {
                GS_BOUNDS_REPORT(a.d_status);
            }
        }
        const unsigned ball = __ballot_sync(0xffffffffu, reach);
        __syncwarp();  // the previous chunk's reads of the buffer are done
        if (TRACE) sw.tr[lane] = make_uint4(0u, 0u, 0u, 0u);
        if (reach) {
            const int pos = __popc(ball & lt);
            const float* cc = a.colors + g * a.channels + a.ch_off;
            const float4 col = make_float4(cc[0], CH > 1 ? cc[1] : 0.0f, CH > 2 ? cc[2] : 0.0f,
                                           CH > 3 ? cc[3] : 0.0f);
            float4 f;
            bool fast = fast_terms(m.x, m.y, qa, qb, qc, op, f);
            fast = fast && fabsf(col.x) < 3.0e38f && fabsf(col.y) < 3.0e38f &&
                   fabsf(col.z) < 3.0e38f && fabsf(col.w) < 3.0e38f;
            // 2: fast form, and o <= 0.98 so o exp(-s) (s >= 0) never reaches
            // the 0.99 clamp, whatever the exponential's 2^-22 rounding
            f.w = fast ? (op <= 0.98f ? 2.0f : 1.0f) : 0.0f;
            sw.mo[pos] = make_float4(m.x, m.y, op, __int_as_float((int32_t)jl));
            sw.q[pos] = make_float4(qa, qb, qc, 0.0f);
            sw.qf[pos] = f;
            sw.col[pos] = col;
        }
        __syncwarp();
        {
            const int nw = __popc(ball);
            for (int i = 0; i < nw; ++i) {
                const float4 mo = sw.mo[i];
                const int32_t j = __float_as_int(mo.w);
                const float4 h = sw.qf[i];  // a/2, b, c/2, fast-form flag
                const float4 col = sw.col[i];
                const float colv[4] = {col.x, col.y, col.z, col.w};
                bool took[kPPT];
                // fast form (warp-uniform): branch-free compositing
                auto fast_pairs = [&](auto clamp_tag) {
                    constexpr bool kClamp = decltype(clamp_tag)::value;
                    const FastColumn fc = fast_column(mo.x, h, px);
                    const float2 qa2 = splat2(fc.qa2), bdx = splat2(fc.bdx), c2 = splat2(h.z);
                    const float2 my = splat2(mo.y), op = splat2(mo.z);
#pragma unroll
                    for (int p = 0; p < kPairs; ++p) {
                        // s = ((a/2 dx) dx + (c/2 dy) dy) + (b dx) dy, per pixel, as
                        // packed operations that round each component as the scalar
                        // ones (intrinsic products, PTX sums: never fused)
                        const float2 dy = add2_rn(my, npy[p]);
                        const float2 qc2 = __fmul2_rn(__fmul2_rn(c2, dy), dy);
                        const float2 qb = __fmul2_rn(bdx, dy);
                        const float2 sv = add2_rn(add2_rn(qa2, qc2), qb);
                        const float2 raw = __fmul2_rn(op, exp_neg2(sv));
                        float2 aw;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int k = 2 * p + e;
                            const float r_e = comp(const_cast<float2&>(raw), e);
                            const float alpha = kClamp ? fminf(r_e, kAlphaClamp) : r_e;
                            took[k] = alpha >= cut[k];
                            if (COUNT) n_eval[k] += done_c[k] ? 0 : 1;
                            // a pair not taken adds exactly 0 (finite colours, T)
                            comp(aw, e) = took[k] ? alpha : 0.0f;
                        }
                        if (STEPS) {
#pragma unroll
                            for (int e = 0; e < 2; ++e)
                                if (took[2 * p + e]) record(2 * p + e, j, comp(T[p], e));
                        }
                        const float2 w = __fmul2_rn(T[p], aw);
#pragma unroll
                        for (int c = 0; c < CH; ++c)
                            acc[p][c] = __ffma2_rn(w, splat2(colv[c]), acc[p][c]);
                        T[p] = __fmul2_rn(T[p], __ffma2_rn(aw, minus_one, one));
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int k = 2 * p + e;
                            last[k] = took[k] ? j : last[k];
                            if (COUNT && took[k]) {
                                ++n_comp[k];
                                n_last[k] = n_eval[k];
                            }
                            const bool stop =
                                took[k] && comp(T[p], e) < a.transmittance_threshold;
                            cut[k] = stop ? INFINITY : cut[k];
                            if (COUNT) done_c[k] = done_c[k] || stop;
                        }
                    }
                };
                if (h.w > 1.5f) {
                    fast_pairs(std::integral_constant<bool, false>{});
                } else if (h.w != 0.0f) {
                    fast_pairs(std::integral_constant<bool, true>{});
                } else {  // exact-order form, with the s >= 0 test
                    const float4 q = sw.q[i];
                    const ColumnTerms ct = column_terms(mo.x, q.x, q.y, px);
                    float alpha[kPPT];
#pragma unroll
                    for (int k = 0; k < kPPT; ++k) {
                        const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, py[k]);
                        alpha[k] = e.alpha;
                        took[k] = e.s >= 0.0f && e.alpha >= cut[k];
                        if (COUNT) n_eval[k] += done_c[k] ? 0 : 1;
                    }
#pragma unroll
                    for (int k = 0; k < kPPT; ++k) {
                        if (!took[k]) continue;
                        float& Tk = comp(T[k >> 1], k & 1);
                        record(k, j, Tk);
                        const float w = Tk * alpha[k];
#pragma unroll
                        for (int c = 0; c < CH; ++c) {
                            float& ak = comp(acc[k >> 1][c], k & 1);
                            ak = __fmaf_rn(w, colv[c], ak);
                        }
                        Tk = Tk * (1.0f - alpha[k]);
                        last[k] = j;
                        if (COUNT) {
                            ++n_comp[k];
                            n_last[k] = n_eval[k];
                        }
                        if (Tk < a.transmittance_threshold) {
                            cut[k] = INFINITY;
                            if (COUNT) done_c[k] = true;
                        }
                    }
                }
                if (TRACE) {
                    // the warp's 4 slot masks, one 16-byte store
                    const uint4 m4 = make_uint4(__ballot_sync(0xffffffffu, took[0]),
                                                __ballot_sync(0xffffffffu, took[1]),
                                                __ballot_sync(0xffffffffu, took[2]),
                                                __ballot_sync(0xffffffffu, took[3]));
                    st_shared_lane0(&sw.tr[j - b0_32].x, m4, lane);
                }
                // leave the chunk early once every pixel of the warp has stopped
                if ((i & 15) == 15) {
                    bool d = true;
#pragma unroll
                    for (int k = 0; k < kPPT; ++k) d &= stopped(k);
                    if (__all_sync(0xffffffffu, d)) break;
                }
            }
        }
        if (TRACE) {
            __syncwarp();
            if (lane < n_raw)
                reinterpret_cast<uint4*>(trace + jl * kTraceWords)[warp] = sw.tr[lane];
        }
    }
    float bg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (a.backgrounds)
#pragma unroll
        for (int c = 0; c < CH; ++c)
            bg[c] = a.backgrounds[(int64_t)tr.c * a.channels + a.ch_off + c];
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        const int y = ps.y0 + k;
        if (ps.x < a.width && y < a.height) {
            const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + ps.x;
            const float Tk = comp(T[k >> 1], k & 1);
            float* o = out_rgb + p * a.channels + a.ch_off;
#pragma unroll
            for (int c = 0; c < CH; ++c) o[c] = comp(acc[k >> 1][c], k & 1) + Tk * bg[c];
            if (!a.first_chunk) continue;
            out_alpha[p] = 1.0f - Tk;
            out_last[p] = last[k];
            if (STEPS) stp.count[p] = n_rec[k];
            if (COUNT) {
                out_counts[3 * p] = n_eval[k];
                out_counts[3 * p + 1] = n_comp[k];
                out_counts[3 * p + 2] = n_last[k];
            }
        }
    }
}

// ----------------------------------------------------------------- backward

// Per-pixel state of one warp's 128 pixels, pixel (slot k, lane l) at index
// k * 32 + l: (T, Q) as one float2 and the upstream colour gradient g[CH]
// as one float4, so a packed pair reads its pixel's state with two loads
// and writes it back with one.  The packed pairs of a round are in
// ascending pixel order, so neighbouring lanes mostly read neighbouring
// entries.
//
// The walk's remainder rem[CH] and running product T_after enter the alpha
// gradient only as  sum_c g_c (color_c - rem_c) + g_a T_after
//   = g . color - Q,   with  Q = g . rem - g_a T_after.
// Both rem_c and T_after follow  x <- alpha y + (1 - alpha) x  (with y =
// color_c and y = 0), so Q follows  Q <- alpha (g . color) + (1 - alpha) Q
// from  Q = g . background - g_a.  One scalar replaces CH + 1 of them.

// Gradient fields in the reduction buffer: colours[CH], then these.
template <int CH>
struct GradLayout {
    static constexpr int kOp = CH, kMx = CH + 1, kMy = CH + 2, kQa = CH + 3, kQb = CH + 4,
                         kQc = CH + 5, kAx = CH + 6, kAy = CH + 7;
};

template <int CH, int F>
struct BwdWarpSmem {
    float2 tq[kWarpPix];  // (T, Q) of pixel k * 32 + lane
    float4 g4[kWarpPix];  // upstream colour gradient g[CH]; with CH < 4 .w = pixel centre y
    int16_t list[kWarpPix];  // packed valid pairs: k * 32 + owner lane
    // entries buffered per reduction: one (entry, field) sum per lane
    static constexpr int kRed = kWarp / F;
    // per (entry, field): the 32 lanes' terms (lanes without a pair hold 0),
    // then 16 bytes of padding, so that row r starts in bank group r mod 8
    // and the 8 lanes of a quarter warp, summing rows r .. r + 7, read chunk
    // i of each without a bank conflict
    float4 red[kRed][F][kWarp / 4 + 1];
    int32_t red_gid[kRed];
};

// One warp's staged entries (trace-driven backward).
struct BwdStage {
    float4 mo[kWarp];   // mx, my, opacity, list position (int bits)
    float4 q[kWarp];    // a, b, c, flatten id (int bits)
    float4 col[kWarp];  // up to 4 channels of the launch's chunk
    uint4 tr[kWarp];    // the warp's trace words
};

// One warp's walk of its tile's list from position wend - 1 down to the
// tile's start, 32 entries at a time (lane l takes entry b1 - 1 - l).  An
// entry is staged -- in walk order, in the warp's own buffer -- when the
// warp has work with it: with the forward's trace, when the warp's trace
// words of it are not all zero; without, when its splat can reach one of
// the warp's pixels.  The flatten id (and the trace words) of a chunk's
// entry are read one chunk ahead, while the warp works through the current
// chunk.  entry(mo, q, col, m4) then runs on the whole warp for each staged
// entry in order: mo = (mx, my, opacity, list position), q = (a, b, c,
// flatten id), col = the chunk's up to 4 colour channels (none when CH is
// 0), m4 = the warp's trace words.  A flatten id outside [0, C*N) (only from
// corrupted input) is reported and the entry dropped.
template <int CH, bool TRACE, typename Entry>
__device__ __forceinline__ void walk_back(const RasterArgs& a, const TileRange& tr,
                                          const TileBox& wb, const uint32_t* __restrict__ trace,
                                          int64_t wend, BwdStage& sw, Entry&& entry) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt();
    const int64_t CN = (int64_t)a.C * a.N;
    auto fetch = [&](int64_t b1, uint4& m4, int64_t& g) {
        const int64_t j = b1 - 1 - lane;
        m4 = make_uint4(0u, 0u, 0u, 0u);
        g = -1;
        if (j >= tr.start) {
            bool want = true;
            if (TRACE) {
                m4 = reinterpret_cast<const uint4*>(trace + j * kTraceWords)[warp];
                want = (m4.x | m4.y | m4.z | m4.w) != 0u;
            }
            if (want) {
                g = a.flatten_ids[j];
                if ((uint64_t)g >= (uint64_t)CN) {
                    GS_BOUNDS_REPORT(a.d_status);
                    g = -1;
                }
            }
        }
    };
    uint4 m4n;
    int64_t gn;
    fetch(wend, m4n, gn);
    for (int64_t b1 = wend; b1 > tr.start; b1 -= kWarp) {
        const int64_t j = b1 - 1 - lane;
        const uint4 m4 = m4n;
        const int64_t g = gn;
        bool take = g >= 0;
        float4 mo = make_float4(0.0f, 0.0f, 0.0f, 0.0f), q = mo;
        if (take) {
            const float2 m = reinterpret_cast<const float2*>(a.means2d)[g];
            const float* qq = a.conics + 3 * g;
            mo = make_float4(m.x, m.y, a.opacities[g], __int_as_float((int32_t)j));
            q = make_float4(qq[0], qq[1], qq[2], __int_as_float((int32_t)g));
            if (!TRACE) take = !cannot_reach(wb, mo.x, mo.y, q.x, q.y, q.z, mo.z);
        }
        const unsigned ball = __ballot_sync(0xffffffffu, take);
        if (ball == 0u) {
            fetch(b1 - kWarp, m4n, gn);
            continue;
        }
        __syncwarp();  // the previous chunk's reads of the buffer are done
        if (take) {
            const int pos = __popc(ball & lt);
            float4 col = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (CH > 0) {
                const float* cc = a.colors + g * a.channels + a.ch_off;
                col = make_float4(cc[0], CH > 1 ? cc[1] : 0.0f, CH > 2 ? cc[2] : 0.0f,
                                  CH > 3 ? cc[3] : 0.0f);
            }
            sw.mo[pos] = mo;
            sw.q[pos] = q;
            sw.col[pos] = col;
            sw.tr[pos] = m4;
        }
        fetch(b1 - kWarp, m4n, gn);
        __syncwarp();
        const int n = __popc(ball);
        for (int i = 0; i < n; ++i) entry(sw.mo[i], sw.q[i], sw.col[i], sw.tr[i]);
    }
}

// A lane's share of every flush: field f of buffered entry e, where
// (e, f) = (lane / F, lane mod F) never changes, so the gradient array, its
// stride per splat and the shared-memory row are worked out once per thread.
struct FlushTask {
    float* base;     // gradient array + field offset
    uint32_t row;    // shared-memory address of red[e][f][0]
    int e;           // buffered entry (kRed or more: no task)
    int stride;      // floats per splat in that array
};

template <int CH, int F>
__device__ __forceinline__ FlushTask flush_task(BwdWarpSmem<CH, F>& w, const RasterArgs& a,
                                                const RasterGrads& gr, int lane) {
    using G = GradLayout<CH>;
    FlushTask t;
    t.e = lane / F;
    const int f = lane - t.e * F;
    const int e = t.e < BwdWarpSmem<CH, F>::kRed ? t.e : 0;
    t.row = (uint32_t)__cvta_generic_to_shared(&w.red[e][f][0]);
    if (f < CH) {
        t.base = gr.grad_colors + a.ch_off + f;
        t.stride = a.channels;
    } else if (f == G::kOp) {
        t.base = gr.grad_opacities;
        t.stride = 1;
    } else if (f <= G::kMy) {
        t.base = gr.grad_means2d + (f - G::kMx);
        t.stride = 2;
    } else if (f <= G::kQc) {
        t.base = gr.grad_conics + (f - G::kQa);
        t.stride = 3;
    } else {
        t.base = gr.grad_means2d_abs + (f - G::kAx);
        t.stride = 2;
    }
    return t;
}

__device__ __forceinline__ float4 lds128(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Sums each buffered (entry, field) over the warp's 32 lanes (a lane without
// a pair wrote 0) and adds it to the splat's gradient with one atomic: lane
// t owns task t.
template <int CH, int F>
__device__ __forceinline__ void flush_reduction(BwdWarpSmem<CH, F>& w, int nslots,
                                                const FlushTask& task, int lane) {
    static_assert(BwdWarpSmem<CH, F>::kRed >= 1, "one reduction task per lane");
    __syncwarp();
    if (task.e < nslots) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < kWarp / 4; ++c) {
            const float4 q = lds128(task.row + 16u * (uint32_t)c);
            acc = __fadd2_rn(acc, make_float2(q.x, q.y));
            acc = __fadd2_rn(acc, make_float2(q.z, q.w));
        }
        const float sum = acc.x + acc.y;
        if (sum != 0.0f)
            atomicAdd(task.base + (int64_t)w.red_gid[task.e] * task.stride, sum);
    }
    __syncwarp();
}

// For each entry the warp's valid (pixel, entry) pairs -- from the forward's
// trace masks with TRACE, else by re-evaluating alpha -- are packed onto
// consecutive lanes, which run the gradient recurrence with the per-pixel
// state in shared memory.  Each packed pair is re-evaluated with the
// forward's arithmetic and re-tested in full before its gradient is taken,
// so both paths give the same result.
template <int CH, bool ABS, bool TRACE>
__global__ void __launch_bounds__(kThreads, GS_BWD_MIN_BLOCKS)
    k_raster_bwd(RasterArgs a, RasterGrads gr, const uint32_t* __restrict__ trace) {
    using G = GradLayout<CH>;
    constexpr int F = CH + (ABS ? 8 : 6);
    __shared__ BwdStage wst[kWarps];
    __shared__ BwdWarpSmem<CH, F> ws[kWarps];
    __shared__ float s_bg[kWarps][4];
    const TileRange tr = tile_range(a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    BwdWarpSmem<CH, F>& w = ws[warp];
    const PixelSlot ps = pixel_slot(tr);
    const float px = (float)ps.x + 0.5f;

    float ra[kPPT], py[kPPT];
    int32_t last[kPPT];
    float bgv[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c)
        bgv[c] = a.backgrounds ? a.backgrounds[(int64_t)tr.c * a.channels + a.ch_off + c] : 0.0f;
    int my_max = -1;
    float sb[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) sb[c] = 0.0f;
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        const int y = ps.y0 + k;
        py[k] = (float)y + 0.5f;
        ra[k] = 0.0f;
        last[k] = -1;
        float gc[CH], ga = 0.0f;
#pragma unroll
        for (int c = 0; c < CH; ++c) gc[c] = 0.0f;
        if (ps.x < a.width && y < a.height) {
            const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + ps.x;
            ra[k] = gr.render_alphas[p];
            last[k] = gr.last_ids[p];
#pragma unroll
            for (int c = 0; c < CH; ++c) gc[c] = gr.grad_render_colors[p * a.channels + a.ch_off + c];
            // the render_alpha gradient's terms are added by the first chunk only
            ga = a.first_chunk ? gr.grad_render_alphas[p] : 0.0f;
        }
        const float Tc = 1.0f - ra[k];
        float Q = -ga;
        float gq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            Q += gc[c] * bgv[c];
            gq[c] = gc[c];
            sb[c] += gc[c] * Tc;
        }
        // with fewer than 4 channels the spare lane holds the pixel centre's y
        w.g4[k * kWarp + lane] = make_float4(gq[0], gq[1], gq[2], CH < 4 ? py[k] : gq[3]);
        w.tq[k * kWarp + lane] = make_float2(Tc, Q);
        if (ra[k] > 0.0f && last[k] > my_max) my_max = last[k];
    }
    if (gr.grad_backgrounds) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sb[c] += __shfl_xor_sync(0xffffffffu, sb[c], o);
            if (lane == 0) s_bg[warp][c] = sb[c];
        }
    }
    __syncthreads();
    if (gr.grad_backgrounds && tid < CH) {
        float v = 0.0f;
        for (int k = 0; k < kWarps; ++k) v += s_bg[k][tid];
        atomicAdd(&gr.grad_backgrounds[(int64_t)tr.c * a.channels + a.ch_off + tid], v);
    }
    if (tr.masked || tr.start == tr.end) return;
    const int warp_max = __reduce_max_sync(0xffffffffu, my_max);
    const unsigned lt = lanemask_lt();
    const int x_tile = tr.tx * kTile;
    const int y_tile = tr.ty * kTile;
    const FlushTask task = flush_task<CH, F>(w, a, gr, lane);
    int nslots = 0;
    // steps 1-3 for one staged entry (m4: the warp's trace words of it)
    auto entry = [&](const float4 mo, const float4 q, const float4 col, const uint4 m4) {
        const int32_t j = __float_as_int(mo.w);
        // 1. which pixels of the warp have a valid pair with this entry
        //    (the sync orders the previous entry's list reads first)
        __syncwarp();
        int count = 0;
        if (TRACE) {
            const unsigned m[kPPT] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int k = 0; k < kPPT; ++k) {
                if ((m[k] >> lane) & 1u)
                    w.list[count + __popc(m[k] & lt)] = (int16_t)(k * kWarp + lane);
                count += __popc(m[k]);
            }
        } else {
            const ColumnTerms ct = column_terms(mo.x, q.x, q.y, px);
#pragma unroll
            for (int k = 0; k < kPPT; ++k) {
                const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, py[k]);
                // T < 1 depends on pairs still being run; the lane that
                // runs this pair tests it
                const bool valid = ra[k] > 0.0f && e.s >= 0.0f &&
                                   e.alpha >= a.alpha_cutoff && last[k] >= j;
                const unsigned m = __ballot_sync(0xffffffffu, valid);
                if (valid) w.list[count + __popc(m & lt)] = (int16_t)(k * kWarp + lane);
                count += __popc(m);
            }
        }
        if (count == 0) return;  // warp-uniform
        __syncwarp();
        // 2. the packed pairs, one per lane
        float v[F];
#pragma unroll
        for (int f = 0; f < F; ++f) v[f] = 0.0f;
        for (int L = lane; L < count; L += kWarp) {
            const int p = w.list[L];
            const int ol = p & 31;
            const float4 g4 = w.g4[p];
            const float pyv = CH < 4 ? g4.w
                                     : (float)(y_tile + ((warp * kWarp + ol) / kTile) * kPPT +
                                               (p >> 5)) + 0.5f;
            const ColumnTerms ct =
                column_terms(mo.x, q.x, q.y, (float)(x_tile + (ol & (kTile - 1))) + 0.5f);
            const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, pyv);
            const float dx = ct.dx;
            const float2 tq = w.tq[p];
            const float Tc = tq.x, Q = tq.y;
            // the packed pairs satisfy render_alpha > 0, s >= 0, alpha >=
            // cutoff and last_id >= j (from the trace, or tested while
            // packing), so alpha is finite and, clamped, below 1; the
            // T < 1 guard depends on the walk and is tested here.  A pair
            // failing it adds nothing and leaves the pixel's state as it
            // was: it runs with alpha 0 and no alpha gradient (no branch
            // around the pair's work)
            const bool ok = Tc < 1.0f;
            const float al = ok ? e.alpha : 0.0f;
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
            const float colv[4] = {col.x, col.y, col.z, col.w};
            const float one_m = 1.0f - al;
            const float Tb = __fdividef(Tc, one_m);
            const float vis = Tb * al;
            float gcol = 0.0f;  // g . color
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const float gcc = gv[c];
                v[c] += gcc * vis;
                gcol += gcc * colv[c];
            }
            const float g_alpha = Tb * (gcol - Q);
            const float g_raw = ok && e.raw < kAlphaClamp ? g_alpha : 0.0f;
            v[G::kOp] += g_raw * e.resp;
            const float g_s = -g_raw * e.raw;
            const float gmx = g_s * (q.x * dx + q.y * e.dy);
            const float gmy = g_s * (q.z * e.dy + q.y * dx);
            v[G::kMx] += gmx;
            v[G::kMy] += gmy;
            v[G::kQa] += g_s * (0.5f * dx * dx);
            v[G::kQb] += g_s * (dx * e.dy);
            v[G::kQc] += g_s * (0.5f * e.dy * e.dy);
            if (ABS) {
                v[G::kAx] += fabsf(gmx);
                v[G::kAy] += fabsf(gmy);
            }
            w.tq[p] = make_float2(Tb, al * gcol + one_m * Q);
        }
        // 3. this entry's terms into the warp's reduction buffer
#pragma unroll
        for (int f = 0; f < F; ++f) reinterpret_cast<float*>(w.red[nslots][f])[lane] = v[f];
        if (lane == 0) w.red_gid[nslots] = __float_as_int(q.w);
        if (++nslots == BwdWarpSmem<CH, F>::kRed) {
            flush_reduction<CH, F>(w, nslots, task, lane);
            nslots = 0;
        }
    };
    // each warp walks the list on its own, from its own pixels' largest last id
    walk_back<CH, TRACE>(a, tr, warp_box(a, tr, warp), trace,
                         min(tr.end, (int64_t)warp_max + 1), wst[warp], entry);
    if (nslots) flush_reduction<CH, F>(w, nslots, task, lane);
}

// ------------------------------------------------- absgrad over many channels

// With more than 4 channels the chunked backward cannot form absgrad: a
// pair's mean-gradient term carries the alpha gradient summed over ALL
// channels, and |.| of that sum is not the sum of |.| of per-chunk parts.
// This pass walks the lists once more, exactly as the chunks do (trace-driven
// or re-evaluating), with the full channel sums -- the pixel's upstream
// colour gradient and the splat's colour are read from global memory for
// each pair -- and adds only |dL/dmeans2d| to grad_means2d_abs.  Per pixel
// the state is (T, Q), Q = sum_c g_c rem_c - g_a T_after, with the chunks'
// recurrence Q <- alpha (g . color) + (1 - alpha) Q from g . background - g_a.
struct AbsWarpSmem {
    static constexpr int kRed = 16;  // entries buffered per reduction (2 fields)
    float2 tq[kWarpPix];
    int16_t list[kWarpPix];
    float4 red[kRed][2][kWarp / 4 + 1];  // rows padded as in BwdWarpSmem
    int32_t red_gid[kRed];
};

template <bool TRACE>
__global__ void __launch_bounds__(kThreads, GS_BWD_MIN_BLOCKS)
    k_raster_bwd_absgrad(RasterArgs a, RasterGrads gr, const uint32_t* __restrict__ trace) {
    constexpr int kRed = AbsWarpSmem::kRed;
    __shared__ BwdStage wst[kWarps];
    __shared__ AbsWarpSmem ws[kWarps];
    const TileRange tr = tile_range(a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    AbsWarpSmem& w = ws[warp];
    const PixelSlot ps = pixel_slot(tr);
    const float px = (float)ps.x + 0.5f;
    const int nch = a.channels;
    int32_t last[kPPT];
    float ra[kPPT], py[kPPT];
    int my_max = -1;
#pragma unroll
    for (int k = 0; k < kPPT; ++k) {
        const int y = ps.y0 + k;
        py[k] = (float)y + 0.5f;
        ra[k] = 0.0f;
        last[k] = -1;
        float Q = 0.0f;
        if (ps.x < a.width && y < a.height) {
            const int64_t p = ((int64_t)tr.c * a.height + y) * a.width + ps.x;
            ra[k] = gr.render_alphas[p];
            last[k] = gr.last_ids[p];
            Q = -gr.grad_render_alphas[p];
            if (a.backgrounds)
                for (int c = 0; c < nch; ++c)
                    Q += gr.grad_render_colors[p * nch + c] * a.backgrounds[(int64_t)tr.c * nch + c];
        }
        w.tq[k * kWarp + lane] = make_float2(1.0f - ra[k], Q);
        if (ra[k] > 0.0f && last[k] > my_max) my_max = last[k];
    }
    __syncwarp();
    if (tr.masked || tr.start == tr.end) return;  // block-uniform
    const int warp_max = __reduce_max_sync(0xffffffffu, my_max);
    const unsigned lt = lanemask_lt();
    const int x_tile = tr.tx * kTile;
    const int y_tile = tr.ty * kTile;
    // flush task of this lane: field (lane & 1) of buffered entry lane / 2
    const int task_e = lane >> 1;
    const uint32_t task_row = (uint32_t)__cvta_generic_to_shared(&w.red[task_e][lane & 1][0]);
    float* const task_base = gr.grad_means2d_abs + (lane & 1);
    auto flush = [&](int nslots) {
        __syncwarp();
        if (task_e < nslots) {
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int c = 0; c < kWarp / 4; ++c) {
                const float4 q = lds128(task_row + 16u * (uint32_t)c);
                acc = __fadd2_rn(acc, make_float2(q.x, q.y));
                acc = __fadd2_rn(acc, make_float2(q.z, q.w));
            }
            const float sum = acc.x + acc.y;
            if (sum != 0.0f) atomicAdd(task_base + (int64_t)w.red_gid[task_e] * 2, sum);
        }
        __syncwarp();
    };
    int nslots = 0;
    auto entry = [&](const float4 mo, const float4 q, const float4, const uint4 m4) {
        const int32_t j = __float_as_int(mo.w);
        const int32_t gid = __float_as_int(q.w);
        __syncwarp();
        int count = 0;
        if (TRACE) {
            const unsigned m[kPPT] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int k = 0; k < kPPT; ++k) {
                if ((m[k] >> lane) & 1u)
                    w.list[count + __popc(m[k] & lt)] = (int16_t)(k * kWarp + lane);
                count += __popc(m[k]);
            }
        } else {
            const ColumnTerms ct = column_terms(mo.x, q.x, q.y, px);
#pragma unroll
            for (int k = 0; k < kPPT; ++k) {
                const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, py[k]);
                const bool valid = ra[k] > 0.0f && e.s >= 0.0f &&
                                   e.alpha >= a.alpha_cutoff && last[k] >= j;
                const unsigned mk = __ballot_sync(0xffffffffu, valid);
                if (valid) w.list[count + __popc(mk & lt)] = (int16_t)(k * kWarp + lane);
                count += __popc(mk);
            }
        }
        if (count == 0) return;  // warp-uniform
        __syncwarp();
        float va = 0.0f, vb = 0.0f;
        const float* const col = a.colors + (int64_t)gid * nch;
        for (int L = lane; L < count; L += kWarp) {
            const int p = w.list[L];
            const int ol = p & 31;
            const int xx = x_tile + (ol & (kTile - 1));
            const int yy = y_tile + ((warp * kWarp + ol) / kTile) * kPPT + (p >> 5);
            const ColumnTerms ct = column_terms(mo.x, q.x, q.y, (float)xx + 0.5f);
            const PairEval e = eval_pair(ct, mo.y, q.z, mo.z, (float)yy + 0.5f);
            const float2 tq = w.tq[p];
            const float Tc = tq.x, Q = tq.y;
            const bool ok = Tc < 1.0f;  // as in the chunks' pair loop
            const float al = ok ? e.alpha : 0.0f;
            const float one_m = 1.0f - al;
            const float Tb = __fdividef(Tc, one_m);
            const float* gp =
                gr.grad_render_colors + (((int64_t)tr.c * a.height + yy) * a.width + xx) * nch;
            float gcol = 0.0f;  // g . color over every channel
            for (int c = 0; c < nch; ++c) gcol += gp[c] * col[c];
            const float g_alpha = Tb * (gcol - Q);
            const float g_raw = ok && e.raw < kAlphaClamp ? g_alpha : 0.0f;
            const float g_s = -g_raw * e.raw;
            va += fabsf(g_s * (q.x * ct.dx + q.y * e.dy));
            vb += fabsf(g_s * (q.z * e.dy + q.y * ct.dx));
            w.tq[p] = make_float2(Tb, al * gcol + one_m * Q);
        }
        reinterpret_cast<float*>(w.red[nslots][0])[lane] = va;
        reinterpret_cast<float*>(w.red[nslots][1])[lane] = vb;
        if (lane == 0) w.red_gid[nslots] = gid;
        if (++nslots == kRed) {
            flush(nslots);
            nslots = 0;
        }
    };
    walk_back<0, TRACE>(a, tr, warp_box(a, tr, warp), trace, min(tr.end, (int64_t)warp_max + 1),
                        wst[warp], entry);
    if (nslots) flush(nslots);
}

// ------------------------------------------------ per-pixel step-trace backward

// The backward over the forward's per-pixel step trace (the trace buffers of
// rlx-metal's traced training step, splat_training.rs): each pixel walks its
// recorded pairs from its last to its first -- no other list entry is
// visited and the transmittance before each pair is read, not recovered by
// division.  A pixel that composited more pairs than were recorded walks its
// tile's list from its last id down instead, with the recovery T_before =
// T / (1 - alpha) (gsplat 1.0.0, raster_backward.c,
// gs_raster_backward_pixel).  Every channel is handled in one pass (colours
// and upstream gradients read from global memory per pair).
//
// One thread per pixel, and the 32 pixels of a warp (two rows of the tile)
// move through their tile's list together: each round takes the largest
// list position any lane still has to visit (its next record, or its next
// entry in the fallback walk), so the lanes at that position all hold the
// same splat; they run their pair, and the warp sums each gradient term over
// its lanes before one atomic per field (a lone lane adds its own terms).
constexpr int kStepThreads = kTile * kTile;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <bool ABS>
__global__ void __launch_bounds__(kStepThreads)
    k_raster_bwd_steps(RasterArgs a, RasterGrads gr, StepTrace stp) {
    const TileRange tr = tile_range(a);
    const int lx = threadIdx.x & (kTile - 1), ly = threadIdx.x / kTile;
    const int lane = threadIdx.x & 31;
    const int x = tr.tx * kTile + lx, y = tr.ty * kTile + ly;
    const bool inside = x < a.width && y < a.height;
    const int nch = a.channels;
    const int64_t p = inside ? ((int64_t)tr.c * a.height + y) * a.width + x : 0;
    const float ra = inside ? gr.render_alphas[p] : 0.0f;
    const float Tfinal = 1.0f - ra;
    const float* bg = a.backgrounds ? a.backgrounds + (int64_t)tr.c * nch : nullptr;
    const float* gp = gr.grad_render_colors + p * nch;
    // dL/dbackground: sum over pixels of g (1 - render_alpha), per channel
    if (gr.grad_backgrounds) {
        for (int c = 0; c < nch; ++c) {
            const float v = warp_sum(inside ? gp[c] * Tfinal : 0.0f);
            if (lane == 0 && v != 0.0f) atomicAdd(&gr.grad_backgrounds[(int64_t)tr.c * nch + c], v);
        }
    }
    const bool live = inside && !tr.masked && ra > 0.0f;
    const float px = (float)x + 0.5f, py = (float)y + 0.5f;
    const int64_t CN = (int64_t)a.C * a.N;
    // Q = g . rem - g_a T_after, from g . background - g_a (see k_raster_bwd)
    float Q = 0.0f;
    if (live) {
        Q = -gr.grad_render_alphas[p];
        if (bg)
            for (int c = 0; c < nch; ++c) Q += gp[c] * bg[c];
    }
    const int n = live ? stp.count[p] : 0;
    // rec: the records hold every pair of the pixel; else the list walk
    const bool rec = n <= stp.max_steps;
    // the lane's next list position to visit (-1: none left) and, from a
    // record, the transmittance before that pair
    int32_t cur = -1;
    float t_rec = 0.0f;
    int s_next = n - 1;  // next record to read
    auto next_record = [&]() {
        cur = -1;
        while (s_next >= 0) {
            const int64_t o = (int64_t)s_next * stp.npix + p;
            --s_next;
            const int32_t j = stp.pos[o];
            if (j < 0 || j >= a.n_isects) {  // only from a corrupted trace
                GS_BOUNDS_REPORT(a.d_status);
                continue;
            }
            cur = j;
            t_rec = stp.T[o];
            return;
        }
    };
    if (live) {
        if (rec) {
            next_record();
        } else {
            const int64_t hi = min((int64_t)gr.last_ids[p], tr.end - 1);
            cur = hi >= tr.start ? (int32_t)hi : -1;
        }
    }
    float Tc = Tfinal;
    while (true) {
        const int32_t j = __reduce_max_sync(0xffffffffu, cur);
        if (j < 0) break;
        const bool mine = cur == j;
        // the entry's splat, the same for every lane
        const int32_t g = a.flatten_ids[j];
        const bool g_ok = (uint64_t)g < (uint64_t)CN;
        if (!g_ok && lane == 0) GS_BOUNDS_REPORT(a.d_status);
        bool take = false;
        float t_before = 0.0f, al = 0.0f, dx = 0.0f;
        PairEval e{0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        float q0 = 0.0f, q1 = 0.0f, q2 = 0.0f;
        if (g_ok) {
            const float2 m = reinterpret_cast<const float2*>(a.means2d)[g];
            const float* q = a.conics + 3 * (int64_t)g;
            q0 = q[0];
            q1 = q[1];
            q2 = q[2];
            if (mine) {
                const ColumnTerms ct = column_terms(m.x, q0, q1, px);
                dx = ct.dx;
                e = eval_pair(ct, m.y, q2, a.opacities[g], py);
                if (rec) {
                    // each record was composited by the forward with these
                    // same operations: only the T < 1 guard remains to test
                    al = Tc < 1.0f ? e.alpha : 0.0f;
                    t_before = t_rec;
                    take = true;
                } else if (e.s >= 0.0f && e.alpha >= a.alpha_cutoff && Tc < 1.0f) {
                    al = e.alpha;
                    t_before = Tc / (1.0f - e.alpha);
                    take = true;
                }
            }
        }
        if (mine) {
            if (rec) next_record();
            else cur = cur - 1 >= tr.start ? cur - 1 : -1;
        }
        const unsigned tm = __ballot_sync(0xffffffffu, take);
        if (tm == 0u) continue;
        const bool lone = (tm & (tm - 1u)) == 0u;
        // one field's terms into the splat's gradient
        auto add = [&](float* dst, float v) {
            if (lone) {
                if (take && v != 0.0f) atomicAdd(dst, v);
            } else {
                v = warp_sum(v);
                if (lane == 0 && v != 0.0f) atomicAdd(dst, v);
            }
        };
        const float* col = a.colors + (int64_t)g * nch;
        const float vis = t_before * al;
        float gcol = 0.0f;
        for (int c = 0; c < nch; ++c) {
            const float gc = take ? gp[c] : 0.0f;
            add(&gr.grad_colors[(int64_t)g * nch + c], gc * vis);
            gcol += gc * col[c];
        }
        const float g_alpha = t_before * (gcol - Q);
        const float g_raw = take && al > 0.0f && e.raw < kAlphaClamp ? g_alpha : 0.0f;
        const float g_s = -g_raw * e.raw;
        const float gmx = g_s * (q0 * dx + q1 * e.dy);
        const float gmy = g_s * (q2 * e.dy + q1 * dx);
        add(&gr.grad_opacities[g], g_raw * e.resp);
        add(&gr.grad_means2d[2 * (int64_t)g], gmx);
        add(&gr.grad_means2d[2 * (int64_t)g + 1], gmy);
        add(&gr.grad_conics[3 * (int64_t)g], g_s * (0.5f * dx * dx));
        add(&gr.grad_conics[3 * (int64_t)g + 1], g_s * (dx * e.dy));
        add(&gr.grad_conics[3 * (int64_t)g + 2], g_s * (0.5f * e.dy * e.dy));
        if (ABS) {
            add(&gr.grad_means2d_abs[2 * (int64_t)g], fabsf(gmx));
            add(&gr.grad_means2d_abs[2 * (int64_t)g + 1], fabsf(gmy));
        }
        if (take) {
            Q = al * gcol + (1.0f - al) * Q;
            Tc = t_before;
        }
    }
}

template <int CH>
void fwd_chunk(const RasterArgs& a, float* render_colors, float* render_alphas,
               int32_t* last_ids, int32_t* pair_counts, uint32_t* trace,
               const StepTrace* steps, cudaStream_t s) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    const dim3 g((unsigned)tiles), b(kThreads);
    if (steps)
        k_raster_fwd<CH, false, false, true><<<g, b, 0, s>>>(a, render_colors, render_alphas,
                                                            last_ids, nullptr, nullptr, *steps);
    else if (pair_counts && trace)
        k_raster_fwd<CH, true, true><<<g, b, 0, s>>>(a, render_colors, render_alphas, last_ids,
                                                     pair_counts, trace);
    else if (pair_counts)
        k_raster_fwd<CH, true, false><<<g, b, 0, s>>>(a, render_colors, render_alphas, last_ids,
                                                      pair_counts, nullptr);
    else if (trace)
        k_raster_fwd<CH, false, true><<<g, b, 0, s>>>(a, render_colors, render_alphas, last_ids,
                                                      nullptr, trace);
    else
        k_raster_fwd<CH, false, false><<<g, b, 0, s>>>(a, render_colors, render_alphas,
                                                       last_ids, nullptr, nullptr);
}

template <int CH>
void bwd_chunk(const RasterArgs& a, const RasterGrads& g, const uint32_t* trace,
               cudaStream_t s) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    const dim3 gd((unsigned)tiles), b(kThreads);
    if (g.grad_means2d_abs) {
        if (trace)
            k_raster_bwd<CH, true, true><<<gd, b, 0, s>>>(a, g, trace);
        else
            k_raster_bwd<CH, true, false><<<gd, b, 0, s>>>(a, g, nullptr);
    } else {
        if (trace)
            k_raster_bwd<CH, false, true><<<gd, b, 0, s>>>(a, g, trace);
        else
            k_raster_bwd<CH, false, false><<<gd, b, 0, s>>>(a, g, nullptr);
    }
}

}  // namespace

// Channels are processed in chunks of up to 4 (one launch each): compositing
// is independent per channel, and every per-splat term of the backward is
// linear in the per-channel sum, so the chunks' atomic contributions add up
// to the full gradient (the render_alpha term is added by the first chunk).
void launch_raster_fwd(RasterArgs a, float* render_colors, float* render_alphas,
                       int32_t* last_ids, int32_t* pair_counts, uint32_t* trace,
                       cudaStream_t s, const StepArgs* step_args) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    if (tiles <= 0) return;
    StepTrace stp{};
    if (step_args)
        stp = StepTrace{step_args->pos, step_args->T, step_args->count, step_args->max_steps,
                        (int64_t)a.C * a.height * a.width};
    for (int off = 0; off < a.channels; off += 4) {
        a.ch_off = off;
        a.first_chunk = off == 0;
        const int ch = a.channels - off < 4 ? a.channels - off : 4;
        int32_t* pc = off == 0 ? pair_counts : nullptr;
        uint32_t* tr = off == 0 ? trace : nullptr;
        const StepTrace* st = off == 0 && step_args ? &stp : nullptr;
        switch (ch) {
            case 1: fwd_chunk<1>(a, render_colors, render_alphas, last_ids, pc, tr, st, s); break;
            case 2: fwd_chunk<2>(a, render_colors, render_alphas, last_ids, pc, tr, st, s); break;
            case 3: fwd_chunk<3>(a, render_colors, render_alphas, last_ids, pc, tr, st, s); break;
            default: fwd_chunk<4>(a, render_colors, render_alphas, last_ids, pc, tr, st, s); break;
        }
    }
}

void launch_raster_bwd_steps(RasterArgs a, const RasterGrads& g, const StepArgs& step_args,
                             cudaStream_t s) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    if (tiles <= 0) return;
    a.ch_off = 0;
    a.first_chunk = 1;
    const StepTrace stp{step_args.pos, step_args.T, step_args.count, step_args.max_steps,
                        (int64_t)a.C * a.height * a.width};
    const dim3 gd((unsigned)tiles), b(kStepThreads);
    if (g.grad_means2d_abs)
        k_raster_bwd_steps<true><<<gd, b, 0, s>>>(a, g, stp);
    else
        k_raster_bwd_steps<false><<<gd, b, 0, s>>>(a, g, stp);
}

void launch_raster_bwd(RasterArgs a, const RasterGrads& g, const uint32_t* trace,
                       cudaStream_t s) {
    const int64_t tiles = (int64_t)a.C * a.tile_width * a.tile_height;
    if (tiles <= 0) return;
    // above 4 channels the chunks leave absgrad to its own full-channel pass
    RasterGrads gc = g;
    if (a.channels > 4) gc.grad_means2d_abs = nullptr;
    for (int off = 0; off < a.channels; off += 4) {
        a.ch_off = off;
        a.first_chunk = off == 0;
        const int ch = a.channels - off < 4 ? a.channels - off : 4;
        switch (ch) {
            case 1: bwd_chunk<1>(a, gc, trace, s); break;
            case 2: bwd_chunk<2>(a, gc, trace, s); break;
            case 3: bwd_chunk<3>(a, gc, trace, s); break;
            default: bwd_chunk<4>(a, gc, trace, s); break;
        }
    }
    if (a.channels > 4 && g.grad_means2d_abs) {
        a.ch_off = 0;
        a.first_chunk = 1;
        const dim3 gd((unsigned)tiles), b(kThreads);
        if (trace)
            k_raster_bwd_absgrad<true><<<gd, b, 0, s>>>(a, g, trace);
        else
            k_raster_bwd_absgrad<false><<<gd, b, 0, s>>>(a, g, nullptr);
    }
}

}  // namespace gs
