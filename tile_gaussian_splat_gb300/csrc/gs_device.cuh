// Device helpers shared by the kernels of libgs_splat_gb300 (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gs_splat.h"

namespace gs {

constexpr int kWarp = 32;

// Flags in the low two bits of a decoupled look-back word; the value sits in
// the upper 62 bits.  0 = not yet published.
constexpr uint64_t kFlagAggregate = 1;  // this block's own count
constexpr uint64_t kFlagPrefix = 2;     // inclusive prefix up to this block
constexpr uint64_t kFlagMask = 3;

// Default upper bound on polls of one look-back word.  A predecessor
// publishes within microseconds; the bound only matters when something has
// already gone wrong, and turns that into GS_ERR_TIMEOUT instead of a hang.
constexpr int kSpinLimit = 1 << 22;

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_i32(const int32_t* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Records the first error in the caller's status word (if any).
__device__ __forceinline__ void report(int32_t* d_status, int code) {
    if (d_status) atomicCAS(d_status, 0, code);
}

// The range-checking build (-DGS_DEBUG_BOUNDS): where an index read from the
// inputs (a list range, a flatten id) falls outside its array, every build
// skips the access; this build also reports GS_ERR_OUT_OF_BOUNDS.
#ifdef GS_DEBUG_BOUNDS
#define GS_BOUNDS_REPORT(d_status) report((d_status), GS_ERR_OUT_OF_BOUNDS)
#else
#define GS_BOUNDS_REPORT(d_status) ((void)0)
#endif

// Errors seen by a look-back wait: the internal abort flag (workspace) stops
// every other waiter at once, the caller's word gets the code.
struct ErrorSink {
    int32_t* abort_flag;  // workspace word, zeroed per call
    int32_t* d_status;    // caller's word or null
    int spin_limit = kSpinLimit;  // polls of one look-back word before GS_ERR_TIMEOUT
    __device__ __forceinline__ void raise(int code) const {
        atomicCAS(abort_flag, 0, code);
        report(d_status, code);
    }
    __device__ __forceinline__ bool aborted() const { return ld_relaxed_i32(abort_flag) != 0; }
};

// Polls *p until a flag is set.  Returns the word, or a word flagged PREFIX
// with value 0 after the bound (the error is raised, results are garbage but
// nothing hangs).
__device__ __forceinline__ uint64_t wait_published(const uint64_t* p, const ErrorSink& err) {
    uint64_t v = ld_relaxed_u64(p);
    int it = 0;
    while ((v & kFlagMask) == 0) {
        if (++it >= err.spin_limit) {
            err.raise(GS_ERR_TIMEOUT);
            return kFlagPrefix;
        }
        if ((it & 255) == 0 && err.aborted()) return kFlagPrefix;
        __nanosleep(32);
        v = ld_relaxed_u64(p);
    }
    return v;
}

// ---- one-dimensional bulk copies (TMA) into shared memory, completed on an
// mbarrier.  Addresses 16-byte aligned, sizes multiples of 16 bytes.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arms the barrier's current phase for `bytes` of bulk-copy data (one arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_to_shared(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Waits, at most `polls` bounded try_wait rounds, for phase `parity` of the
// barrier to complete; false if it did not.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int polls) {
    for (int i = 0; i < polls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// The lanes of the warp whose `valid` is set and whose digit d (its low
// `nbits` bits, nbits <= 8, the same in every lane) equals this lane's:
// one ballot per digit bit, each lane keeping the lanes that agree with it
// on that bit.  All 32 lanes must call it.  In the radix passes' ranking
// (twelve calls back to back per thread) this measured 8-10 % faster per
// emit+sort call than the match.any instruction; in the emission's
// histograms (two calls per pair among other work) match.any stays faster.
__device__ __forceinline__ unsigned digit_peers(uint32_t d, bool valid, int nbits) {
    unsigned pm = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        if (b < nbits) {
            const unsigned bit = (d >> b) & 1u;
            const unsigned bb = __ballot_sync(0xffffffffu, bit);
            pm &= bit ? bb : ~bb;
        }
    }
    return pm;
}

// Block-wide exclusive scan of one int64 per thread (blockDim.x == 32*W).
// `scratch` holds >= 32 int64.  Returns the exclusive prefix; *total gets the
// block sum.  Contains __syncthreads.
template <int THREADS>
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* scratch,
                                                        int64_t* total) {
    constexpr int W = THREADS / kWarp;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t s = lane < W ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < W) scratch[lane] = s;  // inclusive warp totals
    }
    __syncthreads();
    int64_t warp_prefix = warp == 0 ? 0 : scratch[warp - 1];
    *total = scratch[W - 1];
    return warp_prefix + x - v;
}

// Tile rect of one splat (gsplat 1.0.0, intersections.c, gs_bounds) in IEEE
// single precision: sub and div round once each, floor/ceil are exact.  A
// non-finite mean or radius gives the empty rect; values beyond the grid
// clamp to its edge before conversion, so no conversion is out of range.
struct Rect {
    int x0, y0, x1, y1;
};

__device__ __forceinline__ int clamp_to_grid(float v, int maximum) {
    if (!(v > 0.0f)) return 0;
    if (v >= (float)maximum) return maximum;
    return (int)v;
}

// v / ts in IEEE single precision.  When ts is a power of two its
// reciprocal is exact and v * (1 / ts) is the correctly rounded value of the
// same real number as v / ts, so the multiply gives the division's bits
// (subnormal, infinite and NaN results included); inv_ts > 0 selects it and
// is passed only for such ts (exact_tile_inverse).
__device__ __forceinline__ float div_tile(float v, float ts, float inv_ts) {
    return inv_ts > 0.0f ? __fmul_rn(v, inv_ts) : __fdiv_rn(v, ts);
}

__device__ __forceinline__ Rect splat_rect(float mx, float my, float rx, float ry, float ts,
                                           float inv_ts, int tile_width, int tile_height) {
    Rect r = {0, 0, 0, 0};
    if (!(isfinite(mx) && isfinite(my) && isfinite(rx) && isfinite(ry))) return r;
    if (rx <= 0.0f || ry <= 0.0f) return r;
    r.x0 = clamp_to_grid(floorf(div_tile(__fsub_rn(mx, rx), ts, inv_ts)), tile_width);
    r.y0 = clamp_to_grid(floorf(div_tile(__fsub_rn(my, ry), ts, inv_ts)), tile_height);
    r.x1 = clamp_to_grid(ceilf(div_tile(__fadd_rn(mx, rx), ts, inv_ts)), tile_width);
    r.y1 = clamp_to_grid(ceilf(div_tile(__fadd_rn(my, ry), ts, inv_ts)), tile_height);
    return r;
}

}  // namespace gs
