// Throughput probes for the roofline of the raster kernels: how many FP32
// fused multiply-adds (scalar, and packed f32x2) and how many ex2.approx
// special-function operations this GPU completes per second.  Not part of the
// path; the bench times them with CUDA events and divides the raster kernels'
// algorithmic operation counts by the results.
//
// Each thread runs independent dependency chains (enough of them, with 64
// warps per SM, to hide the pipes' latency), and writes the sum of its chains
// so that nothing is dead code.  The values stay in a normal range: the FMA
// chains converge to 1 (x <- 0.999 x + 0.001), the ex2 chains stay in
// [0.5, 1] (x <- 2^-x).
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;

__device__ __forceinline__ float ex2_approx(float v) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(v));
    return y;
}

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) k_peak_probe(int iters, float* __restrict__ out) {
    const int gid = blockIdx.x * kProbeThreads + threadIdx.x;
    float sum = 0.0f;
    if (KIND == 1) {
        float2 v[kChains];
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            v[i] = make_float2(0.5f + 1e-3f * i + 1e-7f * threadIdx.x, 0.25f + 1e-3f * i);
        const float2 a = make_float2(0.999f, 0.999f), b = make_float2(1e-3f, 1e-3f);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int i = 0; i < kChains; ++i) v[i] = __ffma2_rn(v[i], a, b);
        }
#pragma unroll
        for (int i = 0; i < kChains; ++i) sum += v[i].x + v[i].y;
    } else {
        float x[kChains];
#pragma unroll
        for (int i = 0; i < kChains; ++i) x[i] = 0.5f + 1e-3f * i + 1e-7f * threadIdx.x;
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int i = 0; i < kChains; ++i)
                    x[i] = KIND == 0 ? __fmaf_rn(x[i], 0.999f, 1e-3f) : ex2_approx(-x[i]);
        }
#pragma unroll
        for (int i = 0; i < kChains; ++i) sum += x[i];
    }
    out[gid] = sum;
}

}  // namespace

int64_t launch_peak_probe(int kind, int iters, int blocks, float* out, cudaStream_t s) {
    const int64_t threads = (int64_t)blocks * kProbeThreads;
    switch (kind) {
        case 0:
            k_peak_probe<0><<<blocks, kProbeThreads, 0, s>>>(iters, out);
            return threads * iters * 4 * kChains;
        case 1:
            k_peak_probe<1><<<blocks, kProbeThreads, 0, s>>>(iters, out);
            return threads * iters * 4 * kChains * 2;
        default:
            k_peak_probe<2><<<blocks, kProbeThreads, 0, s>>>(iters, out);
            return threads * iters * 4 * kChains;
    }
}

}  // namespace gs
