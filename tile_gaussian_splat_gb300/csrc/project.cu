// EWA projection of 3D Gaussians into the raster path's 2D inputs.
//
// gsplat 1.0.0, data/ext/gsplat_native/projection.c: gs_project_one per
// (camera, Gaussian) pair (camera transform, pinhole Jacobian with the
// frustum clip, J S J^T + eps2d, 3.33-sigma radii, visibility, conic,
// compensation).  Every pair is independent, so the kernel is a plain
// streaming map: one thread per Gaussian, looping over the cameras, so the
// Gaussian's 48 bytes are read from HBM once however many cameras there are.
//
// Arithmetic: the page computes in single precision; here every operation is
// an explicitly rounded IEEE single operation (__fmul_rn, __fadd_rn,
// __fdiv_rn, __fsqrt_rn) in the page's evaluation order, with no
// contraction into FMA, so every output is reproducible bit for bit by any
// IEEE single-precision evaluation in that order.
#include <cstdint>

#include <cuda_runtime.h>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {
namespace {

constexpr int kProjThreads = 256;
constexpr int kCamChunk = 32;  // cameras staged in shared memory at a time

struct Camera {
    float R[9], t[3];
    float fx, skew, cx, k10, fy, cy;
};

__device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float dv(float a, float b) { return __fdiv_rn(a, b); }

// ceil(3.33 sqrt(max(v, 0))) as int32, saturating at 2^31 - 1
__device__ __forceinline__ int32_t radius_of(float v) {
    const float r = ceilf(mul(3.33f, __fsqrt_rn(fmaxf(v, 0.0f))));
    return r >= 2147483648.0f ? 2147483647 : (int32_t)r;
}

// 3x3 product, each entry accumulated from 0 in increasing inner index
__device__ __forceinline__ void mat3_mul(const float* a, const float* b, float* o) {
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < 3; ++k) acc = add(acc, mul(a[i * 3 + k], b[k * 3 + j]));
            o[i * 3 + j] = acc;
        }
}

__global__ void __launch_bounds__(kProjThreads)
    k_project(const float* __restrict__ means, const float* __restrict__ covars,
              const float* __restrict__ viewmats, const float* __restrict__ intrinsics, int C,
              int N, ProjectArgs pa, int32_t* __restrict__ radii, float* __restrict__ means2d,
              float* __restrict__ depths, float* __restrict__ conics,
              float* __restrict__ compensations, float* __restrict__ radii_float) {
    __shared__ float s_gauss[kProjThreads * 12];  // means then covars of the block
    __shared__ Camera s_cam[kCamChunk];
    const int tid = threadIdx.x;
    const int64_t n0 = (int64_t)blockIdx.x * kProjThreads;
    const int nb = (int)min((int64_t)kProjThreads, (int64_t)N - n0);

    // coalesced staging of the block's contiguous mean and covariance runs
    for (int k = tid; k < nb * 3; k += kProjThreads) s_gauss[k] = means[n0 * 3 + k];
    for (int k = tid; k < nb * 9; k += kProjThreads)
        s_gauss[kProjThreads * 3 + k] = covars[n0 * 9 + k];
    __syncthreads();
    float m[3], sig[9];
    if (tid < nb) {
#pragma unroll
        for (int k = 0; k < 3; ++k) m[k] = s_gauss[tid * 3 + k];
#pragma unroll
        for (int k = 0; k < 9; ++k) sig[k] = s_gauss[kProjThreads * 3 + tid * 9 + k];
    }
    const float W = (float)pa.width, H = (float)pa.height;

    for (int c0 = 0; c0 < C; c0 += kCamChunk) {
        const int nc = min(kCamChunk, C - c0);
        __syncthreads();
        for (int k = tid; k < nc; k += kProjThreads) {
            const float* V = viewmats + (int64_t)(c0 + k) * 16;
            const float* K = intrinsics + (int64_t)(c0 + k) * 9;
            Camera& cam = s_cam[k];
            cam.R[0] = V[0]; cam.R[1] = V[1]; cam.R[2] = V[2];
            cam.R[3] = V[4]; cam.R[4] = V[5]; cam.R[5] = V[6];
            cam.R[6] = V[8]; cam.R[7] = V[9]; cam.R[8] = V[10];
            cam.t[0] = V[3]; cam.t[1] = V[7]; cam.t[2] = V[11];
            cam.fx = K[0]; cam.skew = K[1]; cam.cx = K[2];
            cam.k10 = K[3]; cam.fy = K[4]; cam.cy = K[5];
        }
        __syncthreads();
        if (tid >= nb) continue;
        for (int cc = 0; cc < nc; ++cc) {
            const Camera& cam = s_cam[cc];
            // camera-space mean: ((r0 m0 + r1 m1) + r2 m2) + t
            float p[3];
#pragma unroll
            for (int i = 0; i < 3; ++i)
                p[i] = add(add(add(mul(cam.R[i * 3], m[0]), mul(cam.R[i * 3 + 1], m[1])),
                               mul(cam.R[i * 3 + 2], m[2])),
                           cam.t[i]);
            // camera-space covariance (R Sigma) R^T
            float rs[9], rt[9], S[9];
            mat3_mul(cam.R, sig, rs);
#pragma unroll
            for (int i = 0; i < 3; ++i)
#pragma unroll
                for (int j = 0; j < 3; ++j) rt[i * 3 + j] = cam.R[j * 3 + i];
            mat3_mul(rs, rt, S);

            const float depth = p[2];
            const bool out_depth = depth <= pa.near_plane || depth >= pa.far_plane;
            const float z = out_depth ? 1.0f : depth;
            float J[6] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            float u, v;
            if (pa.orthographic) {
                J[0] = cam.fx;
                J[4] = cam.fy;
                u = add(mul(p[0], cam.fx), cam.cx);
                v = add(mul(p[1], cam.fy), cam.cy);
            } else {
                // image extent in normalised coordinates, widened by 0.15 of
                // the image size on each side
                const float wx = dv(mul(0.15f, W), cam.fx);
                const float wy = dv(mul(0.15f, H), cam.fy);
                const float x_lo = -add(dv(cam.cx, cam.fx), wx);
                const float x_hi = add(dv(sub(W, cam.cx), cam.fx), wx);
                const float y_lo = -add(dv(cam.cy, cam.fy), wy);
                const float y_hi = add(dv(sub(H, cam.cy), cam.fy), wy);
                const float tx = mul(fminf(fmaxf(dv(p[0], z), x_lo), x_hi), z);
                const float ty = mul(fminf(fmaxf(dv(p[1], z), y_lo), y_hi), z);
                const float zz = mul(z, z);
                J[0] = dv(cam.fx, z);
                J[2] = dv(mul(-cam.fx, tx), zz);
                J[4] = dv(cam.fy, z);
                J[5] = dv(mul(-cam.fy, ty), zz);
                u = dv(add(add(mul(cam.fx, p[0]), mul(cam.skew, p[1])), mul(cam.cx, z)), z);
                v = dv(add(add(mul(cam.k10, p[0]), mul(cam.fy, p[1])), mul(cam.cy, z)), z);
            }
            // J S J^T, each entry summed over (l, r), r innermost
            float cov[4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float acc = 0.0f;
#pragma unroll
                    for (int l = 0; l < 3; ++l)
#pragma unroll
                        for (int r = 0; r < 3; ++r)
                            acc = add(acc, mul(mul(J[i * 3 + l], S[l * 3 + r]), J[j * 3 + r]));
                    cov[i * 2 + j] = acc;
                }
            const float det0 = sub(mul(cov[0], cov[3]), mul(cov[1], cov[2]));
            cov[0] = add(cov[0], pa.eps2d);
            cov[3] = add(cov[3], pa.eps2d);
            const float det = sub(mul(cov[0], cov[3]), mul(cov[1], cov[2]));
            const float det_safe = det <= 0.0f ? 1e-10f : det;
            const int32_t rx = radius_of(cov[0]);
            const int32_t ry = radius_of(cov[3]);
            const float frx = __int2float_rn(rx), fry = __int2float_rn(ry);
            const bool visible = det > 0.0f && depth > pa.near_plane && depth < pa.far_plane &&
                                 (frx > pa.radius_clip || fry > pa.radius_clip) &&
                                 add(u, frx) > 0.0f && sub(u, frx) < W && add(v, fry) > 0.0f &&
                                 sub(v, fry) < H;
            const int64_t i = (int64_t)(c0 + cc) * N + n0 + tid;
            const int32_t ox = visible ? rx : 0, oy = visible ? ry : 0;
            reinterpret_cast<int2*>(radii)[i] = make_int2(ox, oy);
            reinterpret_cast<float2*>(means2d)[i] = make_float2(u, v);
            depths[i] = depth;
            conics[3 * i] = dv(cov[3], det_safe);
            conics[3 * i + 1] = dv(-add(cov[1], cov[2]), mul(2.0f, det_safe));
            conics[3 * i + 2] = dv(cov[0], det_safe);
            if (compensations)
                compensations[i] = __fsqrt_rn(fmaxf(dv(det0, det_safe), 0.0f));
            if (radii_float)
                reinterpret_cast<float2*>(radii_float)[i] =
                    make_float2(__int2float_rn(ox), __int2float_rn(oy));
        }
    }
}

}  // namespace

void launch_project(const float* means, const float* covars, const float* viewmats,
                    const float* intrinsics, int C, int N, const ProjectArgs& pa, int32_t* radii,
                    float* means2d, float* depths, float* conics, float* compensations,
                    float* radii_float, cudaStream_t s) {
    if (N <= 0) return;
    const unsigned blocks = (unsigned)((N + kProjThreads - 1) / kProjThreads);
    k_project<<<blocks, kProjThreads, 0, s>>>(means, covars, viewmats, intrinsics, C, N, pa,
                                              radii, means2d, depths, conics, compensations,
                                              radii_float);
}

}  // namespace gs
