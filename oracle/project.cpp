// CPU oracle for the EWA projection that produces the raster path's inputs.
//
// TEST INFRASTRUCTURE ONLY.  A plain, slow, single-threaded restatement of
// the projection; only the tests, the smoke check and the bench's
// CPU-baseline leg may load it.  It shares no code, header, table or helper
// with the CUDA library (tile_gaussian_splat_gb300/csrc), and the library
// never calls it.  Built with oracle.cpp into one library (oracle/build.py):
// single precision as on the page, no FMA contraction, so every expression
// rounds in the order written here.
//
// Source (page title, file, function):
//   [G-proj] gsplat 1.0.0, data/ext/gsplat_native/projection.c:
//            gs_mat3_product, gs_camera_covar, gs_clip, gs_project_one,
//            gs_projection_without_gvl (one independent result per
//            (camera, Gaussian) pair), gs_projection_forward (argument set).
//
// Per (camera c, Gaussian n), with the view matrix V (4x4 row-major,
// rotation R = V[0:3, 0:3], translation t = V[0:3, 3]) and intrinsics K (3x3
// row-major):
//   p = R mean + t                    (camera-space mean; depth = p.z)
//   S = R Sigma R^T                   (camera-space covariance)
//   z = p.z unless it lies outside (near, far), else 1
//   perspective: the Jacobian of the pinhole map at p, with x/z and y/z
//     clamped to the image extent widened by 0.15 of its size on each side;
//     means2d = (K row 0 . (x, y, z), K row 1 . (x, y, z)) / z
//   orthographic: Jacobian diag(fx, fy); means2d = (fx x + cx, fy y + cy)
//   cov2d = J S J^T; the determinant before and after adding eps2d to the
//     diagonal; radius_i = ceil(3.33 sqrt(max(cov2d_ii, 0)));
//   visible = det > 0, near < depth < far, a radius above radius_clip and
//     the radius box overlapping the image; radii = visible ? r : 0
//   conic = inverse of cov2d as (a, b, c); compensation = sqrt(max(det0 /
//     det, 0)).  means2d, depths and conics are written for every pair.
//
// Readings where the page is silent:
//   * The page converts ceil(3.33 sqrt(.)) to int32 with a plain cast, which
//     C leaves undefined above 2^31 - 1; here it saturates to 2^31 - 1 (a
//     non-negative value cannot go below 0).
//   * The page's double parameters (eps2d, near, far, radius_clip) are
//     stored as float before use, as its argument struct does.

#include <cmath>
#include <cstdint>

namespace {

// [G-proj] gs_mat3_product: row-by-column, each entry summed from 0 in
// increasing inner index.
void mat3_mul(const float* a, const float* b, float* out) {
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < 3; ++k) acc += a[i * 3 + k] * b[k * 3 + j];
            out[i * 3 + j] = acc;
        }
}

// [G-proj] gs_camera_covar: (R Sigma) R^T.
void rotate_covariance(const float* R, const float* sigma, float* out) {
    float rs[9], rt[9];
    mat3_mul(R, sigma, rs);
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) rt[i * 3 + j] = R[j * 3 + i];
    mat3_mul(rs, rt, out);
}

// [G-proj] gs_clip.
float clamp_to(float v, float lo, float hi) { return fminf(fmaxf(v, lo), hi); }

int32_t radius_of(float variance) {
    const float r = ceilf(3.33f * sqrtf(fmaxf(variance, 0.0f)));
    return r >= 2147483648.0f ? INT32_MAX : (int32_t)r;
}

struct ProjParams {
    int64_t N;
    int width, height, orthographic;
    float eps2d, near_plane, far_plane, radius_clip;
};

// [G-proj] gs_project_one.
void project_pair(const ProjParams& P, const float* mean, const float* sigma, const float* V,
                  const float* K, int32_t* radii, float* means2d, float* depth_out, float* conic,
                  float* compensation) {
    const float R[9] = {V[0], V[1], V[2], V[4], V[5], V[6], V[8], V[9], V[10]};
    float p[3];
    for (int i = 0; i < 3; ++i)
        p[i] = R[i * 3] * mean[0] + R[i * 3 + 1] * mean[1] + R[i * 3 + 2] * mean[2] + V[i * 4 + 3];
    float S[9];
    rotate_covariance(R, sigma, S);

    const float depth = p[2];
    const bool outside_depth = depth <= P.near_plane || depth >= P.far_plane;
    const float z = outside_depth ? 1.0f : depth;
    const float fx = K[0], fy = K[4], cx = K[2], cy = K[5];
    float J[6] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};  // 2x3, row-major
    float uv[2];
    if (P.orthographic) {
        J[0] = fx;
        J[4] = fy;
        uv[0] = p[0] * fx + cx;
        uv[1] = p[1] * fy + cy;
    } else {
        // the image extent in normalised coordinates, widened by 0.15 of the
        // image size on each side
        const float W = (float)P.width, H = (float)P.height;
        const float x_lo = -(cx / fx + 0.15f * W / fx);
        const float x_hi = (W - cx) / fx + 0.15f * W / fx;
        const float y_lo = -(cy / fy + 0.15f * H / fy);
        const float y_hi = (H - cy) / fy + 0.15f * H / fy;
        const float tx = clamp_to(p[0] / z, x_lo, x_hi) * z;
        const float ty = clamp_to(p[1] / z, y_lo, y_hi) * z;
        J[0] = fx / z;
        J[2] = -fx * tx / (z * z);
        J[4] = fy / z;
        J[5] = -fy * ty / (z * z);
        uv[0] = (fx * p[0] + K[1] * p[1] + cx * z) / z;
        uv[1] = (K[3] * p[0] + fy * p[1] + cy * z) / z;
    }
    // J S J^T, each entry summed over (l, r) with r innermost
    float cov[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 2; ++j)
            for (int l = 0; l < 3; ++l)
                for (int r = 0; r < 3; ++r) cov[i * 2 + j] += J[i * 3 + l] * S[l * 3 + r] * J[j * 3 + r];

    const float det0 = cov[0] * cov[3] - cov[1] * cov[2];
    cov[0] += P.eps2d;
    cov[3] += P.eps2d;
    const float det = cov[0] * cov[3] - cov[1] * cov[2];
    const float det_safe = det <= 0.0f ? 1e-10f : det;
    const int32_t rx = radius_of(cov[0]);
    const int32_t ry = radius_of(cov[3]);
    const bool visible = det > 0.0f && depth > P.near_plane && depth < P.far_plane &&
                         ((float)rx > P.radius_clip || (float)ry > P.radius_clip) &&
                         uv[0] + (float)rx > 0.0f && uv[0] - (float)rx < (float)P.width &&
                         uv[1] + (float)ry > 0.0f && uv[1] - (float)ry < (float)P.height;
    radii[0] = visible ? rx : 0;
    radii[1] = visible ? ry : 0;
    means2d[0] = uv[0];
    means2d[1] = uv[1];
    *depth_out = depth;
    conic[0] = cov[3] / det_safe;
    conic[1] = -(cov[1] + cov[2]) / (2.0f * det_safe);
    conic[2] = cov[0] / det_safe;
    if (compensation) *compensation = sqrtf(fmaxf(det0 / det_safe, 0.0f));
}

}  // namespace

extern "C" {

// [G-proj] gs_projection_without_gvl / gs_projection_forward.
// means (N,3), covars (N,3,3), viewmats (C,4,4), intrinsics (C,3,3); outputs
// radii int32 (C,N,2), means2d (C,N,2), depths (C,N), conics (C,N,3),
// compensations (C,N) or NULL.  Returns 0, or 1 on bad sizes.
int orc_project(const float* means, const float* covars, const float* viewmats,
                const float* intrinsics, int64_t C, int64_t N, int width, int height,
                float eps2d, float near_plane, float far_plane, float radius_clip,
                int orthographic, int32_t* radii, float* means2d, float* depths, float* conics,
                float* compensations) {
    if (C < 1 || N < 0 || width < 1 || height < 1) return 1;
    const ProjParams P{N, width, height, orthographic, eps2d, near_plane, far_plane, radius_clip};
    for (int64_t c = 0; c < C; ++c)
        for (int64_t n = 0; n < N; ++n) {
            const int64_t i = c * N + n;
            project_pair(P, means + 3 * n, covars + 9 * n, viewmats + 16 * c, intrinsics + 9 * c,
                         radii + 2 * i, means2d + 2 * i, depths + i, conics + 3 * i,
                         compensations ? compensations + i : nullptr);
        }
    return 0;
}

}  // extern "C"
