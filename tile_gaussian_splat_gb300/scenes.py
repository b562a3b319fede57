"""Seeded synthetic splat scenes for the five workloads of the tile-binned
Gaussian-splat raster path.

This module only draws inputs.  It contains none of the rasterizer's
arithmetic (no tile bounds, no keys, no compositing); both the CUDA library
and the CPU oracle consume the arrays it returns, so the two sides always see
bit-identical inputs.

Every array is a C-contiguous numpy array on the host:

  means2d   float32 (C, N, 2)   pixel-space centres
  radii     float32 (C, N)      isotropic radius (workload 1)
            float32 (C, N, 2)   elliptical radii (rx, ry) (workloads 2-4)
  depths    float32 (C, N)
  conics    float32 (C, N, 3)   (a, b, c) of the inverse 2D covariance
                                [[a, b], [b, c]]
  colors    float32 (C, N, 3)
  opacities float32 (C, N)
  backgrounds float32 (C, 3) or None

The draw order is fixed (means, axis sigmas, rotation, depth, opacity,
colour; cameras drawn one after the other) so a seed names one scene.
The generator is numpy's PCG64, which gives the same stream on x86 and Arm.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

ALPHA_CUTOFF = np.float32(1.0 / 255.0)
TRANSMITTANCE_THRESHOLD = np.float32(1e-4)


@dataclasses.dataclass
class Scene:
    name: str
    C: int
    N: int
    width: int
    height: int
    tile_size: int
    means2d: np.ndarray
    radii: np.ndarray
    depths: np.ndarray
    conics: np.ndarray
    colors: np.ndarray
    opacities: np.ndarray
    backgrounds: np.ndarray | None
    alpha_cutoff: np.float32 = ALPHA_CUTOFF
    transmittance_threshold: np.float32 = TRANSMITTANCE_THRESHOLD

    @property
    def elliptical(self) -> bool:
        return self.radii.ndim == 3

    @property
    def tile_width(self) -> int:
        return (self.width + self.tile_size - 1) // self.tile_size

    @property
    def tile_height(self) -> int:
        return (self.height + self.tile_size - 1) // self.tile_size

    @property
    def channels(self) -> int:
        return self.colors.shape[-1]

    def arrays(self) -> dict:
        return {k: getattr(self, k) for k in
                ("means2d", "radii", "depths", "conics", "colors", "opacities", "backgrounds")}


def _covariance_from_axes(s1, s2, theta):
    """Sigma = R(theta) diag(s1^2, s2^2) R(theta)^T, in float64."""
    ct, st = np.cos(theta), np.sin(theta)
    v1, v2 = s1 * s1, s2 * s2
    sxx = ct * ct * v1 + st * st * v2
    syy = st * st * v1 + ct * ct * v2
    sxy = ct * st * (v1 - v2)
    return sxx, sxy, syy


def _conic(sxx, sxy, syy):
    det = sxx * syy - sxy * sxy
    return np.stack([syy / det, -sxy / det, sxx / det], axis=-1).astype(np.float32)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _loguniform(rng, lo, hi, size):
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size))


def _finish(name, C, N, W, H, ts, means, radii, depths, conics, colors, opac, bg):
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return Scene(name=name, C=C, N=N, width=W, height=H, tile_size=ts,
                 means2d=f32(means), radii=f32(radii), depths=f32(depths),
                 conics=f32(conics), colors=f32(colors), opacities=f32(opac),
                 backgrounds=None if bg is None else f32(bg))


def workload1(seed: int = 0) -> Scene:
    """1 camera, 256 splats, 64x64, tile 16, isotropic radius ceil(3 max sigma)."""
    C, N, W, H = 1, 256, 64, 64
    rng = np.random.Generator(np.random.PCG64(seed))
    means = rng.uniform(0.0, 64.0, (C, N, 2))
    sig = rng.uniform(1.0, 4.0, (C, N, 2))
    theta = rng.uniform(0.0, math.pi, (C, N))
    depth = rng.uniform(1.0, 10.0, (C, N))
    opac = rng.uniform(0.1, 0.9, (C, N))
    rgb = rng.uniform(0.0, 1.0, (C, N, 3))
    sxx, sxy, syy = _covariance_from_axes(sig[..., 0], sig[..., 1], theta)
    radii = np.ceil(3.0 * sig.max(axis=-1))
    return _finish("w1_256_64x64", C, N, W, H, 16, means, radii, depth,
                   _conic(sxx, sxy, syy), rgb, opac, np.zeros((C, 3)))


def _elliptical_radii(sxx, syy):
    return np.stack([np.ceil(3.0 * np.sqrt(sxx)), np.ceil(3.0 * np.sqrt(syy))], axis=-1)


def workload2(seed: int = 0, N: int = 100_000, W: int = 1024, H: int = 1024) -> Scene:
    """1 camera, 100k splats, 1024x1024, elliptical radii, means 10% past borders."""
    C = 1
    rng = np.random.Generator(np.random.PCG64(seed))
    mx = rng.uniform(-0.1 * W, 1.1 * W, (C, N))
    my = rng.uniform(-0.1 * H, 1.1 * H, (C, N))
    sig = _loguniform(rng, 0.5, 16.0, (C, N, 2))
    theta = rng.uniform(0.0, math.pi, (C, N))
    depth = rng.uniform(0.5, 50.0, (C, N))
    opac = _sigmoid(rng.normal(0.0, 1.5, (C, N)))
    rgb = rng.uniform(0.0, 1.0, (C, N, 3))
    sxx, sxy, syy = _covariance_from_axes(sig[..., 0], sig[..., 1], theta)
    return _finish(f"w2_{N}_{W}x{H}", C, N, W, H, 16, np.stack([mx, my], -1),
                   _elliptical_radii(sxx, syy), depth, _conic(sxx, sxy, syy), rgb, opac, None)


def workload3(seed: int = 0, C: int = 4, N: int = 1_000_000, W: int = 1920, H: int = 1080) -> Scene:
    """4 cameras x 1M splats, 1920x1080; 80% of means in 64 clusters
    (std 5% of width), 20% uniform; sigmas log-normal(ln 2, 0.8) in [0.3, 64]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    means = np.empty((C, N, 2))
    sig = np.empty((C, N, 2))
    theta = np.empty((C, N))
    depth = np.empty((C, N))
    opac = np.empty((C, N))
    rgb = np.empty((C, N, 3))
    std = 0.05 * W
    for c in range(C):
        centres = rng.uniform([0.0, 0.0], [W, H], (64, 2))
        in_cluster = rng.uniform(0.0, 1.0, N) < 0.8
        which = rng.integers(0, 64, N)
        clustered = centres[which] + rng.normal(0.0, std, (N, 2))
        uniform = rng.uniform([0.0, 0.0], [W, H], (N, 2))
        means[c] = np.where(in_cluster[:, None], clustered, uniform)
        sig[c] = np.clip(np.exp(rng.normal(math.log(2.0), 0.8, (N, 2))), 0.3, 64.0)
        theta[c] = rng.uniform(0.0, math.pi, N)
        depth[c] = _loguniform(rng, 0.2, 100.0, N)
        opac[c] = _sigmoid(rng.normal(0.0, 2.0, N))
        rgb[c] = rng.uniform(0.0, 1.0, (N, 3))
    sxx, sxy, syy = _covariance_from_axes(sig[..., 0], sig[..., 1], theta)
    return _finish(f"w3_{C}x{N}_{W}x{H}", C, N, W, H, 16, means,
                   _elliptical_radii(sxx, syy), depth, _conic(sxx, sxy, syy), rgb, opac, None)


def workload4(seed: int = 0, N: int = 6_000_000, W: int = 3840, H: int = 2160) -> Scene:
    """1 camera x 6M splats, 3840x2160; 90% of means uniform in a central disk
    of radius 25% of width, 10% uniform; sigmas log-normal(ln 4, 1) in [0.3, 128]."""
    C = 1
    rng = np.random.Generator(np.random.PCG64(seed))
    in_disk = rng.uniform(0.0, 1.0, N) < 0.9
    r = 0.25 * W * np.sqrt(rng.uniform(0.0, 1.0, N))
    phi = rng.uniform(0.0, 2.0 * math.pi, N)
    disk = np.stack([W / 2 + r * np.cos(phi), H / 2 + r * np.sin(phi)], -1)
    uniform = rng.uniform([0.0, 0.0], [W, H], (N, 2))
    means = np.where(in_disk[:, None], disk, uniform)[None]
    sig = np.clip(np.exp(rng.normal(math.log(4.0), 1.0, (C, N, 2))), 0.3, 128.0)
    theta = rng.uniform(0.0, math.pi, (C, N))
    depth = rng.uniform(1.0, 30.0, (C, N))
    opac = rng.uniform(0.05, 0.95, (C, N))
    rgb = rng.uniform(0.0, 1.0, (C, N, 3))
    sxx, sxy, syy = _covariance_from_axes(sig[..., 0], sig[..., 1], theta)
    return _finish(f"w4_{N}_{W}x{H}", C, N, W, H, 16, means,
                   _elliptical_radii(sxx, syy), depth, _conic(sxx, sxy, syy), rgb, opac, None)


def upstream_grads(C: int, H: int, W: int, channels: int = 3, seed: int = 1):
    """dL/d(render_colors) (C,H,W,ch) and dL/d(render_alphas) (C,H,W,1), N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    g_rgb = rng.standard_normal((C, H, W, channels)).astype(np.float32)
    g_a = rng.standard_normal((C, H, W, 1)).astype(np.float32)
    return g_rgb, g_a


def random_small(seed: int, C: int = 1, N: int = 16, W: int = 32, H: int = 32,
                 tile_size: int = 16, elliptical: bool = True, sigma=(1.0, 5.0),
                 opacity=(0.05, 0.95), background: bool = True, radius_scale: float = 3.0,
                 channels: int = 3) -> Scene:
    """Small generic scene (tests): uniform means inside the image, uniform sigmas,
    `channels` colour channels per splat uniform in [0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    means = rng.uniform([0.0, 0.0], [W, H], (C, N, 2))
    sig = rng.uniform(sigma[0], sigma[1], (C, N, 2))
    theta = rng.uniform(0.0, math.pi, (C, N))
    depth = rng.uniform(1.0, 10.0, (C, N))
    opac = rng.uniform(opacity[0], opacity[1], (C, N))
    rgb = rng.uniform(0.0, 1.0, (C, N, channels))
    sxx, sxy, syy = _covariance_from_axes(sig[..., 0], sig[..., 1], theta)
    if elliptical:
        radii = np.stack([np.ceil(radius_scale * np.sqrt(sxx)),
                          np.ceil(radius_scale * np.sqrt(syy))], axis=-1)
    else:
        radii = np.ceil(radius_scale * sig.max(axis=-1))
    bg = rng.uniform(0.0, 1.0, (C, channels)) if background else None
    return _finish(f"small_{seed}", C, N, W, H, tile_size, means, radii, depth,
                   _conic(sxx, sxy, syy), rgb, opac, bg)


WORKLOADS = {
    1: workload1,
    2: workload2,
    3: workload3,
    4: workload4,
}


def workload(k: int, seed: int = 0) -> Scene:
    """Workload 5 is workload 2's scene (its backward adds upstream_grads, seed 1)."""
    if k == 5:
        return workload2(seed)
    return WORKLOADS[k](seed)


# ---------------------------------------------------------------------------
# 3D inputs of the projection that produces the 2D splats.
#
#   means       float32 (N, 3)      world-space centres
#   covars      float32 (N, 3, 3)   world-space covariances (symmetric)
#   viewmats    float32 (C, 4, 4)   world-to-camera, row-major [R | t; 0 0 0 1]
#   intrinsics  float32 (C, 3, 3)   [[fx, skew, cx], [0, fy, cy], [0, 0, 1]]
#
# Camera convention of the pinhole map: x right, y down, z forward.


@dataclasses.dataclass
class Scene3D:
    name: str
    width: int
    height: int
    means: np.ndarray
    covars: np.ndarray
    viewmats: np.ndarray
    intrinsics: np.ndarray
    eps2d: float = 0.3
    near_plane: float = 0.01
    far_plane: float = 1e10
    radius_clip: float = 0.0

    @property
    def C(self) -> int:
        return self.viewmats.shape[0]

    @property
    def N(self) -> int:
        return self.means.shape[0]


def random_rotations(rng, n):
    """n rotation matrices (float64) from uniformly drawn unit quaternions."""
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    w, x, y, z = q[:, 0], q[:, 1], q[:, 2], q[:, 3]
    return np.stack([
        1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y),
        2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x),
        2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)], axis=1).reshape(n, 3, 3)


def look_at(eye, target, up=(0.0, -1.0, 0.0)):
    """World-to-camera 4x4 (float64) for a camera at `eye` looking at `target`,
    z forward, y down (the `up` hint points up in the image)."""
    eye = np.asarray(eye, np.float64)
    f = np.asarray(target, np.float64) - eye
    f /= np.linalg.norm(f)
    down = -np.asarray(up, np.float64)
    r = np.cross(down, f)
    r /= np.linalg.norm(r)
    d = np.cross(f, r)
    R = np.stack([r, d, f])  # rows: camera axes in world coordinates
    V = np.eye(4)
    V[:3, :3] = R
    V[:3, 3] = -R @ eye
    return V


def _covars_from_scales(rng, scales):
    R = random_rotations(rng, scales.shape[0])
    M = R * scales[:, None, :]
    return M @ np.transpose(M, (0, 2, 1))


def scene3d(seed: int = 0, C: int = 4, N: int = 1_000_000, W: int = 1920, H: int = 1080,
            focal: float = 1100.0) -> Scene3D:
    """Gaussians in the cube [-1, 1]^3 (64 clusters, std 0.15, plus 20 %
    uniform), axis scales log-normal(mean ln 0.01, std 0.8) clipped to
    [1e-4, 0.5], uniform orientations; C cameras on a circle of radius 3
    around the origin at height 0.5, all looking at the origin, focal
    `focal` px, principal point at the image centre."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_bg = N // 5
    centres = rng.uniform(-0.8, 0.8, (64, 3))
    which = rng.integers(0, 64, N - n_bg)
    means = np.concatenate([centres[which] + rng.normal(0.0, 0.15, (N - n_bg, 3)),
                            rng.uniform(-1.0, 1.0, (n_bg, 3))])
    scales = np.clip(np.exp(rng.normal(math.log(0.01), 0.8, (N, 3))), 1e-4, 0.5)
    covars = _covars_from_scales(rng, scales)
    views, Ks = [], []
    for c in range(C):
        a = 2 * math.pi * c / C + 0.3
        views.append(look_at((3.0 * math.cos(a), -0.5, 3.0 * math.sin(a)), (0.0, 0.0, 0.0)))
        Ks.append([[focal, 0.0, W / 2], [0.0, focal, H / 2], [0.0, 0.0, 1.0]])
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return Scene3D(name=f"proj_{C}x{N}_{W}x{H}", width=W, height=H, means=f32(means),
                   covars=f32(covars), viewmats=f32(np.stack(views)), intrinsics=f32(Ks))


def scene3d_edge(seed: int = 0, N: int = 4000, W: int = 200, H: int = 120) -> Scene3D:
    """Small scene (tests) that exercises every branch of the projection: two
    cameras (one with skew and off-centre principal point), Gaussians in
    front of, behind and beside the cameras, some far outside the frustum,
    some at the near plane, a few with degenerate (rank-deficient or zero)
    and a few with huge covariances."""
    rng = np.random.Generator(np.random.PCG64(seed))
    means = rng.uniform([-6.0, -4.0, -3.0], [6.0, 4.0, 12.0], (N, 3))
    scales = np.exp(rng.uniform(math.log(1e-3), math.log(2.0), (N, 3)))
    covars = _covars_from_scales(rng, scales)
    k = N // 40
    covars[:k] = 0.0                                   # zero covariance
    covars[k:2 * k, 2, :] = 0.0                        # rank-deficient
    covars[k:2 * k, :, 2] = 0.0
    covars[2 * k:3 * k] *= 1e12                        # huge radius
    covars[5 * k:6 * k] *= 1e16                        # radius saturates / det overflows
    means[3 * k:4 * k, 2] = 0.01                       # on the near plane
    means[4 * k:5 * k, :2] *= 50.0                     # far outside the frustum
    views = [look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0)),
             look_at((3.0, -1.0, -3.0), (0.2, 0.1, 1.0))]
    Ks = [[[180.0, 0.0, W / 2], [0.0, 170.0, H / 2], [0.0, 0.0, 1.0]],
          [[150.0, 2.5, 0.4 * W], [0.0, 160.0, 0.6 * H], [0.0, 0.0, 1.0]]]
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return Scene3D(name=f"proj_edge_{seed}", width=W, height=H, means=f32(means),
                   covars=f32(covars), viewmats=f32(np.stack(views)), intrinsics=f32(Ks))
