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
