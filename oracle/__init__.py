"""CPU oracle of the tile-binned Gaussian-splat raster path (ctypes binding).

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may import this package.  It is a plain, slow restatement of what
the path computes (oracle.cpp) and shares no code with the CUDA library.

Every function takes and returns host numpy arrays.
"""

from __future__ import annotations

import ctypes as ct
import os

import numpy as np

from . import build as _build

_lib = None
_lib_omp = None

P = ct.c_void_p
I64 = ct.c_int64
I32 = ct.c_int
F32 = ct.c_float
F64 = ct.c_double


def lib(omp=False):
    """The single-threaded oracle, or (omp=True) its OpenMP build, which runs
    the raster pixel loops on every host core (timing only)."""
    global _lib, _lib_omp
    if omp:
        if _lib_omp is None:
            _lib_omp = _load(_build.build(omp=True))
        return _lib_omp
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


def threads_omp():
    """Threads the OpenMP build uses (OMP_NUM_THREADS, else every core)."""
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def _load(path):
    L = ct.CDLL(path)
    L.orc_tile_bits.argtypes = [I32, I32]
    L.orc_tile_bits.restype = I32
    L.orc_bounds.argtypes = [P, P, I32, I64, I64, I32, I32, I32, P]
    L.orc_bounds.restype = None
    L.orc_isect_count.argtypes = [P, P, I32, I64, I64, I32, I32, I32, P]
    L.orc_isect_count.restype = I64
    L.orc_isect_emit.argtypes = [P, P, I32, P, I64, I64, I32, I32, I32, P, P, I64]
    L.orc_isect_emit.restype = I64
    L.orc_sort_stable.argtypes = [P, P, I64]
    L.orc_sort_stable.restype = None
    L.orc_sort_lsd.argtypes = [P, P, I64]
    L.orc_sort_lsd.restype = I32
    L.orc_tile_offsets.argtypes = [P, I64, I32, I32, I32, P]
    L.orc_tile_offsets.restype = I32
    L.orc_rasterize_fwd.argtypes = [P, P, P, P, P, P, I64, I64, I32, I32, I32, I32, I32, I32,
                                    P, P, I64, F32, F32, P, I64, P, P, P, P, P, F32, F32,
                                    P, P, I32, P, P, P]
    L.orc_rasterize_fwd.restype = I32
    L.orc_rasterize_fwd_f64.argtypes = [P, P, P, P, P, I64, I64, I32, I32, I32, I32, I32, I32,
                                        P, P, I64, F64, F64, P, P, P]
    L.orc_rasterize_fwd_f64.restype = I32
    L.orc_rasterize_bwd.argtypes = [P, P, P, P, P, P, I64, I64, I32, I32, I32, I32, I32, I32,
                                    P, P, I64, F32, P, P, P, P, P, I64, P, P, P, P, P, P, P,
                                    F32, P, P, I32, P, P, P]
    L.orc_rasterize_bwd.restype = I32
    L.orc_bin_splats.argtypes = [P, P, I32, P, I64, I64, I32, I32, I32, I64, P, P]
    L.orc_bin_splats.restype = I64
    L.orc_project.argtypes = [P, P, P, P, I64, I64, I32, I32, F32, F32, F32, F32, I32, P, P,
                              P, P, P]
    L.orc_project.restype = I32
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ct.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def tile_bits(tile_width: int, tile_height: int) -> int:
    return int(lib().orc_tile_bits(tile_width, tile_height))


def bounds(means2d, radii, tile_size, tile_width, tile_height):
    """Tile rect (x0, y0, x1, y1) per splat, shape (C, N, 4) int32."""
    means2d = _c(means2d, np.float32)
    radii = _c(radii, np.float32)
    C, N = means2d.shape[:2]
    out = np.empty((C, N, 4), np.int32)
    lib().orc_bounds(_ptr(means2d), _ptr(radii), int(radii.ndim == 3), C, N, tile_size,
                     tile_width, tile_height, _ptr(out))
    return out


def isect_tiles(means2d, radii, depths, tile_size, tile_width, tile_height, sort=True,
                sort_impl="stable"):
    """(tiles_per_gauss (C,N) int32, keys (I,) uint64, flatten_ids (I,) int32)."""
    means2d = _c(means2d, np.float32)
    radii = _c(radii, np.float32)
    depths = _c(depths, np.float32)
    C, N = means2d.shape[:2]
    ell = int(radii.ndim == 3)
    tpg = np.empty((C, N), np.int32)
    total = lib().orc_isect_count(_ptr(means2d), _ptr(radii), ell, C, N, tile_size, tile_width,
                                  tile_height, _ptr(tpg))
    keys = np.empty(total, np.uint64)
    ids = np.empty(total, np.int32)
    w = lib().orc_isect_emit(_ptr(means2d), _ptr(radii), ell, _ptr(depths), C, N, tile_size,
                             tile_width, tile_height, _ptr(keys), _ptr(ids), total)
    assert w == total
    if sort and total > 1:
        sort_pairs(keys, ids, impl=sort_impl)
    return tpg, keys, ids


def sort_pairs(keys, ids, impl="stable"):
    """Sorts (keys uint64, ids int32) in place, stable, ascending by key."""
    assert keys.dtype == np.uint64 and ids.dtype == np.int32
    assert keys.flags.c_contiguous and ids.flags.c_contiguous
    if impl == "stable":
        lib().orc_sort_stable(_ptr(keys), _ptr(ids), keys.size)
    elif impl == "lsd":
        if lib().orc_sort_lsd(_ptr(keys), _ptr(ids), keys.size) != 0:
            raise MemoryError("oracle radix sort could not allocate")
    else:
        raise ValueError(impl)


class KeyOutOfGrid(ValueError):
    pass


def tile_offsets(keys, C, tile_width, tile_height):
    keys = _c(keys, np.uint64)
    out = np.empty((C, tile_height, tile_width), np.int32)
    rc = lib().orc_tile_offsets(_ptr(keys), keys.size, C, tile_width, tile_height, _ptr(out))
    if rc == 3:
        raise KeyOutOfGrid("intersection key is outside the tile grid")
    return out


def rasterize_fwd(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                  tile_size, offsets, flatten_ids, alpha_cutoff, transmittance_threshold,
                  pixels=None, tie_rel=0.0, tie_rel_T=None, out=None, omp=False,
                  max_steps=0):
    """Forward compositing.  Returns dict(render_colors (C,H,W,ch),
    render_alphas (C,H,W,1), last_ids (C,H,W), stats [evaluated, composited,
    near-tie pixels], near_tie (C,H,W) uint8 (near-threshold decisions per
    pixel), tie_splats (C,N), comp_hash (C,H,W) uint64 (FNV-1a hash of the
    composited list positions, in order))."""
    means2d = _c(means2d, np.float32)
    conics = _c(conics, np.float32)
    colors = _c(colors, np.float32)
    opacities = _c(opacities, np.float32)
    backgrounds = _c(backgrounds, np.float32)
    masks = _c(masks, np.int32)
    offsets = _c(offsets, np.int32)
    flatten_ids = _c(flatten_ids, np.int32)
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    TH, TW = offsets.shape[1], offsets.shape[2]
    if out is None:
        out = dict(render_colors=np.zeros((C, height, width, ch), np.float32),
                   render_alphas=np.zeros((C, height, width, 1), np.float32),
                   last_ids=np.full((C, height, width), -2, np.int32),
                   near_tie=np.zeros((C, height, width), np.uint8))
    out["tie_splats"] = np.zeros((C, N), np.uint8)
    if "comp_hash" not in out:
        out["comp_hash"] = np.zeros((C, height, width), np.uint64)
    stats = np.zeros(3, np.int64)
    if max_steps > 0:
        out["step_pos"] = np.full((max_steps, C, height, width), -1, np.int32)
        out["step_T"] = np.zeros((max_steps, C, height, width), np.float32)
        out["step_count"] = np.zeros((C, height, width), np.int32)
    px = None if pixels is None else _c(pixels, np.int64)
    rc = lib(omp).orc_rasterize_fwd(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, TW, TH, _ptr(offsets),
        _ptr(flatten_ids), flatten_ids.size, float(alpha_cutoff), float(transmittance_threshold),
        _ptr(px), 0 if px is None else px.size, _ptr(out["render_colors"]),
        _ptr(out["render_alphas"]), _ptr(out["last_ids"]), _ptr(stats), _ptr(out["near_tie"]),
        float(tie_rel), float(tie_rel if tie_rel_T is None else tie_rel_T),
        _ptr(out["tie_splats"]), _ptr(out["comp_hash"]), int(max_steps),
        _ptr(out.get("step_pos")), _ptr(out.get("step_T")), _ptr(out.get("step_count")))
    if rc != 0:
        raise ValueError("oracle forward: bad arguments")
    out["stats"] = stats
    return out


def rasterize_fwd_f64(means2d, conics, colors, opacities, backgrounds, width, height, tile_size,
                      offsets, flatten_ids, alpha_cutoff, transmittance_threshold):
    """Double-precision forward (finite-difference twin).  Returns
    (render_colors (C,H,W,ch), render_alphas (C,H,W), margins[3])."""
    d = lambda a: _c(a, np.float64)
    means2d, conics, colors, opacities = d(means2d), d(conics), d(colors), d(opacities)
    backgrounds = d(backgrounds)
    offsets = _c(offsets, np.int32)
    flatten_ids = _c(flatten_ids, np.int32)
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    TH, TW = offsets.shape[1], offsets.shape[2]
    rgb = np.zeros((C, height, width, ch), np.float64)
    alpha = np.zeros((C, height, width), np.float64)
    margins = np.zeros(3, np.float64)
    rc = lib().orc_rasterize_fwd_f64(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds), C, N, ch,
        width, height, tile_size, TW, TH, _ptr(offsets), _ptr(flatten_ids), flatten_ids.size,
        float(alpha_cutoff), float(transmittance_threshold), _ptr(rgb), _ptr(alpha),
        _ptr(margins))
    if rc != 0:
        raise ValueError("oracle f64 forward: bad arguments")
    return rgb, alpha, margins


def rasterize_bwd(means2d, conics, colors, opacities, backgrounds, masks, width, height,
                  tile_size, offsets, flatten_ids, alpha_cutoff, render_alphas, last_ids,
                  grad_render_colors, grad_render_alphas, want_grad_backgrounds=None,
                  absgrad=False, pixels=None, tie_rel=0.0, magnitudes=False, omp=False,
                  steps=None):
    """Backward.  Returns dict(grad_means2d, grad_conics, grad_colors,
    grad_opacities, grad_backgrounds (or None), grad_means2d_abs (or None),
    near_tie (C,H,W) uint8, and with magnitudes=True mag_* arrays: per
    gradient element the sum of |per-pair term|).  steps: the forward's step
    records (step_pos, step_T, step_count) from rasterize_fwd(max_steps=K);
    pixels they hold entirely read T before each pair instead of dividing."""
    means2d = _c(means2d, np.float32)
    conics = _c(conics, np.float32)
    colors = _c(colors, np.float32)
    opacities = _c(opacities, np.float32)
    backgrounds = _c(backgrounds, np.float32)
    masks = _c(masks, np.int32)
    offsets = _c(offsets, np.int32)
    flatten_ids = _c(flatten_ids, np.int32)
    render_alphas = _c(render_alphas, np.float32)
    last_ids = _c(last_ids, np.int32)
    grad_render_colors = _c(grad_render_colors, np.float32)
    grad_render_alphas = _c(grad_render_alphas, np.float32)
    C, N = means2d.shape[:2]
    ch = colors.shape[-1]
    TH, TW = offsets.shape[1], offsets.shape[2]
    if want_grad_backgrounds is None:
        want_grad_backgrounds = backgrounds is not None
    out = dict(grad_means2d=np.empty((C, N, 2), np.float32),
               grad_conics=np.empty((C, N, 3), np.float32),
               grad_colors=np.empty((C, N, ch), np.float32),
               grad_opacities=np.empty((C, N), np.float32),
               grad_backgrounds=np.empty((C, ch), np.float32) if want_grad_backgrounds else None,
               grad_means2d_abs=np.empty((C, N, 2), np.float32) if absgrad else None,
               near_tie=np.zeros((C, height, width), np.uint8),
               tie_splats=np.zeros((C, N), np.uint8))
    px = None if pixels is None else _c(pixels, np.int64)
    mags = np.zeros((6 + ch) * C * N, np.float64) if magnitudes else None
    if steps is not None:
        st_pos, st_T, st_cnt = (_c(steps[0], np.int32), _c(steps[1], np.float32),
                                _c(steps[2], np.int32))
        K = st_pos.shape[0]
    else:
        st_pos = st_T = st_cnt = None
        K = 0
    rc = lib(omp).orc_rasterize_bwd(
        _ptr(means2d), _ptr(conics), _ptr(colors), _ptr(opacities), _ptr(backgrounds),
        _ptr(masks), C, N, ch, width, height, tile_size, TW, TH, _ptr(offsets),
        _ptr(flatten_ids), flatten_ids.size, float(alpha_cutoff), _ptr(render_alphas),
        _ptr(last_ids), _ptr(grad_render_colors), _ptr(grad_render_alphas), _ptr(px),
        0 if px is None else px.size, _ptr(out["grad_means2d"]), _ptr(out["grad_conics"]),
        _ptr(out["grad_colors"]), _ptr(out["grad_opacities"]), _ptr(out["grad_backgrounds"]),
        _ptr(out["grad_means2d_abs"]), _ptr(out["near_tie"]), float(tie_rel), _ptr(mags),
        _ptr(out["tie_splats"]), K, _ptr(st_pos), _ptr(st_T), _ptr(st_cnt))
    if rc != 0:
        raise ValueError("oracle backward: bad arguments")
    if magnitudes:
        CN = C * N
        out["mag_means2d"] = mags[:2 * CN].reshape(C, N, 2)
        out["mag_conics"] = mags[2 * CN:5 * CN].reshape(C, N, 3)
        out["mag_colors"] = mags[5 * CN:(5 + ch) * CN].reshape(C, N, ch)
        out["mag_opacities"] = mags[(5 + ch) * CN:].reshape(C, N)
    return out


def render(scene, sort=True, pixels=None, tie_rel=0.0, tie_rel_T=None):
    """Whole forward path on a scenes.Scene-like object: isect, sort,
    offsets, forward.  Returns (isect dict, forward dict)."""
    tpg, keys, ids = isect_tiles(scene.means2d, scene.radii, scene.depths, scene.tile_size,
                                 scene.tile_width, scene.tile_height, sort=sort)
    offsets = tile_offsets(keys, scene.C, scene.tile_width, scene.tile_height)
    fwd = rasterize_fwd(scene.means2d, scene.conics, scene.colors, scene.opacities,
                        scene.backgrounds, None, scene.width, scene.height, scene.tile_size,
                        offsets, ids, scene.alpha_cutoff, scene.transmittance_threshold,
                        pixels=pixels, tie_rel=tie_rel, tie_rel_T=tie_rel_T)
    return dict(tiles_per_gauss=tpg, keys=keys, flatten_ids=ids, offsets=offsets), fwd


def bin_splats(means2d, radii, depths, tile_size, tile_width, tile_height, capacity):
    """Fixed-capacity bin lists: (bins int32 (C, TH, TW, M) with -1 after each
    bin's splats, counts int32 (C, TH, TW), the largest count)."""
    means2d = _c(means2d, np.float32)
    radii = _c(radii, np.float32)
    depths = _c(depths, np.float32)
    C, N = means2d.shape[:2]
    bins = np.empty((C, tile_height, tile_width, capacity), np.int32)
    counts = np.empty((C, tile_height, tile_width), np.int32)
    largest = lib().orc_bin_splats(_ptr(means2d), _ptr(radii), int(radii.ndim == 3),
                                   _ptr(depths), C, N, tile_size, tile_width, tile_height,
                                   capacity, _ptr(bins), _ptr(counts))
    return bins, counts, int(largest)


def project(means, covars, viewmats, intrinsics, width, height, eps2d=0.3, near_plane=0.01,
            far_plane=1e10, radius_clip=0.0, compensation=False, orthographic=False):
    """EWA projection (project.cpp).  means (N,3), covars (N,3,3), viewmats
    (C,4,4), intrinsics (C,3,3).  Returns dict(radii int32 (C,N,2), means2d
    (C,N,2), depths (C,N), conics (C,N,3), compensations (C,N) or None)."""
    means = _c(means, np.float32)
    covars = _c(covars, np.float32)
    viewmats = _c(viewmats, np.float32)
    intrinsics = _c(intrinsics, np.float32)
    N = means.shape[0]
    C = viewmats.shape[0]
    out = dict(radii=np.empty((C, N, 2), np.int32), means2d=np.empty((C, N, 2), np.float32),
               depths=np.empty((C, N), np.float32), conics=np.empty((C, N, 3), np.float32),
               compensations=np.empty((C, N), np.float32) if compensation else None)
    rc = lib().orc_project(_ptr(means), _ptr(covars), _ptr(viewmats), _ptr(intrinsics), C, N,
                           int(width), int(height), float(eps2d), float(near_plane),
                           float(far_plane), float(radius_clip), int(bool(orthographic)),
                           _ptr(out["radii"]), _ptr(out["means2d"]), _ptr(out["depths"]),
                           _ptr(out["conics"]), _ptr(out["compensations"]))
    if rc:
        raise ValueError("orc_project: bad sizes")
    return out
