"""Pins of the oracle's forward compositing and backward against what the
pages and the mathematics fix: a hand-computed composite, a closed-form
single splat, a bit-exact tile-filtered brute force, an untiled brute force,
monotone transmittance, the termination and mask readings, central finite
differences of a double-precision forward, and two exact adjoint identities.

Sources: gsplat 1.0.0, data/ext/gsplat_native/raster_backward.c
(gs_raster_backward_pixel: pixel centre, quadratic form, alpha clamp and
skip, valid-pair test and gradient recurrences) and rlx-metal 0.2.9,
src/splat_training.rs (alpha_cutoff 1/255, transmittance_threshold)."""

import ctypes
import ctypes.util

import numpy as np
import pytest

import oracle
from conftest import read_golden
from tile_gaussian_splat_gb300 import scenes

CUT = np.float32(1.0 / 255.0)
THR = np.float32(1e-4)


def _setup(s):
    iso = {}
    iso["tpg"], iso["keys"], iso["ids"] = oracle.isect_tiles(
        s.means2d, s.radii, s.depths, s.tile_size, s.tile_width, s.tile_height)
    iso["offsets"] = oracle.tile_offsets(iso["keys"], s.C, s.tile_width, s.tile_height)
    return iso


def _fwd(s, iso, masks=None, ids=None, tie_rel=0.0, cut=None, thr=None, tie_rel_T=None):
    return oracle.rasterize_fwd(
        s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, masks, s.width, s.height,
        s.tile_size, iso["offsets"], iso["ids"] if ids is None else ids,
        s.alpha_cutoff if cut is None else cut,
        s.transmittance_threshold if thr is None else thr, tie_rel=tie_rel, tie_rel_T=tie_rel_T)


def _scene(means, conics, colors, opac, depths, radii, W, H, bg=None):
    f = lambda a: np.ascontiguousarray(np.asarray(a, np.float32)[None])
    return scenes.Scene(name="hand", C=1, N=len(opac), width=W, height=H, tile_size=16,
                        means2d=f(means), radii=f(radii), depths=f(depths), conics=f(conics),
                        colors=f(colors), opacities=f(opac),
                        backgrounds=None if bg is None else f(bg))


# ---------------------------------------------------------------- forward


def test_two_splats_golden():
    (x, y), (r, g, b, a, last) = [[int(v) for v in row[0]] for row in read_golden(
        "two_splats.txt")][0], [float(v) for v in read_golden("two_splats.txt")[0][1]]
    s = _scene([[7.5, 7.5], [7.5, 7.5]], [[1, 0, 1], [1, 0, 1]], [[1, 0, 0], [0, 1, 0]],
               [0.5, 0.5], [1.0, 2.0], [3.0, 3.0], 16, 16, bg=[0, 0, 1])
    out = _fwd(s, _setup(s))
    assert out["render_colors"][0, y, x].tolist() == [r, g, b]
    assert out["render_alphas"][0, y, x, 0] == a
    assert out["last_ids"][0, y, x] == int(last)


def test_single_splat_closed_form():
    m, q, o, col, bg = (23.3, 17.9), (0.11, 0.03, 0.07), 0.8, (0.2, 0.5, 0.9), (0.3, 0.1, 0.6)
    s = _scene([m], [q], [col], [o], [4.0], [40.0], 48, 48, bg=bg)
    iso = _setup(s)
    out = _fwd(s, iso)
    ys, xs = np.mgrid[0:48, 0:48]
    dx, dy = m[0] - (xs + 0.5), m[1] - (ys + 0.5)
    sig = 0.5 * (q[0] * dx * dx + q[2] * dy * dy) + q[1] * dx * dy
    al = np.minimum(0.99, o * np.exp(-sig))
    al = np.where(al >= 1 / 255, al, 0.0)
    rgb = al[..., None] * np.array(col) + (1 - al[..., None]) * np.array(bg)
    np.testing.assert_allclose(out["render_alphas"][0, ..., 0], al, atol=1e-6, rtol=0)
    np.testing.assert_allclose(out["render_colors"][0], rgb, atol=1e-6, rtol=0)
    # the one splat is entry `start` of every tile's list (last_id is a list position)
    start = iso["offsets"][0][ys // 16, xs // 16]
    np.testing.assert_array_equal(out["last_ids"][0], np.where(al > 0, start, -1))


_libm = ctypes.CDLL(ctypes.util.find_library("m"))
_libm.expf.restype = ctypes.c_float
_libm.expf.argtypes = [ctypes.c_float]


def _tile_filtered_brute(s):
    """Per pixel: every splat whose tile rect (interval overlap with the tile)
    holds the pixel's tile, in (depth bits, splat index) order, composited in
    float32 scalars with libm expf -- the same operations in the same order,
    so the image must be bit-identical to the oracle's."""
    f = np.float32
    C, N, W, H, ts = s.C, s.N, s.width, s.height, s.tile_size
    rects = oracle.bounds(s.means2d, s.radii, ts, s.tile_width, s.tile_height)
    rgb = np.zeros((C, H, W, 3), np.float32)
    alpha = np.zeros((C, H, W), np.float32)
    last_rank = np.full((C, H, W), -1, np.int64)
    dbits = s.depths.view(np.uint32)
    for c in range(C):
        order = sorted(range(N), key=lambda n: (int(dbits[c, n]), n))
        for ty in range(s.tile_height):
            for tx in range(s.tile_width):
                # splat n covers tile (tx, ty) iff the tile is inside its rect
                lst = [n for n in order if rects[c, n, 0] <= tx < rects[c, n, 2]
                       and rects[c, n, 1] <= ty < rects[c, n, 3]]
                for y in range(ty * ts, min(H, (ty + 1) * ts)):
                    for x in range(tx * ts, min(W, (tx + 1) * ts)):
                        T, acc, last = f(1), [f(0)] * 3, -1
                        px, py = f(x) + f(0.5), f(y) + f(0.5)
                        for rank, n in enumerate(lst):
                            dx = s.means2d[c, n, 0] - px
                            dy = s.means2d[c, n, 1] - py
                            a, b, cc = s.conics[c, n]
                            sg = f(0.5) * (a * dx * dx + cc * dy * dy) + b * dx * dy
                            if not sg >= 0:
                                continue
                            raw = s.opacities[c, n] * f(_libm.expf(f(-sg)))
                            al = f(0.99) if raw > f(0.99) else raw
                            if al < s.alpha_cutoff:
                                continue
                            w = T * al
                            acc = [acc[k] + w * s.colors[c, n, k] for k in range(3)]
                            T = T * (f(1) - al)
                            last = rank
                            if T < s.transmittance_threshold:
                                break
                        bg = s.backgrounds[c] if s.backgrounds is not None else np.zeros(3, f)
                        rgb[c, y, x] = [acc[k] + T * bg[k] for k in range(3)]
                        alpha[c, y, x] = f(1) - T
                        last_rank[c, y, x] = last
    return rgb, alpha, last_rank


@pytest.mark.parametrize("seed", [0, 1])
def test_tile_filtered_brute_force_bit_exact(seed):
    s = scenes.random_small(seed, C=2, N=14, W=40, H=36, sigma=(1.0, 6.0))  # ragged tiles
    iso = _setup(s)
    out = _fwd(s, iso)
    rgb, alpha, last_rank = _tile_filtered_brute(s)
    np.testing.assert_array_equal(out["render_colors"], rgb)
    np.testing.assert_array_equal(out["render_alphas"][..., 0], alpha)
    # last_id is a list position: convert to the rank inside the tile's list
    TW, TH = s.tile_width, s.tile_height
    ys, xs = np.mgrid[0:s.height, 0:s.width]
    for c in range(s.C):
        t = (c * TH + ys // 16) * TW + xs // 16
        start = iso["offsets"].reshape(-1)[t]
        li = out["last_ids"][c]
        np.testing.assert_array_equal(np.where(li >= 0, li - start, -1), last_rank[c])


def _untiled_brute(s):
    """Per pixel, every splat of the camera in depth order, no tiles (float64)."""
    C, N, W, H = s.C, s.N, s.width, s.height
    ys, xs = np.mgrid[0:H, 0:W]
    px, py = xs + 0.5, ys + 0.5
    rgb = np.zeros((C, H, W, 3))
    T = np.ones((C, H, W))
    for c in range(C):
        done = np.zeros((H, W), bool)
        order = sorted(range(N), key=lambda n: (int(s.depths.view(np.uint32)[c, n]), n))
        for n in order:
            dx, dy = float(s.means2d[c, n, 0]) - px, float(s.means2d[c, n, 1]) - py
            a, b, cc = (float(v) for v in s.conics[c, n])
            sg = 0.5 * (a * dx * dx + cc * dy * dy) + b * dx * dy
            al = np.minimum(0.99, float(s.opacities[c, n]) * np.exp(-sg))
            use = (sg >= 0) & (al >= float(s.alpha_cutoff)) & ~done
            w = np.where(use, T[c] * al, 0.0)
            rgb[c] += w[..., None] * s.colors[c, n].astype(np.float64)
            T[c] = np.where(use, T[c] * (1 - al), T[c])
            done |= use & (T[c] < float(s.transmittance_threshold))
        if s.backgrounds is not None:
            rgb[c] += T[c][..., None] * s.backgrounds[c].astype(np.float64)
    return rgb, 1 - T


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_untiled_brute_force_with_covering_radii(seed):
    # radius 3.5 sigma covers every pixel where alpha >= 1/255 can hold
    # (o exp(-s) >= 1/255 needs s <= ln(255 * 0.99) = 5.53, i.e. 3.33 sigma),
    # so tiling drops nothing and the tiled image equals the untiled one.
    s = scenes.random_small(seed, C=1, N=16, W=48, H=40, radius_scale=3.5)
    out = _fwd(s, _setup(s), tie_rel=1e-4)
    rgb, alpha = _untiled_brute(s)
    ok = out["near_tie"] == 0
    assert ok.mean() > 0.99
    np.testing.assert_allclose(out["render_colors"][ok], rgb[ok], atol=2e-6, rtol=0)
    np.testing.assert_allclose(out["render_alphas"][..., 0][ok], alpha[ok], atol=2e-6, rtol=0)


def test_untiled_brute_force_detects_tile_truncation():
    # with the workloads' 3 sigma radii some pixels lose a contribution that
    # passes the cutoff outside the rect: the comparison above can fail
    s = scenes.random_small(3, C=1, N=16, W=48, H=40, radius_scale=2.0)
    out = _fwd(s, _setup(s))
    rgb, _ = _untiled_brute(s)
    assert np.abs(out["render_colors"] - rgb).max() > 1e-3


def test_transmittance_monotone_along_list():
    s = scenes.random_small(7, C=1, N=24, W=16, H=16, sigma=(2.0, 8.0))  # one tile
    iso = _setup(s)
    L = iso["ids"].size
    prev = np.zeros((16, 16))
    for k in range(L + 1):
        iso_k = dict(offsets=np.zeros((1, 1, 1), np.int32), ids=iso["ids"][:k])
        a = _fwd(s, iso_k)["render_alphas"][0, ..., 0].astype(np.float64)
        assert (a >= prev).all() and (a < 1).all()
        prev = a


def test_termination_after_crossing_splat():
    # three opaque splats at the pixel centre: T = 1 -> 0.0099999905 -> 9.99998e-5 < 1e-4,
    # so the second is composited, becomes last_id, and the third is never reached
    q = [[1, 0, 1]] * 3
    s = _scene([[7.5, 7.5]] * 3, q, [[1, 0, 0], [0, 1, 0], [0, 0, 1]], [0.99] * 3,
               [1.0, 2.0, 3.0], [3.0] * 3, 16, 16)
    out = _fwd(s, _setup(s))
    f = np.float32
    T1 = f(1) - f(0.99)
    T2 = T1 * (f(1) - f(0.99))
    assert T2 < THR
    assert out["last_ids"][0, 7, 7] == 1
    assert out["render_alphas"][0, 7, 7, 0] == f(1) - T2
    assert out["render_colors"][0, 7, 7, 2] == 0.0
    # the same pair with a threshold just below T2 composites all three
    out2 = _fwd(s, _setup(s), thr=T2 * f(0.5))
    assert out2["last_ids"][0, 7, 7] == 2


def test_opaque_front_limit():
    s = _scene([[7.5, 7.5], [7.5, 7.5]], [[1, 0, 1]] * 2, [[1, 1, 1], [0, 0, 0]], [1.0, 1.0],
               [1.0, 2.0], [3.0, 3.0], 16, 16)
    out = _fwd(s, _setup(s))
    # raw alpha 1 is clamped to 0.99, so the front splat leaves T = 0.01
    np.testing.assert_allclose(out["render_alphas"][0, 7, 7, 0], 1 - 0.01 * 0.01, atol=1e-6)
    np.testing.assert_allclose(out["render_colors"][0, 7, 7], [0.99] * 3, atol=1e-6)


def test_masked_tile_gives_background():
    s = scenes.random_small(2, C=1, N=12, W=32, H=32)
    iso = _setup(s)
    masks = np.array([[[1, 0], [1, 1]]], np.int32)
    out = _fwd(s, iso, masks=masks)
    np.testing.assert_array_equal(out["render_colors"][0, 0:16, 16:32],
                                  np.broadcast_to(s.backgrounds[0], (16, 16, 3)))
    assert (out["render_alphas"][0, 0:16, 16:32] == 0).all()
    assert (out["last_ids"][0, 0:16, 16:32] == -1).all()
    ref = _fwd(s, iso)
    np.testing.assert_array_equal(out["render_colors"][0, 16:], ref["render_colors"][0, 16:])


def test_last_id_within_tile_range():
    s = scenes.workload1()
    iso = _setup(s)
    out = _fwd(s, iso)
    ys, xs = np.mgrid[0:64, 0:64]
    t = (ys // 16) * 4 + xs // 16
    off = iso["offsets"].reshape(-1)
    start, end = off[t], np.append(off[1:], iso["ids"].size)[t]
    li = out["last_ids"][0]
    assert ((li == -1) | ((li >= start) & (li < end))).all()
    assert ((out["render_alphas"][0, ..., 0] > 0) == (li >= 0)).all()


# --------------------------------------------------------------- backward


def _loss_f64(s, iso, g_rgb, g_a, **over):
    p = dict(means2d=s.means2d, conics=s.conics, colors=s.colors, opacities=s.opacities)
    p.update(over)
    rgb, alpha, margins = oracle.rasterize_fwd_f64(
        p["means2d"], p["conics"], p["colors"], p["opacities"], s.backgrounds, s.width,
        s.height, s.tile_size, iso["offsets"], iso["ids"], float(s.alpha_cutoff),
        float(s.transmittance_threshold))
    return float((rgb * g_rgb).sum() + (alpha * g_a[..., 0]).sum()), margins


def _bwd(s, iso, fwd, g_rgb, g_a, masks=None, absgrad=False):
    return oracle.rasterize_bwd(
        s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, masks, s.width, s.height,
        s.tile_size, iso["offsets"], iso["ids"], s.alpha_cutoff, fwd["render_alphas"],
        fwd["last_ids"], g_rgb, g_a, absgrad=absgrad)


def _fd_scene(seed, **kw):
    """A scene whose every pair stays >= 1e-3 (relative) away from the cutoff,
    the 0.99 clamp and the threshold, so the loss is smooth under the steps."""
    for k in range(200):
        s = scenes.random_small(seed * 1000 + k, **kw)
        iso = _setup(s)
        _, m = _loss_f64(s, iso, np.zeros((s.C, s.height, s.width, 3)),
                         np.zeros((s.C, s.height, s.width, 1)))
        if m.min() > 1e-3:
            return s, iso
    raise RuntimeError("no smooth scene found")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_backward_matches_finite_differences(seed):
    s, iso = _fd_scene(seed, C=1, N=10, W=32, H=32, sigma=(1.5, 5.0), opacity=(0.3, 0.95))
    rng = np.random.default_rng(seed)
    g_rgb = rng.standard_normal((1, 32, 32, 3)).astype(np.float32)
    g_a = rng.standard_normal((1, 32, 32, 1)).astype(np.float32)
    fwd = _fwd(s, iso)
    got = _bwd(s, iso, fwd, g_rgb, g_a)
    # steps small enough that no decision (cutoff, clamp, threshold) is
    # crossed inside +-h: the scene keeps every pair >= 1e-3 away from them
    checks = [("means2d", "grad_means2d", 1e-5), ("conics", "grad_conics", 1e-6),
              ("colors", "grad_colors", 1e-5), ("opacities", "grad_opacities", 1e-6)]
    for name, gname, h in checks:
        base = getattr(s, name).astype(np.float64)
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            hi, lo = base.copy(), base.copy()
            hi[idx] += h
            lo[idx] -= h
            Lp, _ = _loss_f64(s, iso, g_rgb, g_a, **{name: hi})
            Lm, _ = _loss_f64(s, iso, g_rgb, g_a, **{name: lo})
            fd[idx] = (Lp - Lm) / (2 * h)
        g = got[gname].astype(np.float64)
        scale = np.abs(fd).max()
        np.testing.assert_allclose(g, fd, rtol=1e-3, atol=1e-5 * scale, err_msg=gname)


def test_backward_clamp_and_termination_paths():
    # an opacity-0.995 splat under the 0.99 clamp (its raw alpha gradient is
    # zero where clamped) and a stack that drives T below the threshold
    s = _scene([[12.2, 11.7], [13.1, 12.4], [11.5, 13.3], [12.7, 12.9]],
               [[0.05, 0.01, 0.06], [0.08, -0.02, 0.05], [0.06, 0.0, 0.06], [0.04, 0.01, 0.05]],
               [[0.9, 0.1, 0.2], [0.2, 0.8, 0.3], [0.1, 0.3, 0.9], [0.5, 0.5, 0.5]],
               [0.995, 0.98, 0.97, 0.9], [1.0, 2.0, 3.0, 4.0], [20.0] * 4, 24, 24, bg=[0.2, 0.3, 0.4])
    iso = _setup(s)
    rng = np.random.default_rng(11)
    g_rgb = rng.standard_normal((1, 24, 24, 3)).astype(np.float32)
    g_a = rng.standard_normal((1, 24, 24, 1)).astype(np.float32)
    fwd = _fwd(s, iso)
    assert (fwd["last_ids"] >= 0).any()
    got = _bwd(s, iso, fwd, g_rgb, g_a)
    for name, gname, h in [("opacities", "grad_opacities", 1e-5), ("colors", "grad_colors", 1e-5),
                           ("means2d", "grad_means2d", 1e-4)]:
        base = getattr(s, name).astype(np.float64)
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            hi, lo = base.copy(), base.copy()
            hi[idx] += h
            lo[idx] -= h
            fd[idx] = (_loss_f64(s, iso, g_rgb, g_a, **{name: hi})[0]
                       - _loss_f64(s, iso, g_rgb, g_a, **{name: lo})[0]) / (2 * h)
        scale = np.abs(fd).max()
        # pixels that sit exactly on a threshold crossing make the loss
        # piecewise: compare with a looser relative bound here
        np.testing.assert_allclose(got[gname], fd, rtol=2e-2, atol=2e-3 * scale, err_msg=gname)


def test_color_adjoint_identity_and_background_closed_form():
    # L is linear in the colours: sum_j dL/dc_j . c_j = sum_p g . (rgb_p - T_p bg)
    # and dL/dbg = sum_p g T_p, with T_p = 1 - render_alpha_p
    s = scenes.random_small(9, C=2, N=30, W=48, H=32)
    iso = _setup(s)
    rng = np.random.default_rng(5)
    g_rgb = rng.standard_normal((2, 32, 48, 3)).astype(np.float32)
    g_a = rng.standard_normal((2, 32, 48, 1)).astype(np.float32)
    fwd = _fwd(s, iso)
    got = _bwd(s, iso, fwd, g_rgb, g_a, absgrad=True)
    T = 1.0 - fwd["render_alphas"].astype(np.float64)
    rgb = fwd["render_colors"].astype(np.float64)
    bg = s.backgrounds.astype(np.float64)[:, None, None, :]
    lhs = (got["grad_colors"].astype(np.float64) * s.colors).sum()
    rhs = (g_rgb * (rgb - T * bg)).sum()
    np.testing.assert_allclose(lhs, rhs, rtol=2e-5)
    np.testing.assert_allclose(got["grad_backgrounds"], (g_rgb * T).sum(axis=(1, 2)),
                               rtol=1e-5, atol=1e-4)
    assert (got["grad_means2d_abs"] >= np.abs(got["grad_means2d"]) * (1 - 1e-6)).all()


def test_backward_masked_tiles_only_background():
    s = scenes.random_small(4, C=1, N=12, W=32, H=32)
    iso = _setup(s)
    masks = np.zeros((1, 2, 2), np.int32)
    fwd = _fwd(s, iso, masks=masks)
    g_rgb = np.ones((1, 32, 32, 3), np.float32)
    g_a = np.ones((1, 32, 32, 1), np.float32)
    got = _bwd(s, iso, fwd, g_rgb, g_a, masks=masks)
    for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities"):
        assert (got[k] == 0).all()
    np.testing.assert_allclose(got["grad_backgrounds"], [[1024.0] * 3])


@pytest.mark.parametrize("seed", [0, 5])
def test_double_twin_matches_float_forward(seed):
    # the double-precision forward (used for finite differences) is the same
    # recurrence: away from decisions it agrees with the float forward to
    # float rounding, which pins it to everything the float forward is pinned to
    s = scenes.random_small(seed, C=2, N=20, W=48, H=32)
    iso = _setup(s)
    f32 = _fwd(s, iso, tie_rel=1e-3, tie_rel_T=1e-2)
    rgb, alpha, _ = oracle.rasterize_fwd_f64(
        s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, s.width, s.height,
        s.tile_size, iso["offsets"], iso["ids"], float(s.alpha_cutoff),
        float(s.transmittance_threshold))
    ok = f32["near_tie"] == 0
    assert ok.mean() > 0.9
    np.testing.assert_allclose(f32["render_colors"][ok], rgb[ok], atol=2e-6, rtol=0)
    np.testing.assert_allclose(f32["render_alphas"][..., 0][ok], alpha[ok], atol=2e-6, rtol=0)


# ------------------------------------------- cutoff and threshold readings


def test_cutoff_zero_takes_vanishing_pairs():
    # a splat whose alpha at the pixel is exactly 0 (s huge) is skipped under
    # the default cutoff but taken under a zero cutoff: its position becomes
    # the last id while the colour and T stay those of the front splat
    s = _scene([[7.5, 7.5], [7.5, 7.5]], [[1, 0, 1], [1e4, 0, 1e4]], [[1, 0, 0], [0, 1, 0]],
               [0.5, 0.5], [1.0, 2.0], [3.0, 3.0], 16, 16)
    iso = _setup(s)
    x, y = 12, 7  # centre (12.5, 7.5), dx = -5: s = 12.5 for the first, 1.25e5 for the second
    a = _fwd(s, iso, cut=np.float32(1.0 / 255.0))
    b = _fwd(s, iso, cut=np.float32(0.0))
    alpha0 = 0.5 * np.exp(-12.5)
    assert alpha0 < 1.0 / 255.0  # the front splat is itself below the default cutoff
    assert a["last_ids"][0, y, x] == -1
    assert b["last_ids"][0, y, x] == 1
    # render_alpha = 1 - T carries the float rounding of T = 1 - alpha0
    np.testing.assert_allclose(b["render_alphas"][0, y, x, 0], alpha0, atol=1.2e-7)
    np.testing.assert_allclose(b["render_colors"][0, y, x], [alpha0, 0, 0], rtol=1e-5)


def test_threshold_zero_never_stops_and_high_threshold_stops_at_first():
    # three opaque splats over the same pixel: T = 0.01^k after k of them.
    # Threshold 0: all three are composited (T never falls below 0); a
    # threshold above 0.01 stops after the first
    s = _scene([[7.5, 7.5]] * 3, [[1, 0, 1]] * 3, [[1, 0, 0], [0, 1, 0], [0, 0, 1]],
               [0.99, 0.99, 0.99], [1.0, 2.0, 3.0], [3.0, 3.0, 3.0], 16, 16)
    iso = _setup(s)
    x, y = 7, 7  # the centre pixel: s = 0, alpha = 0.99
    a = _fwd(s, iso, thr=np.float32(0.0))
    b = _fwd(s, iso, thr=np.float32(0.999))
    assert a["last_ids"][0, y, x] == 2
    np.testing.assert_allclose(a["render_alphas"][0, y, x, 0], 1 - 0.01 ** 3, rtol=1e-6)
    np.testing.assert_allclose(a["render_colors"][0, y, x], [0.99, 0.0099, 0.000099], rtol=1e-5)
    assert b["last_ids"][0, y, x] == 0
    np.testing.assert_allclose(b["render_colors"][0, y, x], [0.99, 0, 0], rtol=1e-6)


# ------------------------------------------------------------------- absgrad


def test_absgrad_four_pixels_golden():
    # one splat whose per-pixel mean-gradient terms change sign across the
    # pixels: absgrad is the sum of their absolute values, not |their sum|
    rows = read_golden("absgrad_four_pixels.txt")
    pixels = [[float(v) for v in r[0]] for r in rows if len(r) == 1]
    (gx, gy), (ax, ay) = [[float(v) for v in part] for part in rows[-1]]
    s = _scene([[8.0, 8.0]], [[0.25, 0.0, 0.25]], [[1.0, 0.0, 0.0]], [0.5], [1.0], [3.0],
               16, 16)
    iso = _setup(s)
    g_rgb = np.zeros((1, 16, 16, 3), np.float32)
    for x, y, g in pixels:
        g_rgb[0, int(y), int(x), 0] = g
    g_a = np.zeros((1, 16, 16, 1), np.float32)
    fwd = _fwd(s, iso)
    got = _bwd(s, iso, fwd, g_rgb, g_a, absgrad=True)
    np.testing.assert_allclose(got["grad_means2d"][0, 0], [gx, gy], rtol=1e-6)
    np.testing.assert_allclose(got["grad_means2d_abs"][0, 0], [ax, ay], rtol=1e-6)


@pytest.mark.parametrize("seed", [0, 3])
def test_absgrad_is_sum_of_per_pixel_finite_differences(seed):
    # absgrad of splat g = sum over pixels p of |dL_p/dmean_g|, where L_p is
    # pixel p's share of the loss (g_p . rgb_p + g_a,p alpha_p).  Each
    # per-pixel derivative is a central difference of the double-precision
    # forward: one pair of forward runs per (splat, axis) gives the whole
    # image, hence every pixel's difference at once
    s, iso = _fd_scene(seed, C=1, N=10, W=32, H=32, sigma=(1.5, 5.0), opacity=(0.3, 0.95))
    rng = np.random.default_rng(100 + seed)
    g_rgb = rng.standard_normal((1, 32, 32, 3)).astype(np.float32)
    g_a = rng.standard_normal((1, 32, 32, 1)).astype(np.float32)
    got = _bwd(s, iso, _fwd(s, iso), g_rgb, g_a, absgrad=True)

    def per_pixel_loss(means):
        rgb, alpha, _ = oracle.rasterize_fwd_f64(
            means, s.conics, s.colors, s.opacities, s.backgrounds, s.width, s.height,
            s.tile_size, iso["offsets"], iso["ids"], float(s.alpha_cutoff),
            float(s.transmittance_threshold))
        return (rgb * g_rgb).sum(axis=-1) + alpha * g_a[..., 0]

    h = 1e-5
    base = s.means2d.astype(np.float64)
    ref_abs = np.zeros_like(base)
    ref_sum = np.zeros_like(base)
    for n in range(s.N):
        for k in range(2):
            hi, lo = base.copy(), base.copy()
            hi[0, n, k] += h
            lo[0, n, k] -= h
            fd = (per_pixel_loss(hi) - per_pixel_loss(lo)) / (2 * h)
            ref_abs[0, n, k] = np.abs(fd).sum()
            ref_sum[0, n, k] = fd.sum()
    # the terms do change sign: |sum| is well below the sum of |terms|
    assert (np.abs(ref_sum) < 0.5 * ref_abs).any()
    scale = ref_abs.max()
    np.testing.assert_allclose(got["grad_means2d_abs"], ref_abs, rtol=1e-3, atol=1e-5 * scale)
    np.testing.assert_allclose(got["grad_means2d"], ref_sum, rtol=1e-3, atol=1e-5 * scale)


def test_many_channels_reduce_to_three_channel_runs():
    # channels are independent in the compositing and every gradient term is
    # a per-channel sum: a 300-channel scene whose colours repeat one
    # 3-channel scene 100 times renders that scene 100 times over, and its
    # colour gradients are the 3-channel ones (with the upstream gradient
    # repeated, the opacity and geometry gradients scale by 100)
    s3 = scenes.random_small(12, C=1, N=40, W=48, H=32)
    iso = _setup(s3)
    rng = np.random.default_rng(7)
    g3 = rng.standard_normal((1, 32, 48, 3)).astype(np.float32)
    ga = np.zeros((1, 32, 48, 1), np.float32)
    f3 = _fwd(s3, iso)
    b3 = _bwd(s3, iso, f3, g3, ga)
    s300 = scenes.random_small(12, C=1, N=40, W=48, H=32)
    s300.colors = np.ascontiguousarray(np.tile(s3.colors, (1, 1, 100)))
    s300.backgrounds = np.ascontiguousarray(np.tile(s3.backgrounds, (1, 100)))
    f300 = _fwd(s300, iso)
    assert f300["render_colors"].shape[-1] == 300
    np.testing.assert_array_equal(f300["render_colors"],
                                  np.tile(f3["render_colors"], (1, 1, 1, 100)))
    np.testing.assert_array_equal(f300["last_ids"], f3["last_ids"])
    b300 = _bwd(s300, iso, f300, np.tile(g3, (1, 1, 1, 100)), ga)
    np.testing.assert_allclose(b300["grad_colors"], np.tile(b3["grad_colors"], (1, 1, 100)),
                               rtol=1e-6, atol=1e-7)
    for k in ("grad_opacities", "grad_means2d", "grad_conics"):
        np.testing.assert_allclose(b300[k], 100 * b3[k].astype(np.float64), rtol=2e-4,
                                   atol=1e-4 * np.abs(100 * b3[k]).max(), err_msg=k)


def _fnv(positions):
    h = 14695981039346656037
    for j in positions:
        h = ((h ^ j) * 1099511628211) % (1 << 64)
    return h


def test_composite_hash_lists_the_composited_positions():
    # the two stacked splats of the golden case: the centre pixel composites
    # list positions 0 and 1; a pixel only the wider back splat reaches
    # composites position 1 alone; a pixel beyond both composites nothing
    s = _scene([[7.5, 7.5], [7.5, 7.5]], [[1, 0, 1], [0.02, 0, 0.02]], [[1, 0, 0], [0, 1, 0]],
               [0.5, 0.5], [1.0, 2.0], [3.0, 12.0], 16, 16)
    out = _fwd(s, _setup(s))
    assert out["comp_hash"][0, 7, 7] == _fnv([0, 1])
    x = 12  # dx = -5: s = 12.5 for the front splat (alpha 2e-6), 0.25 for the back one
    assert out["last_ids"][0, 7, x] == 1
    assert out["comp_hash"][0, 7, x] == _fnv([1])
    s.means2d[:] = 40.0  # nothing reaches any pixel of the tile it still lists
    out = _fwd(s, _setup(s))
    assert (out["comp_hash"] == _fnv([])).all()


# ------------------------------------------------------------ step trace


def test_step_records_golden():
    # the golden two-splat pixel composites list positions 0 then 1, with T
    # 1 before the front splat and 0.5 before the back one (exact)
    s = _scene([[7.5, 7.5], [7.5, 7.5]], [[1, 0, 1], [1, 0, 1]], [[1, 0, 0], [0, 1, 0]],
               [0.5, 0.5], [1.0, 2.0], [3.0, 3.0], 16, 16, bg=[0, 0, 1])
    iso = _setup(s)
    out = oracle.rasterize_fwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, None,
                               16, 16, 16, iso["offsets"], iso["ids"], CUT, THR, max_steps=4)
    assert out["step_count"][0, 7, 7] == 2
    assert out["step_pos"][:2, 0, 7, 7].tolist() == [0, 1]
    assert out["step_T"][:2, 0, 7, 7].tolist() == [1.0, 0.5]
    assert (out["step_pos"][2:, 0, 7, 7] == -1).all()  # records past the count: untouched


def _fwd_steps(s, iso, K):
    return oracle.rasterize_fwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, None,
                                s.width, s.height, s.tile_size, iso["offsets"], iso["ids"],
                                s.alpha_cutoff, s.transmittance_threshold, max_steps=K)


@pytest.mark.parametrize("seed", [0, 1])
def test_step_backward_matches_finite_differences(seed):
    # the backward over the step records (T before each pair read, not
    # recovered) against central differences of the double forward
    s, iso = _fd_scene(seed, C=1, N=10, W=32, H=32, sigma=(1.5, 5.0), opacity=(0.3, 0.95))
    rng = np.random.default_rng(seed + 20)
    g_rgb = rng.standard_normal((1, 32, 32, 3)).astype(np.float32)
    g_a = rng.standard_normal((1, 32, 32, 1)).astype(np.float32)
    fwd = _fwd_steps(s, iso, 64)
    assert fwd["step_count"].max() <= 64
    got = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, None,
                               32, 32, 16, iso["offsets"], iso["ids"], s.alpha_cutoff,
                               fwd["render_alphas"], fwd["last_ids"], g_rgb, g_a,
                               steps=(fwd["step_pos"], fwd["step_T"], fwd["step_count"]))
    for name, gname, h in [("means2d", "grad_means2d", 1e-5), ("opacities", "grad_opacities", 1e-6),
                           ("colors", "grad_colors", 1e-5), ("conics", "grad_conics", 1e-6)]:
        base = getattr(s, name).astype(np.float64)
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            hi, lo = base.copy(), base.copy()
            hi[idx] += h
            lo[idx] -= h
            fd[idx] = (_loss_f64(s, iso, g_rgb, g_a, **{name: hi})[0]
                       - _loss_f64(s, iso, g_rgb, g_a, **{name: lo})[0]) / (2 * h)
        np.testing.assert_allclose(got[gname], fd, rtol=1e-3, atol=1e-5 * np.abs(fd).max(),
                                   err_msg=gname)


def test_step_backward_equals_walk_where_recovery_is_exact_and_falls_back():
    # with every opacity <= 0.5, T stays >= 0.5^k well away from 0 and the
    # division recovery loses nothing measurable: the two backwards agree to
    # float rounding.  With max_steps = 1 every pixel with two or more pairs
    # takes the walk: the result is the walk's, bit for bit, for those pixels
    s = scenes.random_small(31, C=2, N=40, W=48, H=32, opacity=(0.05, 0.5))
    iso = _setup(s)
    rng = np.random.default_rng(3)
    g_rgb = rng.standard_normal((2, 32, 48, 3)).astype(np.float32)
    g_a = rng.standard_normal((2, 32, 48, 1)).astype(np.float32)
    walk = None
    for K in (64, 1):
        fwd = _fwd_steps(s, iso, K)
        args = (s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, None, 48, 32, 16,
                iso["offsets"], iso["ids"], s.alpha_cutoff, fwd["render_alphas"],
                fwd["last_ids"], g_rgb, g_a)
        walk = oracle.rasterize_bwd(*args)
        st = oracle.rasterize_bwd(*args, steps=(fwd["step_pos"], fwd["step_T"],
                                                fwd["step_count"]))
        for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities",
                  "grad_backgrounds"):
            if K == 64:
                np.testing.assert_allclose(st[k], walk[k], rtol=2e-5,
                                           atol=2e-6 * np.abs(walk[k]).max(), err_msg=k)
    # K = 1: pixels with one pair read its T (= 1, exact either way), the rest walk
    multi = (fwd["step_count"] > 1)
    assert multi.any()
    for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities"):
        np.testing.assert_allclose(st[k], walk[k], rtol=1e-6, atol=1e-9, err_msg=k)
