"""Pins of the oracle's tile bounds, counts and key emission against what the
gsplat listing fixes (gsplat 1.0.0, intersections.c: gs_tile_bits, gs_bounds,
gs_isect_tiles) -- hand-derived tables and an independent brute force."""

import math

import numpy as np
import pytest

import oracle
from conftest import read_golden
from tile_gaussian_splat_gb300 import scenes


@pytest.mark.parametrize("tw,th,bits", [
    (1, 1, 0), (2, 1, 1), (3, 3, 4), (4, 4, 4), (5, 3, 4), (64, 64, 12),
    (120, 68, 13), (240, 135, 15), (256, 128, 15), (257, 128, 16), (1, 0, 0),
])
def test_tile_bits_closed_form(tw, th, bits):
    # fewest b with 2^b >= tw*th: ceil(log2(tw*th)), 0 for a grid of <= 1 tile
    n = tw * th
    assert (0 if n <= 1 else math.ceil(math.log2(n))) == bits
    assert oracle.tile_bits(tw, th) == bits


def test_bounds_golden_table():
    rows = read_golden("bounds_cases.txt")
    assert len(rows) >= 14
    means = np.array([[float(r[0][0]), float(r[0][1])] for r in rows], np.float32)[None]
    radii = np.array([[float(r[0][2]), float(r[0][3])] for r in rows], np.float32)[None]
    expect = np.array([[int(v) for v in r[1][:4]] for r in rows], np.int32)
    counts = np.array([int(r[1][4]) for r in rows], np.int32)
    rect = oracle.bounds(means, radii, 16, 4, 4)[0]
    np.testing.assert_array_equal(rect, expect)
    tpg, keys, ids = oracle.isect_tiles(means, radii, np.ones_like(means[..., 0]), 16, 4, 4)
    np.testing.assert_array_equal(tpg[0], counts)
    assert keys.size == counts.sum()


def _covered_brute(m, r, ts, ntiles):
    """Tiles t with [t*ts, (t+1)*ts) meeting the open interval (m - r, m + r).
    Exact in Python floats for the quarter-pixel inputs used below."""
    if r <= 0:
        return []
    return [t for t in range(ntiles) if (t + 1) * ts > m - r and t * ts < m + r]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("elliptical", [False, True])
def test_isect_matches_interval_overlap_brute_force(seed, elliptical):
    # Quarter-pixel means and radii: (m +- r) / 16 is exact in float32, so the
    # floor/ceil rect must equal the exact interval-overlap tile set.
    rng = np.random.default_rng(seed)
    C, N, W, H, ts = 2, 120, 80, 48, 16  # ragged grid: TW=5, TH=3
    TW, TH = 5, 3
    means = rng.integers(-160, 4 * W + 160, (C, N, 2)).astype(np.float32) / 4
    if elliptical:
        radii = rng.integers(-4, 120, (C, N, 2)).astype(np.float32) / 4
    else:
        radii = rng.integers(-4, 120, (C, N)).astype(np.float32) / 4
    depths = rng.uniform(0.5, 9.0, (C, N)).astype(np.float32)
    depths[0, :10] = depths[0, 10]  # equal depths: ties broken by splat index
    tpg, keys, ids = oracle.isect_tiles(means, radii, depths, ts, TW, TH, sort=False)
    tb = oracle.tile_bits(TW, TH)
    exp_keys, exp_ids, exp_tpg = [], [], np.zeros((C, N), np.int32)
    for c in range(C):
        for n in range(N):
            mx, my = float(means[c, n, 0]), float(means[c, n, 1])
            rx = float(radii[c, n, 0] if elliptical else radii[c, n])
            ry = float(radii[c, n, 1] if elliptical else radii[c, n])
            if rx <= 0 or ry <= 0:
                continue
            xs = _covered_brute(mx, rx, ts, TW)
            ys = _covered_brute(my, ry, ts, TH)
            exp_tpg[c, n] = len(xs) * len(ys)
            dbits = int(depths[c, n:n + 1].view(np.uint32)[0])
            for ty in ys:
                for tx in xs:
                    upper = (c << tb) | (ty * TW + tx)
                    exp_keys.append((upper << 32) | dbits)
                    exp_ids.append(c * N + n)
    np.testing.assert_array_equal(tpg, exp_tpg)
    np.testing.assert_array_equal(keys, np.array(exp_keys, np.uint64))
    np.testing.assert_array_equal(ids, np.array(exp_ids, np.int32))
    # sorted: ascending by key, equal keys in emission order
    _, sk, si = oracle.isect_tiles(means, radii, depths, ts, TW, TH, sort=True)
    order = sorted(range(len(exp_keys)), key=lambda k: (exp_keys[k], k))
    np.testing.assert_array_equal(sk, np.array(exp_keys, np.uint64)[order])
    np.testing.assert_array_equal(si, np.array(exp_ids, np.int32)[order])


def test_key_layout_fields():
    s = scenes.workload1()
    tpg, keys, ids = oracle.isect_tiles(s.means2d, s.radii, s.depths, 16, 4, 4, sort=False)
    tb = oracle.tile_bits(4, 4)
    assert tb == 4
    upper = keys >> np.uint64(32)
    tile = upper & np.uint64((1 << tb) - 1)
    cam = upper >> np.uint64(tb)
    assert (cam == 0).all() and (tile < 16).all()
    low = (keys & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    np.testing.assert_array_equal(low, s.depths.reshape(-1).view(np.uint32)[ids])
    # ids appear in non-decreasing splat order with tpg[i] copies each
    np.testing.assert_array_equal(ids, np.repeat(np.arange(256, dtype=np.int32), tpg[0]))


def test_workload2_has_its_intended_scale():
    # 100k elliptical splats on a 1024^2 image with 10 % of means past each
    # border: about 0.63 M intersections, about 73 % of splats on screen
    s = scenes.workload2()
    tpg, keys, ids = oracle.isect_tiles(s.means2d, s.radii, s.depths, 16, 64, 64, sort=False)
    assert 600_000 < keys.size < 700_000
    assert 0.70 < (tpg > 0).mean() < 0.77
