"""Pins of the oracle's fixed-capacity bin lists (the bin_faces layout of the
pytorch3d fine rasterizer, rasterize_meshes.cu, RasterizeMeshesFineCudaKernel:
(N, BH, BW, M) int32 with a -1 sentinel) against the sorted-key path, a
different algorithm over the same intersections: a stable sort of all 64-bit
keys (gsplat 1.0.0, intersections.c, gs_radix_sort_without_gvl) followed by
the tile offsets (gs_offset_encode).  Each bin must be exactly its tile's
slice of the sorted flatten ids."""

import numpy as np
import pytest

import oracle
from tile_gaussian_splat_gb300 import scenes


def _sorted_lists(s):
    _, keys, ids = oracle.isect_tiles(s.means2d, s.radii, s.depths, s.tile_size, s.tile_width,
                                      s.tile_height)
    offs = oracle.tile_offsets(keys, s.C, s.tile_width, s.tile_height).reshape(-1)
    ends = np.append(offs[1:], ids.size)
    return [ids[o:e] for o, e in zip(offs, ends)]


def _scene(kind):
    if kind == "w1":
        return scenes.workload1()
    if kind == "cams":
        return scenes.random_small(3, C=3, N=800, W=90, H=70, sigma=(0.5, 12.0))
    if kind == "ties":
        # many equal and negative depths: order by raw depth bits, then index
        s = scenes.random_small(4, C=2, N=600, W=64, H=48, sigma=(1.0, 8.0))
        rng = np.random.default_rng(0)
        s.depths = rng.choice(np.array([1.5, 2.0, -0.5, 0.0, -0.0], np.float32),
                              s.depths.shape).astype(np.float32)
        return s
    raise KeyError(kind)


@pytest.mark.parametrize("kind", ["w1", "cams", "ties"])
def test_bins_equal_sorted_tile_slices(kind):
    s = _scene(kind)
    lists = _sorted_lists(s)
    M = max(len(v) for v in lists) + 3
    bins, counts, largest = oracle.bin_splats(s.means2d, s.radii, s.depths, s.tile_size,
                                              s.tile_width, s.tile_height, M)
    assert largest == M - 3
    b = bins.reshape(-1, M)
    for t, v in enumerate(lists):
        assert counts.reshape(-1)[t] == v.size
        np.testing.assert_array_equal(b[t, :v.size], v)
        assert (b[t, v.size:] == -1).all()


def test_bins_overflow_keeps_the_nearest():
    s = _scene("cams")
    lists = _sorted_lists(s)
    largest = max(len(v) for v in lists)
    M = largest // 2
    bins, counts, got_largest = oracle.bin_splats(s.means2d, s.radii, s.depths, s.tile_size,
                                                  s.tile_width, s.tile_height, M)
    assert got_largest == largest
    b = bins.reshape(-1, M)
    over = 0
    for t, v in enumerate(lists):
        assert counts.reshape(-1)[t] == v.size  # true counts, also past M
        k = min(v.size, M)
        np.testing.assert_array_equal(b[t, :k], v[:k])
        over += v.size > M
    assert over > 0


def test_bins_hand_example():
    # one 32x16 image (2 tiles), three splats: splat 2 covers both tiles,
    # splats 0 and 1 only the left one; depths 2, -1, 2 -> left tile order
    # by raw bits: 0 (2.0), 2 (2.0, later index), 1 (-1.0: sign bit set)
    means = np.array([[[8.0, 8.0], [4.0, 4.0], [16.0, 8.0]]], np.float32)
    radii = np.array([[2.0, 2.0, 6.0]], np.float32)
    depths = np.array([[2.0, -1.0, 2.0]], np.float32)
    bins, counts, largest = oracle.bin_splats(means, radii, depths, 16, 2, 1, 4)
    np.testing.assert_array_equal(counts, [[[3, 1]]])
    np.testing.assert_array_equal(bins[0, 0, 0], [0, 2, 1, -1])
    np.testing.assert_array_equal(bins[0, 0, 1], [2, -1, -1, -1])
    assert largest == 3
