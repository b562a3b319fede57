"""Pins of the oracle's stable key sort (two independent sorts must agree and
equal an independent library sort) and of its tile offsets (gsplat 1.0.0,
intersections.c: gs_radix_sort_without_gvl, gs_offset_encode)."""

import numpy as np
import pytest

import oracle


def _pairs(rng, n, distinct):
    keys = rng.choice(rng.integers(0, 2**63, distinct, dtype=np.uint64) * np.uint64(2)
                      + rng.integers(0, 2, distinct, dtype=np.uint64), n)
    return keys.astype(np.uint64), np.arange(n, dtype=np.int32)


@pytest.mark.parametrize("n,distinct", [(0, 1), (1, 1), (2, 1), (1000, 7), (5000, 5000),
                                        (20011, 300)])
def test_lsd_equals_stable_and_numpy(n, distinct):
    rng = np.random.default_rng(n + distinct)
    keys, ids = _pairs(rng, n, distinct)
    k1, i1 = keys.copy(), ids.copy()
    k2, i2 = keys.copy(), ids.copy()
    oracle.sort_pairs(k1, i1, impl="stable")
    oracle.sort_pairs(k2, i2, impl="lsd")
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(i1, i2)
    perm = np.argsort(keys, kind="stable")
    np.testing.assert_array_equal(k1, keys[perm])
    np.testing.assert_array_equal(i1, ids[perm])
    # stability: equal keys keep ascending original positions
    if n > 1:
        same = k1[1:] == k1[:-1]
        assert (i1[1:][same] > i1[:-1][same]).all()


def test_lsd_uses_all_64_bits():
    keys = np.array([1 << 63, 1, 1 << 40, 0, (1 << 63) + 1, 1 << 8], np.uint64)
    ids = np.arange(6, dtype=np.int32)
    oracle.sort_pairs(keys, ids, impl="lsd")
    np.testing.assert_array_equal(ids, [3, 1, 5, 2, 0, 4])


def _brute_offsets(keys, C, TW, TH):
    tb = oracle.tile_bits(TW, TH)
    counts = np.zeros(C * TW * TH, np.int64)
    for k in keys.tolist():
        upper = k >> 32
        counts[(upper >> tb) * TW * TH + (upper & ((1 << tb) - 1))] += 1
    return counts


@pytest.mark.parametrize("C,TW,TH", [(1, 4, 4), (3, 5, 3), (2, 1, 1), (1, 7, 9)])
def test_offsets_invariants(C, TW, TH):
    rng = np.random.default_rng(C * 100 + TW * 10 + TH)
    tb = oracle.tile_bits(TW, TH)
    n = 3000
    cam = rng.integers(0, C, n, dtype=np.uint64)
    tile = rng.integers(0, TW * TH, n, dtype=np.uint64)
    depth = rng.integers(0, 2**32, n, dtype=np.uint64)
    keys = (((cam << np.uint64(tb)) | tile) << np.uint64(32)) | depth
    ids = np.arange(n, dtype=np.int32)
    oracle.sort_pairs(keys, ids)
    off = oracle.tile_offsets(keys, C, TW, TH).reshape(-1)
    counts = _brute_offsets(keys, C, TW, TH)
    assert off[0] == 0
    assert (np.diff(off) >= 0).all()
    end = np.append(off[1:], n)
    np.testing.assert_array_equal(end - off, counts)
    flat_tile = (keys >> np.uint64(32 + tb)) * np.uint64(TW * TH) + \
        ((keys >> np.uint64(32)) & np.uint64((1 << tb) - 1))
    for t in range(C * TW * TH):
        assert (flat_tile[off[t]:end[t]] == t).all()
    # counting, so the same offsets come from unsorted keys
    np.testing.assert_array_equal(
        oracle.tile_offsets(keys[rng.permutation(n)], C, TW, TH).reshape(-1), off)


def test_offsets_empty_and_errors():
    np.testing.assert_array_equal(oracle.tile_offsets(np.zeros(0, np.uint64), 2, 3, 3),
                                  np.zeros((2, 3, 3), np.int32))
    tb = oracle.tile_bits(3, 3)  # 4 bits, 9 tiles: tile ids 9..15 are outside
    bad_tile = np.array([np.uint64(12) << np.uint64(32)], np.uint64)
    with pytest.raises(oracle.KeyOutOfGrid):
        oracle.tile_offsets(bad_tile, 1, 3, 3)
    bad_cam = np.array([np.uint64(2 << tb) << np.uint64(32)], np.uint64)
    with pytest.raises(oracle.KeyOutOfGrid):
        oracle.tile_offsets(bad_cam, 2, 3, 3)
