"""GPU parity of intersection, sort and tile ranges (gs_isect_tiles,
gs_tile_offsets, gs_sort_pairs) against the oracle: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, gpu_isect, scene_to_dev, to_dev, u64
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu


def _check_isect(s, sort=True):
    d = scene_to_dev(s)
    st = gs.new_status(DEV)
    tpg, keys, ids = gpu_isect(s, d, sort=sort, status=st)
    gs.check_status(st)
    r_tpg, r_keys, r_ids = oracle.isect_tiles(s.means2d, s.radii, s.depths, s.tile_size,
                                              s.tile_width, s.tile_height, sort=sort)
    np.testing.assert_array_equal(tpg.cpu().numpy(), r_tpg)
    assert keys.numel() == r_keys.size
    np.testing.assert_array_equal(u64(keys), r_keys)
    np.testing.assert_array_equal(ids.cpu().numpy(), r_ids)
    if keys.numel():
        off = gs.gs_tile_offsets(keys, s.C, s.tile_width, s.tile_height, d_status=st) \
            if sort else None
        if sort:
            gs.check_status(st)
            np.testing.assert_array_equal(
                off.cpu().numpy(), oracle.tile_offsets(r_keys, s.C, s.tile_width, s.tile_height))
    return r_keys.size


@pytest.mark.parametrize("k", [1, 2, 5])
@pytest.mark.parametrize("sort", [True, False])
def test_workloads_small(k, sort):
    assert _check_isect(scenes.workload(k), sort=sort) > 0


@pytest.mark.parametrize("seed", range(4))
def test_random_multi_camera_ragged(seed):
    # 3 cameras, ragged 200x120 image (13x8 tiles), big radii: many tiles per splat,
    # I spans several sort tiles with a ragged tail
    s = scenes.random_small(seed, C=3, N=4000, W=200, H=120, sigma=(0.5, 12.0),
                            elliptical=seed % 2 == 0)
    n = _check_isect(s)
    assert n > 3 * 3072


@pytest.mark.parametrize("seed", range(3))
def test_emission_long_runs_and_empty_splats(seed):
    # the emission hands each warp 64 consecutive splats (in depth order) and
    # writes their keys 32 at a time, a key's splat found from the round's
    # splat-start bits or carried over from the previous round: splats of
    # hundreds of tiles (many rounds with no start), long stretches of splats
    # off screen (no keys), and single-tile splats side by side, in a
    # depth order that mixes them, must give the oracle's keys bit for bit
    s = scenes.random_small(30 + seed, C=2, N=3000, W=640, H=360, sigma=(0.5, 2.0))
    rng = np.random.default_rng(seed)
    kind = rng.integers(0, 10, (s.C, s.N))
    big = kind == 0            # about 10 %: radii of 60-200 px
    gone = (kind >= 1) & (kind <= 4)  # about 40 %: entirely off screen
    s.radii[big] = rng.uniform(60.0, 200.0, (int(big.sum()), 2)).astype(np.float32)
    s.means2d[gone] = np.float32(-1000.0)
    # runs of equal depth so that long stretches of one kind meet in the order
    s.depths[:] = np.where(big, 1.0, np.where(gone, 2.0, 3.0)).astype(np.float32)
    s.depths[:, ::97] = np.float32(2.5)
    n = _check_isect(s)
    assert n > 10 * 3072


def test_equal_depths_keep_splat_order():
    # many equal depths and equal keys: the sort must be stable
    s = scenes.random_small(7, C=2, N=20000, W=256, H=256, sigma=(0.5, 6.0))
    s.depths[:] = np.round(s.depths * 2) / 2  # 19 distinct depths
    _check_isect(s)


def test_negative_and_special_depths():
    s = scenes.random_small(8, C=1, N=5000, W=128, H=96)
    s.depths[0, ::3] *= -1.0
    s.depths[0, 1::7] = 0.0
    s.depths[0, 2::11] = -0.0
    _check_isect(s)


def test_degenerate_splats():
    s = scenes.random_small(9, C=1, N=3000, W=64, H=64)
    s.radii[0, ::5] = 0.0
    s.radii[0, 1::9] = -3.0
    s.means2d[0, 2::13] = np.nan
    s.radii[0, 3::17] = np.inf
    s.means2d[0, 4::19] = 1e30
    s.means2d[0, 5::23] = -1e30
    _check_isect(s)


def test_empty_and_invisible():
    s = scenes.random_small(1, C=2, N=0, W=64, H=64)
    assert _check_isect(s) == 0
    s = scenes.random_small(1, C=2, N=100, W=64, H=64)
    s.means2d[:] = -1000.0
    assert _check_isect(s) == 0


def test_single_tile_grid():
    s = scenes.random_small(2, C=1, N=500, W=16, H=16)
    assert _check_isect(s) > 0


def test_three_tile_passes():
    # 256x256 tiles (16 bits) and 3 cameras (2 bits): three 8-bit camera|tile
    # passes, so emission starts in the workspace buffer and the passes
    # alternate twice before the widening one
    s = scenes.random_small(5, C=3, N=3000, W=4096, H=4096, sigma=(2.0, 60.0))
    assert gs.gs_tile_bits(s.tile_width, s.tile_height) == 16
    assert _check_isect(s) > 0


def test_max_camera_bits():
    # tile_bits + camera bits == 32: 2^16 tiles (256x256 grid), 2^16 cameras
    C = 65536
    rng = np.random.default_rng(3)
    s = scenes.random_small(3, C=1, N=1, W=16, H=16)
    s.C, s.N, s.width, s.height = C, 1, 4096, 4096
    s.means2d = rng.uniform(0, 4096, (C, 1, 2)).astype(np.float32)
    s.radii = rng.uniform(1, 40, (C, 1, 2)).astype(np.float32)
    s.depths = rng.uniform(1, 5, (C, 1)).astype(np.float32)
    assert gs.gs_tile_bits(256, 256) == 16
    _check_isect(s)


def test_too_many_key_bits_rejected():
    s = scenes.random_small(3, C=65537, N=1, W=16, H=16)
    d = scene_to_dev(s)
    with pytest.raises(gs.GsError) as e:
        gs.gs_isect_tiles(d["means2d"], d["radii"], d["depths"], 16, 256, 256)
    assert e.value.code == 1


def test_count_mismatch_reported():
    s = scenes.random_small(4, C=1, N=300, W=64, H=64)
    d = scene_to_dev(s)
    tpg, keys, ids = gpu_isect(s, d)
    I = keys.numel()
    ws = torch.empty(gs.gs_isect_workspace_size(1, 300, 4, 4, I - 1, True), dtype=torch.uint8,
                     device=DEV)
    st = gs.new_status(DEV)
    k2 = torch.empty(I - 1, dtype=torch.int64, device=DEV)
    i2 = torch.empty(I - 1, dtype=torch.int32, device=DEV)
    rc = gs.lib().gs_isect_tiles(gs._ptr(d["means2d"]), gs._ptr(d["radii"]), 1,
                                 gs._ptr(d["depths"]), 1, 300, 16, 4, 4, 1, None, None,
                                 gs._ptr(k2), gs._ptr(i2), I - 1, gs._ptr(ws), ws.numel(),
                                 gs._ptr(st), gs._stream())
    assert rc == 0
    assert int(st.item()) == 8


def test_tile_offsets_errors():
    tb = gs.gs_tile_bits(3, 3)
    good = (np.uint64(4) << np.uint64(32)) | np.uint64(7)
    bad_tile = np.uint64(12) << np.uint64(32)
    bad_cam = np.uint64(2 << tb) << np.uint64(32)
    for keys, code in [([good, bad_tile], 3), ([bad_cam], 3),
                       ([good, np.uint64(1) << np.uint64(32)], 7)]:
        k = torch.from_numpy(np.array(keys, np.uint64).view(np.int64)).to(DEV)
        st = gs.new_status(DEV)
        gs.gs_tile_offsets(k, 2, 3, 3, d_status=st)
        assert int(st.item()) == code
    st = gs.new_status(DEV)
    off = gs.gs_tile_offsets(torch.empty(0, dtype=torch.int64, device=DEV), 2, 3, 3, d_status=st)
    assert (off == 0).all() and int(st.item()) == 0


@pytest.mark.parametrize("n,distinct,begin,end", [
    (0, 1, 0, 64), (1, 1, 0, 64), (2, 2, 0, 64), (3071, 50, 0, 64), (3072, 3072, 0, 64),
    (3073, 3, 0, 64), (100_000, 1000, 0, 64), (250_007, 250_007, 0, 64), (100_000, 77, 32, 47),
    (65_536, 9, 5, 13)])
def test_sort_pairs(n, distinct, begin, end):
    rng = np.random.default_rng(n + distinct + begin)
    pool = rng.integers(0, 2**63, distinct, dtype=np.uint64) * np.uint64(2) + \
        rng.integers(0, 2, distinct, dtype=np.uint64)
    keys = rng.choice(pool, n).astype(np.uint64) if n else np.zeros(0, np.uint64)
    vals = np.arange(n, dtype=np.int32)
    k = torch.from_numpy(keys.view(np.int64).copy()).to(DEV)
    v = torch.from_numpy(vals.copy()).to(DEV)
    st = gs.new_status(DEV)
    gs.gs_sort_pairs(k, v, begin, end, d_status=st)
    gs.check_status(st)
    width = end - begin
    mask = np.uint64((1 << width) - 1) if width < 64 else np.uint64(2**64 - 1)
    digits = (keys >> np.uint64(begin)) & mask
    perm = np.argsort(digits, kind="stable")
    np.testing.assert_array_equal(u64(k), keys[perm])
    np.testing.assert_array_equal(v.cpu().numpy(), vals[perm])
    if begin == 0 and end == 64:
        rk, rv = keys.copy(), vals.copy()
        oracle.sort_pairs(rk, rv)
        np.testing.assert_array_equal(u64(k), rk)
        np.testing.assert_array_equal(v.cpu().numpy(), rv)


@pytest.mark.parametrize("koff,voff", [(0, 0), (1, 1), (0, 2), (1, 3)])
@pytest.mark.parametrize("n", [5, 2048 * 3 + 7, 100_003])
def test_sort_pairs_unaligned_buffers(n, koff, voff):
    # the radix passes bring each tile's values in by a bulk copy of their
    # 16-byte aligned middle plus plain loads of the ragged ends: keys 8 bytes
    # and values 4, 8 or 12 bytes past a 16-byte boundary sort exactly as
    # aligned ones, and the elements beside the slices stay untouched
    rng = np.random.default_rng(n + 7 * koff + voff)
    pool = rng.integers(0, 2**63, max(n // 3, 1), dtype=np.uint64)
    keys = rng.choice(pool, n).astype(np.uint64)
    vals = np.arange(n, dtype=np.int32)
    kbuf = torch.full((n + 2,), -7, dtype=torch.int64, device=DEV)
    vbuf = torch.full((n + 4,), -7, dtype=torch.int32, device=DEV)
    k = kbuf[koff:koff + n]
    v = vbuf[voff:voff + n]
    k.copy_(torch.from_numpy(keys.view(np.int64).copy()))
    v.copy_(torch.from_numpy(vals.copy()))
    assert (k.data_ptr() % 16 != 0) == (koff == 1) and (v.data_ptr() % 16) == 4 * voff
    st = gs.new_status(DEV)
    gs.gs_sort_pairs(k, v, 0, 64, d_status=st)
    gs.check_status(st)
    perm = np.argsort(keys, kind="stable")
    np.testing.assert_array_equal(u64(k), keys[perm])
    np.testing.assert_array_equal(v.cpu().numpy(), vals[perm])
    kb, vb = kbuf.cpu().numpy(), vbuf.cpu().numpy()
    assert (np.delete(kb, np.arange(koff, koff + n)) == -7).all()
    assert (np.delete(vb, np.arange(voff, voff + n)) == -7).all()


def test_repeat_runs_bit_identical():
    # races in the scan/sort would show up as run-to-run differences
    s = scenes.workload2()
    d = scene_to_dev(s)
    a = gpu_isect(s, d)
    for _ in range(3):
        b = gpu_isect(s, d)
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("n", [1, 3, 4, 5, 127, 128, 129, 1003, 70_001])
def test_tile_offsets_aligned_and_unaligned(n):
    # four keys per thread with 16-byte loads when aligned, scalar loads when
    # not; the key before a thread's first comes from the neighbouring lane:
    # both give the oracle's offsets bit for bit, at every tail length
    C, TW, TH = 2, 7, 5
    tb = gs.gs_tile_bits(TW, TH)
    rng = np.random.default_rng(n)
    cam = rng.integers(0, C, n).astype(np.uint64)
    tile = rng.integers(0, TW * TH, n).astype(np.uint64)
    upper = np.sort((cam << np.uint64(tb)) | tile)
    keys = (upper << np.uint64(32)) | rng.integers(0, 2**32, n, dtype=np.uint64)
    ref = oracle.tile_offsets(keys, C, TW, TH)
    buf = torch.from_numpy(np.concatenate([keys[:1], keys]).view(np.int64)).to(DEV)
    for k in (buf[1:].clone(), buf[1:]):  # 16-byte aligned copy, then an 8-byte offset view
        st = gs.new_status(DEV)
        off = gs.gs_tile_offsets(k, C, TW, TH, d_status=st)
        assert int(st.item()) == 0
        np.testing.assert_array_equal(off.cpu().numpy(), ref)


@pytest.mark.parametrize("pos", [512, 513, 515, 516, 640, 999])
def test_tile_offsets_errors_inside_long_lists(pos):
    # an unsorted step or an out-of-grid key at group starts, ends and lane
    # boundaries of the vector path is reported
    C, TW, TH = 1, 8, 8
    n = 1000
    rng = np.random.default_rng(pos)
    # one descending step at pos: tiles 10..20 before it, 0..9 from it on
    unsorted = np.concatenate([np.sort(rng.integers(10, 21, pos)),
                               np.sort(rng.integers(0, 10, n - pos))]).astype(np.uint64)
    # keys from pos on all past the grid (and sorted, so no other error)
    grid = np.sort(rng.integers(0, TW * TH, n)).astype(np.uint64)
    grid[pos:] = np.uint64(TW * TH + 3)
    for u, code in ((unsorted, 7), (grid, 3)):
        keys = torch.from_numpy((u << np.uint64(32)).view(np.int64)).to(DEV)
        st = gs.new_status(DEV)
        gs.gs_tile_offsets(keys, C, TW, TH, d_status=st)
        assert int(st.item()) == code, (code, pos)


@pytest.mark.parametrize("ts", [1, 8, 10, 13, 32])
def test_tile_sizes_power_of_two_and_not(ts):
    # the bounds divide by the tile size; for powers of two the kernels
    # multiply by the exact reciprocal instead (the same correctly rounded
    # value), for other sizes they divide: both bit-exact to the oracle's
    # float division, including means +- radii on exact tile edges and
    # quarter-pixel offsets
    s = scenes.random_small(40 + ts, C=2, N=5000, W=203, H=117, tile_size=ts,
                            sigma=(0.3, 9.0))
    rng = np.random.default_rng(ts)
    edge = rng.integers(0, 2 * s.N, 500)
    m = s.means2d.reshape(-1, 2)
    r = s.radii.reshape(-1, 2)
    m[edge % s.N] = (rng.integers(0, 12, (500, 2)) * ts + r[edge % s.N]).astype(np.float32)
    m[edge[:250] % s.N] += np.float32(0.25)
    _check_isect(s)
