"""GPU parity of the fixed-capacity bin lists (gs_bin_splats) and of the
raster calls over them (gs_rasterize_fwd_bins / gs_rasterize_bwd_bins).

* bins and bin_counts bit for bit equal to the oracle's (no overflow), and
  at full size equal to the sorted path's tile slices of flatten_ids;
* on overflow: GS_ERR_CAPACITY, exact counts, and every kept entry one of
  the tile's splats, in compositing order;
* compositing over bins gives the same images as over the sorted lists
  (the same splat sequence per tile), last ids mapped between the two
  position spaces; the backward the same gradients up to atomic order.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, gpu_forward, scene_to_dev, to_dev
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu


def _ties_scene():
    s = scenes.random_small(4, C=2, N=600, W=64, H=48, sigma=(1.0, 8.0))
    rng = np.random.default_rng(0)
    s.depths = rng.choice(np.array([1.5, 2.0, -0.5, 0.0, -0.0], np.float32),
                          s.depths.shape).astype(np.float32)
    return s


def _scene(kind):
    return {"w1": scenes.workload1, "w2": scenes.workload2, "ties": _ties_scene,
            "cams": lambda: scenes.random_small(3, C=3, N=800, W=90, H=70,
                                                sigma=(0.5, 12.0)),
            # bins of 2-3.4k entries beside smaller ones: both merge kernels
            "mid": lambda: scenes.random_small(6, C=2, N=9000, W=400, H=300,
                                               sigma=(0.5, 60.0)),
            # every bin about 15k entries: the bitonic network of the largest
            # capacities
            "big": lambda: scenes.random_small(5, C=1, N=15000, W=64, H=48,
                                               sigma=(30.0, 60.0))}[kind]()


def _gpu_bins(s, d, M, status=None):
    bins, counts = gs.gs_bin_splats(d["means2d"], d["radii"], d["depths"], s.tile_size,
                                    s.tile_width, s.tile_height, M, d_status=status)
    torch.cuda.synchronize()
    return bins.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("kind", ["w1", "w2", "ties", "cams", "mid", "big"])
def test_bins_bit_exact(kind):
    s = _scene(kind)
    _, _, largest = oracle.bin_splats(s.means2d, s.radii, s.depths, s.tile_size, s.tile_width,
                                      s.tile_height, 1)
    M = largest + 5
    rb, rc, _ = oracle.bin_splats(s.means2d, s.radii, s.depths, s.tile_size, s.tile_width,
                                  s.tile_height, M)
    st = gs.new_status(DEV)
    b, c = _gpu_bins(s, scene_to_dev(s), M, st)
    gs.check_status(st)
    np.testing.assert_array_equal(c, rc)
    np.testing.assert_array_equal(b, rb)


@pytest.mark.parametrize("kind", ["cams", "mid"])
def test_bins_overflow(kind):
    s = _scene(kind)
    _, rc, largest = oracle.bin_splats(s.means2d, s.radii, s.depths, s.tile_size, s.tile_width,
                                       s.tile_height, 1)
    # "mid": a capacity above 2048, so that the bins it cuts are the larger ones
    M = max(1, largest // 3) if kind == "cams" else largest * 2 // 3
    full, _, _ = oracle.bin_splats(s.means2d, s.radii, s.depths, s.tile_size, s.tile_width,
                                   s.tile_height, largest)
    st = gs.new_status(DEV)
    b, c = _gpu_bins(s, scene_to_dev(s), M, st)
    assert int(st.item()) == 2  # GS_ERR_CAPACITY
    np.testing.assert_array_equal(c, rc)
    key = lambda ids: (s.depths.reshape(-1)[ids].view(np.uint32).astype(np.uint64) << 32) | ids
    fb = full.reshape(-1, largest)
    for t, (row, n) in enumerate(zip(b.reshape(-1, M), c.reshape(-1))):
        k = min(n, M)
        assert (row[k:] == -1).all()
        kept = row[:k]
        assert np.isin(kept, fb[t, :n]).all()
        assert (np.diff(key(kept.astype(np.uint64))) > 0).all()


@pytest.mark.slow
def test_bins_full_size_equal_sorted_slices():
    s = scenes.workload(3)
    d = scene_to_dev(s)
    f = gpu_forward(s, d)
    offs = f["offsets"].cpu().numpy().reshape(-1).astype(np.int64)
    ids = f["flatten_ids"].cpu().numpy()
    ends = np.append(offs[1:], ids.size)
    largest = int((ends - offs).max())
    M = (largest + 31) // 32 * 32
    st = gs.new_status(DEV)
    b, c = _gpu_bins(s, d, M, st)
    gs.check_status(st)
    np.testing.assert_array_equal(c.reshape(-1), ends - offs)
    b = b.reshape(-1, M)
    # every slot k < count holds the tile's k-th sorted id, the rest -1
    k = np.arange(M)[None, :]
    cnt = (ends - offs)[:, None]
    src = np.where(k < cnt, offs[:, None] + k, 0)
    want = np.where(k < cnt, ids[np.minimum(src, ids.size - 1)], -1)
    np.testing.assert_array_equal(b, want)


def _raster_both(s, masks=None, trace=False):
    d = scene_to_dev(s)
    f = gpu_forward(s, d, masks=masks)
    offs = f["offsets"].cpu().numpy().reshape(-1).astype(np.int64)
    ids = f["flatten_ids"]
    ends = np.append(offs[1:], ids.numel())
    M = int((ends - offs).max()) + 2
    bins, counts = gs.gs_bin_splats(d["means2d"], d["radii"], d["depths"], 16, s.tile_width,
                                    s.tile_height, M)
    m = None if masks is None else to_dev(masks)
    tr_b = torch.zeros((bins.numel(), 8), dtype=torch.int32, device=DEV) if trace else None
    rgb, alpha, last = gs.gs_rasterize_fwd_bins(
        d["means2d"], d["conics"], d["colors"], d["opacities"], d["backgrounds"], m, s.width,
        s.height, 16, bins, counts, s.alpha_cutoff, s.transmittance_threshold, trace=tr_b)
    torch.cuda.synchronize()
    return d, f, offs, M, bins, counts, (rgb, alpha, last), tr_b, m


@pytest.mark.parametrize("kind", ["w2", "ties"])
def test_forward_over_bins_equals_sorted(kind):
    s = _scene(kind)
    d, f, offs, M, bins, counts, (rgb, alpha, last), _, _ = _raster_both(s)
    assert torch.equal(rgb, f["render_colors"])
    assert torch.equal(alpha, f["render_alphas"])
    # last ids: position t * M + k in the bins <-> offsets[t] + k in the lists
    lb = last.cpu().numpy().astype(np.int64)
    ls = f["last_ids"].cpu().numpy().astype(np.int64)
    assert ((lb < 0) == (ls < 0)).all()
    t = lb[lb >= 0] // M
    np.testing.assert_array_equal(lb[lb >= 0] - t * M + offs[t], ls[ls >= 0])


def test_backward_over_bins_equals_sorted():
    s = scenes.random_small(3, C=2, N=4000, W=150, H=90, sigma=(0.5, 10.0))
    masks = np.random.default_rng(1).integers(0, 2, (2, 6, 10)).astype(np.int32)
    d, f, offs, M, bins, counts, (rgb, alpha, last), tr_b, m = _raster_both(s, masks, trace=True)
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=2)
    fs = gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                             d["backgrounds"], m, s.width, s.height, 16, f["offsets"],
                             f["flatten_ids"], s.alpha_cutoff, s.transmittance_threshold)
    a = gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                            d["backgrounds"], m, s.width, s.height, 16, f["offsets"],
                            f["flatten_ids"], s.alpha_cutoff, fs[1], fs[2], to_dev(g_rgb),
                            to_dev(g_a), absgrad=True)
    for trace in (None, tr_b):
        b = gs.gs_rasterize_bwd_bins(d["means2d"], d["conics"], d["colors"], d["opacities"],
                                     d["backgrounds"], m, s.width, s.height, 16, bins, counts,
                                     s.alpha_cutoff, alpha, last, to_dev(g_rgb), to_dev(g_a),
                                     absgrad=True, trace=trace)
        for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities",
                  "grad_means2d_abs", "grad_backgrounds"):
            x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
            scale = np.abs(x).max() + 1e-30
            np.testing.assert_allclose(y, x, rtol=1e-4, atol=1e-6 * scale, err_msg=k)


def test_bins_empty_and_invisible():
    for N, far in ((0, False), (50, True)):
        s = scenes.random_small(6, C=2, N=N, W=64, H=48)
        if far:
            s.means2d[:] = -1000.0
        st = gs.new_status(DEV)
        b, c = _gpu_bins(s, scene_to_dev(s), 8, st)
        gs.check_status(st)
        assert (c == 0).all() and (b == -1).all()


def test_bin_argument_errors():
    s = scenes.workload1()
    d = scene_to_dev(s)
    for M in (0, 16385):
        with pytest.raises(gs.GsError) as e:
            gs.gs_bin_splats(d["means2d"], d["radii"], d["depths"], 16, 4, 4, M)
        assert e.value.code == 1
