"""Parity at full size, in the launch configuration the bench times.

Workloads 3 (4 x 1M splats, 1920x1080) and 4 (6M splats, 3840x2160):
  * tiles_per_gauss, sorted keys, flatten_ids and offsets: bit-exact over
    everything (the oracle's stable sort runs on all intersections);
  * forward: every pixel of the heaviest tiles plus random pixels, computed
    one by one by the oracle;
  * backward: the upstream gradient is nonzero only on sampled tiles, so the
    oracle's walk over those pixels alone gives every splat's exact gradient
    (a pixel with zero upstream gradient adds zero to every term).
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, TIE_ALPHA, TIE_T, compare_forward, flipped_pixels, gpu_forward,
                      log_parity, scene_to_dev, to_dev, u64)
from test_gpu_raster import _compare_grads, _gpu_fwd_with_trace, _walked_splats
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_pixels(s, offsets, rng, n_random=3000, n_heavy=6):
    TW, TH = s.tile_width, s.tile_height
    flat = offsets.reshape(-1).astype(np.int64)
    lens = np.diff(np.append(flat, np.iinfo(np.int64).max))
    lens[-1] = 0
    heavy = np.argsort(-lens)[:n_heavy]
    pix = []
    for t in heavy:
        c, loc = divmod(int(t), TW * TH)
        ty, tx = divmod(loc, TW)
        for y in range(ty * 16, min(s.height, ty * 16 + 16)):
            for x in range(tx * 16, min(s.width, tx * 16 + 16)):
                pix.append((c * s.height + y) * s.width + x)
    pix += rng.integers(0, s.C * s.width * s.height, n_random).tolist()
    return np.unique(np.array(pix, np.int64)), heavy


def _tile_pixels(s, tiles):
    pix = []
    for t in tiles:
        c, loc = divmod(int(t), s.tile_width * s.tile_height)
        ty, tx = divmod(loc, s.tile_width)
        for y in range(ty * 16, min(s.height, ty * 16 + 16)):
            for x in range(tx * 16, min(s.width, tx * 16 + 16)):
                pix.append((c * s.height + y) * s.width + x)
    return np.array(pix, np.int64)


@pytest.mark.parametrize("k", [3, 4])
def test_full_size_workload(k):
    s = scenes.workload(k)
    d = scene_to_dev(s)
    got = gpu_forward(s, d)
    torch.cuda.synchronize()
    r_tpg, r_keys, r_ids = oracle.isect_tiles(s.means2d, s.radii, s.depths, 16, s.tile_width,
                                              s.tile_height)
    np.testing.assert_array_equal(got["tiles_per_gauss"].cpu().numpy(), r_tpg)
    np.testing.assert_array_equal(u64(got["keys"]), r_keys)
    np.testing.assert_array_equal(got["flatten_ids"].cpu().numpy(), r_ids)
    r_off = oracle.tile_offsets(r_keys, s.C, s.tile_width, s.tile_height)
    np.testing.assert_array_equal(got["offsets"].cpu().numpy(), r_off)
    del r_keys

    rng = np.random.default_rng(k)
    pix, heavy = _sample_pixels(s, r_off, rng)
    ref = oracle.rasterize_fwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, None,
                               s.width, s.height, 16, r_off, r_ids, s.alpha_cutoff,
                               s.transmittance_threshold, pixels=pix, tie_rel=TIE_ALPHA,
                               tie_rel_T=TIE_T)
    ties = compare_forward(ref, got, s, pixels=pix)
    # the sample is biased to the heaviest tiles (lists of thousands of
    # entries), where a near tie on some entry is likelier
    assert ties <= 0.05 * pix.size

    # backward with the upstream gradient on 8 sampled tiles only (heaviest first)
    tiles = np.concatenate([heavy[:4], rng.choice(s.C * s.tile_width * s.tile_height, 4)])
    bp = _tile_pixels(s, tiles)
    g_rgb = np.zeros((s.C, s.height, s.width, 3), np.float32)
    g_a = np.zeros((s.C, s.height, s.width, 1), np.float32)
    g_rgb.reshape(-1, 3)[bp] = rng.standard_normal((bp.size, 3)).astype(np.float32)
    g_a.reshape(-1)[bp] = rng.standard_normal(bp.size).astype(np.float32)
    # the GPU walks the oracle's forward state at those pixels (zero elsewhere:
    # render_alpha 0 makes every pair invalid).  Splats that took part in a
    # near-tie decision -- a backward alpha within TIE_ALPHA of the cutoff or
    # clamp, or a forward stop within TIE_T of the threshold -- are nudged by
    # 1 % in opacity (a deterministic change of the seeded input, as in
    # test_gpu_raster), so the GPU forward that the chain below runs makes
    # the oracle's decisions
    for it in range(4):
        refb = oracle.rasterize_fwd(s.means2d, s.conics, s.colors, s.opacities, None, None,
                                    s.width, s.height, 16, r_off, r_ids, s.alpha_cutoff,
                                    s.transmittance_threshold, pixels=bp, tie_rel=TIE_ALPHA,
                                    tie_rel_T=TIE_T)
        ra = np.zeros((s.C, s.height, s.width, 1), np.float32)
        li = np.full((s.C, s.height, s.width), -1, np.int32)
        ra.reshape(-1)[bp] = refb["render_alphas"].reshape(-1)[bp]
        li.reshape(-1)[bp] = refb["last_ids"].reshape(-1)[bp]
        rb = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, None, None,
                                  s.width, s.height, 16, r_off, r_ids, s.alpha_cutoff, ra, li,
                                  g_rgb, g_a, pixels=bp, tie_rel=TIE_ALPHA, magnitudes=True)
        tie = rb["tie_splats"].astype(bool) | refb["tie_splats"].astype(bool)
        if not tie.any() or it == 3:
            break
        s.opacities[tie] *= np.where(s.opacities[tie] < 0.98, 1.01, 0.99).astype(np.float32)
    d["opacities"] = to_dev(s.opacities)
    gb = gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"], None,
                             None, s.width, s.height, 16, got["offsets"], got["flatten_ids"],
                             s.alpha_cutoff, to_dev(ra), to_dev(li), to_dev(g_rgb), to_dev(g_a))
    torch.cuda.synchronize()
    touched = (rb["mag_opacities"] > 0).reshape(-1)
    assert touched.sum() > 1000
    excluded = _walked_splats(s, r_off, r_ids, np.nonzero(rb["near_tie"].reshape(-1))[0], [li])
    assert (excluded.reshape(-1) & touched).sum() <= 0.05 * touched.sum()
    _compare_grads(rb, gb, excluded)

    # the chain the bench times, at full size in its launch configuration:
    # the GPU forward (with the trace) on the same scene, then the
    # trace-driven GPU backward on the GPU's own forward state, compared with
    # the oracle's backward on that same state.  Every pixel carries GPU
    # state, but only the sampled tiles have a nonzero upstream gradient, so
    # the oracle's walk over those tiles gives every gradient
    f, tr = _gpu_fwd_with_trace(s, d)
    gc = gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"], None,
                             None, s.width, s.height, 16, f["offsets"], f["flatten_ids"],
                             s.alpha_cutoff, f["render_alphas"], f["last_ids"], to_dev(g_rgb),
                             to_dev(g_a), trace=tr)
    torch.cuda.synchronize()
    compare_forward(refb, f, s, pixels=bp)
    rb = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, None, None, s.width,
                              s.height, 16, r_off, r_ids, s.alpha_cutoff,
                              f["render_alphas"].cpu().numpy(), f["last_ids"].cpu().numpy(),
                              g_rgb, g_a, pixels=bp, tie_rel=TIE_ALPHA, magnitudes=True)
    # of the pixels flagged near a decision, leave out those where the GPU's
    # composited positions differ from the oracle's (and near-clamp pairs)
    excl_pix, flagged, flipped = flipped_pixels(refb, rb, tr, f, s.width, s.height)
    log_parity(kind="chain", flagged_pixels=flagged, flipped_pixels=flipped,
               left_out_pixels=int(excl_pix.size))
    excluded = _walked_splats(s, r_off, r_ids, excl_pix, [li, f["last_ids"].cpu().numpy()])
    assert (excluded.reshape(-1) & touched).sum() <= 0.05 * touched.sum()
    _compare_grads(rb, gc, excluded)
