"""The per-pixel step trace (gs_rasterize_fwd_steps / gs_rasterize_bwd_steps,
the trace buffers of rlx-metal 0.2.9, splat_training.rs): the forward's
records are exactly the pairs it composited (the same positions as the mask
trace, and as the oracle's composited positions away from near-tie pixels),
and the backward over them -- with every pixel recorded, and with a small
max_steps that sends most pixels to the list-walk fallback -- matches the
oracle's backward on the same forward state at 1e-3 relative."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (TIE_ALPHA, compare_forward, flipped_pixels, gpu_comp_hash, log_parity,
                      scene_to_dev, to_dev)
from test_gpu_raster import (_chain_scene, _compare_grads, _gpu_fwd_with_trace,
                             _oracle_bwd_state, _walked_splats)
from tile_gaussian_splat_gb300 import binding as gs

pytestmark = pytest.mark.gpu


def _steps_fwd(s, d, f, masks, K):
    return gs.gs_rasterize_fwd_steps(d["means2d"], d["conics"], d["colors"], d["opacities"],
                                     d["backgrounds"], None if masks is None else to_dev(masks),
                                     s.width, s.height, 16, f["offsets"], f["flatten_ids"],
                                     s.alpha_cutoff, s.transmittance_threshold, K)


@pytest.mark.parametrize("case", ["w5", "ragged_bg_masks"])
def test_step_records_are_the_composited_pairs(case):
    s, masks = _chain_scene(case)
    iso, ref, _, _, _ = _oracle_bwd_state(s, masks=masks, nudges=3, fwd_ties=True)
    d = scene_to_dev(s)
    f, tr = _gpu_fwd_with_trace(s, d, masks=masks)
    K = 512
    rgb, alpha, last, (pos, tb, cnt) = _steps_fwd(s, d, f, masks, K)
    torch.cuda.synchronize()
    # the same forward arithmetic: images bit for bit
    assert torch.equal(rgb, f["render_colors"]) and torch.equal(alpha, f["render_alphas"])
    assert torch.equal(last, f["last_ids"])
    cnt_h = cnt.cpu().numpy().reshape(-1)
    assert cnt_h.max() <= K
    pos_h = pos.cpu().numpy().reshape(K, -1)
    tb_h = tb.cpu().numpy().reshape(K, -1)
    # against the mask trace (every pixel with a composite) and the oracle
    # (every pixel away from a near-tie decision): the same positions in order
    comp = np.nonzero(cnt_h > 0)[0]
    rng = np.random.default_rng(0)
    sample = rng.choice(comp, min(4000, comp.size), replace=False)
    gh = gpu_comp_hash(tr, f["offsets"], f["last_ids"], sample, s.width, s.height)
    rh = ref["comp_hash"].reshape(-1)
    tie = ref["near_tie"].reshape(-1) > 0
    for p in sample.tolist():
        h = 14695981039346656037
        for j in pos_h[:cnt_h[p], p].tolist():
            h = ((h ^ j) * 1099511628211) % (1 << 64)
        assert h == gh[p]
        if not tie[p]:
            assert h == int(rh[p])
        # T before the first pair is 1, and it never grows
        t = tb_h[:cnt_h[p], p]
        assert t[0] == 1.0 and (np.diff(t) <= 0).all() and (t > 0).all()
    log_parity(kind="steps", pixels_with_composites=int(comp.size), checked=int(sample.size),
               max_steps_seen=int(cnt_h.max()))


@pytest.mark.parametrize("K", [512, 4])
@pytest.mark.parametrize("case", ["w5", "ragged_bg_masks"])
def test_step_backward_matches_oracle(case, K):
    # K = 512 records every pixel's pairs; K = 4 leaves most pixels to the
    # list-walk fallback
    s, masks = _chain_scene(case)
    iso, ref, _, g_rgb, g_a = _oracle_bwd_state(s, masks=masks, absgrad=True, nudges=3,
                                                fwd_ties=True)
    d = scene_to_dev(s)
    f, tr = _gpu_fwd_with_trace(s, d, masks=masks)
    rgb, alpha, last, steps = _steps_fwd(s, d, f, masks, K)
    got = gs.gs_rasterize_bwd_steps(d["means2d"], d["conics"], d["colors"], d["opacities"],
                                    d["backgrounds"], None if masks is None else to_dev(masks),
                                    s.width, s.height, 16, f["offsets"], f["flatten_ids"],
                                    s.alpha_cutoff, alpha, last, steps, to_dev(g_rgb),
                                    to_dev(g_a), absgrad=True)
    torch.cuda.synchronize()
    over = int((steps[2] > K).sum())
    if K == 4:
        assert over > 0.3 * int((steps[2] > 0).sum())
    # the oracle's backward on the same forward state: the GPU's alphas, last
    # ids and step records (a pixel they hold entirely reads T before each
    # pair; the others walk their list and divide, on both sides)
    rb = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, masks,
                              s.width, s.height, 16, iso["offsets"], iso["flatten_ids"],
                              s.alpha_cutoff, alpha.cpu().numpy(), last.cpu().numpy(), g_rgb,
                              g_a, absgrad=True, tie_rel=TIE_ALPHA, magnitudes=True,
                              steps=tuple(t.cpu().numpy() for t in steps))
    excl_pix, flagged, flipped = flipped_pixels(ref, rb, tr, f, s.width, s.height)
    log_parity(kind="steps_chain", max_steps=K, fallback_pixels=over, flagged_pixels=flagged,
               flipped_pixels=flipped, left_out_pixels=int(excl_pix.size))
    excluded = _walked_splats(s, iso["offsets"], iso["flatten_ids"], excl_pix,
                              [ref["last_ids"], last.cpu().numpy()])
    touched = rb["mag_opacities"] > 0
    assert (excluded & touched).sum() <= 0.02 * touched.sum()
    _compare_grads(rb, got, excluded)
    np.testing.assert_allclose(got["grad_means2d_abs"].cpu().numpy()[~excluded],
                               rb["grad_means2d_abs"][~excluded], rtol=1e-3, atol=1e-5)
    if s.backgrounds is not None:
        np.testing.assert_allclose(got["grad_backgrounds"].cpu().numpy(),
                                   rb["grad_backgrounds"], rtol=1e-4, atol=1e-3)


def test_step_backward_many_channels():
    # every channel in one pass: 7 channels (two chunks in the mask-trace
    # path) with absgrad, against the oracle's backward over the same records
    from tile_gaussian_splat_gb300 import scenes
    s = scenes.random_small(24, C=2, N=3000, W=100, H=70, sigma=(0.5, 10.0), channels=7)
    iso, ref, _, g_rgb, g_a = _oracle_bwd_state(s, absgrad=True, nudges=3, fwd_ties=True)
    d = scene_to_dev(s)
    f, tr = _gpu_fwd_with_trace(s, d)
    rgb, alpha, last, steps = _steps_fwd(s, d, f, None, 64)
    got = gs.gs_rasterize_bwd_steps(d["means2d"], d["conics"], d["colors"], d["opacities"],
                                    d["backgrounds"], None, s.width, s.height, 16, f["offsets"],
                                    f["flatten_ids"], s.alpha_cutoff, alpha, last, steps,
                                    to_dev(g_rgb), to_dev(g_a), absgrad=True)
    torch.cuda.synchronize()
    rb = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, None,
                              s.width, s.height, 16, iso["offsets"], iso["flatten_ids"],
                              s.alpha_cutoff, alpha.cpu().numpy(), last.cpu().numpy(), g_rgb,
                              g_a, absgrad=True, tie_rel=TIE_ALPHA, magnitudes=True,
                              steps=tuple(t.cpu().numpy() for t in steps))
    excl_pix, flagged, flipped = flipped_pixels(ref, rb, tr, f, s.width, s.height)
    excluded = _walked_splats(s, iso["offsets"], iso["flatten_ids"], excl_pix,
                              [ref["last_ids"], last.cpu().numpy()])
    _compare_grads(rb, got, excluded)
    np.testing.assert_allclose(got["grad_means2d_abs"].cpu().numpy()[~excluded],
                               rb["grad_means2d_abs"][~excluded], rtol=1e-3, atol=1e-5)
    np.testing.assert_allclose(got["grad_backgrounds"].cpu().numpy(), rb["grad_backgrounds"],
                               rtol=1e-4, atol=1e-3)
