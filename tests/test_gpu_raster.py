"""GPU parity of forward compositing and the backward (gs_rasterize_fwd,
gs_rasterize_bwd) against the oracle: last_ids exact and RGBA within 1e-5
max-abs away from near-tie pixels; gradients within 1e-3 relative with a
1e-6 absolute floor."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, TIE_ALPHA, TIE_T, compare_forward, flipped_pixels, gpu_forward,
                      log_parity, scene_to_dev, to_dev)
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu


def _oracle_forward(s, masks=None):
    iso, fwd = oracle.render(s, tie_rel=TIE_ALPHA, tie_rel_T=TIE_T)
    if masks is not None:
        fwd = oracle.rasterize_fwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds,
                                   masks, s.width, s.height, s.tile_size, iso["offsets"],
                                   iso["flatten_ids"], s.alpha_cutoff,
                                   s.transmittance_threshold, tie_rel=TIE_ALPHA, tie_rel_T=TIE_T)
    return iso, fwd


@pytest.mark.parametrize("k", [1, 2])
def test_forward_workloads(k):
    s = scenes.workload(k)
    iso, ref = _oracle_forward(s)
    got = gpu_forward(s, scene_to_dev(s))
    ties = compare_forward(ref, got, s)
    assert ties <= 1e-2 * s.C * s.width * s.height


@pytest.mark.parametrize("seed,W,H,C", [(0, 100, 70, 2), (1, 33, 17, 1), (2, 257, 129, 3)])
def test_forward_ragged_with_background(seed, W, H, C):
    s = scenes.random_small(seed, C=C, N=3000, W=W, H=H, sigma=(0.5, 10.0))
    iso, ref = _oracle_forward(s)
    compare_forward(ref, gpu_forward(s, scene_to_dev(s)), s)


def test_forward_masks():
    s = scenes.random_small(5, C=2, N=2000, W=96, H=64)
    rng = np.random.default_rng(0)
    masks = rng.integers(0, 2, (2, 4, 6)).astype(np.int32)
    iso, ref = _oracle_forward(s, masks=masks)
    got = gpu_forward(s, scene_to_dev(s), masks=masks)
    compare_forward(ref, got, s)


def test_forward_dense_stack_terminates():
    # heavy overlap: most pixels stop on the transmittance threshold
    s = scenes.random_small(6, C=1, N=6000, W=64, H=64, sigma=(3.0, 12.0), opacity=(0.5, 0.99))
    iso, ref = _oracle_forward(s)
    got = gpu_forward(s, scene_to_dev(s))
    compare_forward(ref, got, s)
    T = 1 - ref["render_alphas"]
    assert (T < s.transmittance_threshold).mean() > 0.5


def test_forward_empty_lists():
    s = scenes.random_small(7, C=1, N=10, W=64, H=48)
    s.means2d[:] = -500.0
    iso, ref = _oracle_forward(s)
    got = gpu_forward(s, scene_to_dev(s))
    compare_forward(ref, got, s)
    assert (got["last_ids"] == -1).all()


def _oracle_bwd_state(s, masks=None, absgrad=True, seed=1, nudges=1, fwd_ties=False):
    """Oracle forward and backward of the scene.  Splats whose backward alpha
    lies within TIE_ALPHA of the cutoff or the clamp (and, with fwd_ties, the
    splats of every near-tie decision of the forward) get their opacity
    scaled by 1 % (`nudges` rounds, a deterministic change of the seeded
    input that moves them off the decision).  Returns (iso, ref, rb, g_rgb,
    g_a)."""
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, channels=s.channels, seed=seed)
    for it in range(nudges + 1):
        iso, ref = _oracle_forward(s, masks=masks)
        rb = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds,
                                  masks, s.width, s.height, s.tile_size, iso["offsets"],
                                  iso["flatten_ids"], s.alpha_cutoff, ref["render_alphas"],
                                  ref["last_ids"], g_rgb, g_a, absgrad=absgrad,
                                  tie_rel=TIE_ALPHA, magnitudes=True)
        tie = rb["tie_splats"].astype(bool)
        if fwd_ties:
            tie |= ref["tie_splats"].astype(bool)
        if not tie.any() or it == nudges:
            break
        s.opacities[tie] *= np.where(s.opacities[tie] < 0.98, 1.01, 0.99).astype(np.float32)
    return iso, ref, rb, g_rgb, g_a


def _walked_splats(s, offsets, flatten_ids, pixels, lasts):
    """Splats at list positions start .. last of each given pixel (flat index
    (c H + y) W + x), for each array of last ids in `lasts`: a decision
    flipped at entry j of a pixel changes that pixel's terms for the splats
    at entries <= j."""
    excluded = np.zeros(s.C * s.N, bool)
    offs = offsets.reshape(-1)
    for p in pixels:
        c, rem = divmod(int(p), s.width * s.height)
        t = (c * s.tile_height + (rem // s.width) // 16) * s.tile_width + (rem % s.width) // 16
        last = max(int(l.reshape(-1)[p]) for l in lasts)
        if last >= offs[t]:
            excluded[flatten_ids[offs[t]:last + 1]] = True
    return excluded.reshape(s.C, s.N)


def _bwd_case(s, masks=None, absgrad=True, seed=1, nudges=1):
    """Oracle and GPU backward on the same (oracle) forward state.  The GPU
    backward re-decides every pair with the GPU's arithmetic, which is the
    GPU forward's: at the pixels flagged near a decision, the GPU forward's
    composited positions (from its trace) are compared with the oracle's,
    and the walked part of a pixel where they differ (or with a pair near
    the 0.99 clamp) is left out."""
    iso, ref, rb, g_rgb, g_a = _oracle_bwd_state(s, masks, absgrad, seed, nudges)
    d = scene_to_dev(s)
    # the GPU backward gets the oracle's forward state, so it is compared alone
    got = gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                              d["backgrounds"], to_dev(masks), s.width, s.height, s.tile_size,
                              to_dev(iso["offsets"]), to_dev(iso["flatten_ids"]), s.alpha_cutoff,
                              to_dev(ref["render_alphas"]), to_dev(ref["last_ids"]),
                              to_dev(g_rgb), to_dev(g_a), absgrad=absgrad)
    torch.cuda.synchronize()
    f, tr = _gpu_fwd_with_trace(s, d, masks=masks)
    excl_pix, flagged, flipped = flipped_pixels(ref, rb, tr, f, s.width, s.height)
    log_parity(kind="decisions", flagged_pixels=flagged, flipped_pixels=flipped,
               left_out_pixels=int(excl_pix.size))
    excluded = _walked_splats(s, iso["offsets"], iso["flatten_ids"], excl_pix,
                              [ref["last_ids"], f["last_ids"].cpu().numpy()])
    return rb, got, excluded


def _compare_grads(rb, got, excluded, rtol=1e-3, atol=1e-6, cancel_rel=1e-4, loose_rel=4e-6):
    """Strict bound |g - r| <= rtol |r| + atol on every element whose sum is
    not dominated by cancellation; elements whose |r| is below cancel_rel of
    the sum of |terms| (the float-summation error scale of any order) are held
    to loose_rel of that sum instead.  Returns (checked, cancellation-bound)
    counts."""
    stats = [0, 0]
    for name, mag, w in [("grad_means2d", "mag_means2d", 2), ("grad_conics", "mag_conics", 3),
                         ("grad_colors", "mag_colors", rb["grad_colors"].shape[-1]),
                         ("grad_opacities", "mag_opacities", 1)]:
        g = got[name].cpu().numpy().astype(np.float64)
        r = rb[name].astype(np.float64)
        m = rb[mag]
        keep = ~excluded if w == 1 else np.repeat(~excluded[..., None], w, axis=-1)
        g, r, m = g[keep], r[keep], m[keep]
        err = np.abs(g - r)
        cancel = np.abs(r) < cancel_rel * m
        strict_bad = (err > rtol * np.abs(r) + atol) & ~cancel
        assert not strict_bad.any(), (
            f"{name}: {strict_bad.sum()} of {g.size} off; worst err "
            f"{err[strict_bad].max()} (ref {r[strict_bad][np.argmax(err[strict_bad])]})")
        loose_bad = (err > loose_rel * m + atol) & cancel
        assert not loose_bad.any(), f"{name}: {loose_bad.sum()} cancellation-bound elements off"
        stats[0] += g.size
        stats[1] += int(cancel.sum())
    touched = int((rb["mag_opacities"] > 0).sum())
    log_parity(kind="backward", splats_with_terms=touched,
               excluded_splats=int((excluded & (rb["mag_opacities"] > 0)).sum()),
               elements_checked=stats[0], cancellation_bound_elements=stats[1])
    return stats


def test_backward_workload5():
    s = scenes.workload(5)
    rb, got, excluded = _bwd_case(s, absgrad=True)
    assert excluded.mean() < 0.02
    checked, cancel = _compare_grads(rb, got, excluded)
    assert cancel < 1e-3 * checked
    np.testing.assert_allclose(got["grad_means2d_abs"].cpu().numpy()[~excluded],
                               rb["grad_means2d_abs"][~excluded], rtol=1e-3, atol=1e-5)


@pytest.mark.parametrize("seed,W,H,C", [(0, 100, 70, 2), (2, 257, 129, 1)])
def test_backward_ragged_with_background(seed, W, H, C):
    s = scenes.random_small(seed, C=C, N=3000, W=W, H=H, sigma=(0.5, 10.0))
    rb, got, excluded = _bwd_case(s)
    _compare_grads(rb, got, excluded)
    np.testing.assert_allclose(got["grad_backgrounds"].cpu().numpy(), rb["grad_backgrounds"],
                               rtol=1e-4, atol=1e-3)


def test_many_cameras():
    # 37 small cameras (3 x 2 tiles each, the last row and column ragged):
    # tile -> camera indexing, per-camera backgrounds and their gradients,
    # and the keys' camera bits (6 of them) through the forward and backward
    s = scenes.random_small(12, C=37, N=300, W=40, H=24, sigma=(0.5, 6.0))
    iso, ref = _oracle_forward(s)
    compare_forward(ref, gpu_forward(s, scene_to_dev(s)), s)
    rb, got, excluded = _bwd_case(s)
    _compare_grads(rb, got, excluded)
    np.testing.assert_allclose(got["grad_backgrounds"].cpu().numpy(), rb["grad_backgrounds"],
                               rtol=1e-4, atol=1e-3)


def test_backward_masks_and_dense_stack():
    s = scenes.random_small(6, C=1, N=6000, W=64, H=64, sigma=(3.0, 12.0), opacity=(0.5, 0.99))
    masks = np.array([[[1, 0, 1, 1], [1, 1, 0, 1], [1, 1, 1, 1], [0, 1, 1, 1]]], np.int32)
    rb, got, excluded = _bwd_case(s, masks=masks)
    _compare_grads(rb, got, excluded)


def _gpu_fwd_with_trace(s, d, masks=None):
    f = gpu_forward(s, d, masks=masks)
    trace = torch.empty((f["flatten_ids"].numel(), 8), dtype=torch.int32, device=DEV)
    gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"], d["backgrounds"],
                        None if masks is None else to_dev(masks), s.width, s.height, 16,
                        f["offsets"], f["flatten_ids"], s.alpha_cutoff,
                        s.transmittance_threshold, trace=trace,
                        out=(f["render_colors"], f["render_alphas"], f["last_ids"]))
    return f, trace


def _chain_scene(case):
    if case == "w5":
        return scenes.workload(5), None
    s = scenes.random_small(3, C=2, N=4000, W=150, H=90, sigma=(0.5, 10.0))
    return s, np.random.default_rng(1).integers(0, 2, (2, 6, 10)).astype(np.int32)


@pytest.mark.parametrize("trace", [False, True])
@pytest.mark.parametrize("case", ["w5", "ragged_bg_masks"])
def test_forward_then_backward_on_gpu_state(case, trace):
    # the chain the bench times: the GPU forward's own render_alphas, last_ids
    # (and, with trace, its per-entry composite masks) feed the GPU backward.
    # The forward is compared with the oracle's forward; the backward with the
    # oracle's backward on the same (GPU) forward state, at 1e-3 rel + 1e-6.
    # (render_alpha near 1 carries a few ulp of the exponential's difference,
    # which the division-based T recovery turns into a relative error of
    # 1e-3 and more; the oracle's own forward state would compare the two
    # forwards a second time.)  Pixels flagged near a decision where the GPU's
    # composited positions differ from the oracle's are left out (counted)
    s, masks = _chain_scene(case)
    iso, ref, _, g_rgb, g_a = _oracle_bwd_state(s, masks=masks, absgrad=True, nudges=3,
                                                fwd_ties=True)
    d = scene_to_dev(s)
    f, tr = _gpu_fwd_with_trace(s, d, masks=masks)
    compare_forward(ref, f, s)
    got = gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                              d["backgrounds"], to_dev(masks), s.width, s.height, 16,
                              f["offsets"], f["flatten_ids"], s.alpha_cutoff, f["render_alphas"],
                              f["last_ids"], to_dev(g_rgb), to_dev(g_a), absgrad=True,
                              trace=tr if trace else None)
    torch.cuda.synchronize()
    rb = oracle.rasterize_bwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, masks,
                              s.width, s.height, 16, iso["offsets"], iso["flatten_ids"],
                              s.alpha_cutoff, f["render_alphas"].cpu().numpy(),
                              f["last_ids"].cpu().numpy(), g_rgb, g_a, absgrad=True,
                              tie_rel=TIE_ALPHA, magnitudes=True)
    excl_pix, flagged, flipped = flipped_pixels(ref, rb, tr, f, s.width, s.height)
    log_parity(kind="chain", flagged_pixels=flagged, flipped_pixels=flipped,
               left_out_pixels=int(excl_pix.size))
    excluded = _walked_splats(s, iso["offsets"], iso["flatten_ids"], excl_pix,
                              [ref["last_ids"], f["last_ids"].cpu().numpy()])
    touched = rb["mag_opacities"] > 0
    assert touched.sum() > 1000
    assert (excluded & touched).sum() <= 0.02 * touched.sum()
    checked, cancel = _compare_grads(rb, got, excluded)
    assert cancel < 1e-3 * checked
    np.testing.assert_allclose(got["grad_means2d_abs"].cpu().numpy()[~excluded],
                               rb["grad_means2d_abs"][~excluded], rtol=1e-3, atol=1e-5)
    if s.backgrounds is not None:
        np.testing.assert_allclose(got["grad_backgrounds"].cpu().numpy(),
                                   rb["grad_backgrounds"], rtol=1e-4, atol=1e-3)


def test_raster_argument_errors():
    s = scenes.random_small(1, C=1, N=10, W=32, H=32)
    d = scene_to_dev(s)
    off = torch.zeros((1, 2, 2), dtype=torch.int32, device=DEV)
    ids = torch.zeros(0, dtype=torch.int32, device=DEV)
    with pytest.raises(gs.GsError) as e:
        gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"], None, None,
                            32, 32, 8, off, ids, 1 / 255, 1e-4)
    assert e.value.code == 1


@pytest.mark.parametrize("case", ["w2", "ragged_bg_masks", "dense"])
def test_backward_trace_equals_recompute(case):
    # the trace only tells the backward which pairs to revisit: the gradients
    # must match the re-evaluating path up to the order of float atomics
    masks = None
    if case == "w2":
        s = scenes.workload(2)
    elif case == "ragged_bg_masks":
        s = scenes.random_small(3, C=2, N=4000, W=150, H=90, sigma=(0.5, 10.0))
        masks = np.random.default_rng(1).integers(0, 2, (2, 6, 10)).astype(np.int32)
    else:
        s = scenes.random_small(6, C=1, N=6000, W=64, H=64, sigma=(3.0, 12.0),
                                opacity=(0.5, 0.99))
    d = scene_to_dev(s)
    f, tr = _gpu_fwd_with_trace(s, d, masks=masks)
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=2)
    args = (d["means2d"], d["conics"], d["colors"], d["opacities"], d["backgrounds"],
            None if masks is None else to_dev(masks), s.width, s.height, 16, f["offsets"],
            f["flatten_ids"], s.alpha_cutoff, f["render_alphas"], f["last_ids"], to_dev(g_rgb),
            to_dev(g_a))
    a = gs.gs_rasterize_bwd(*args, absgrad=True)
    b = gs.gs_rasterize_bwd(*args, absgrad=True, trace=tr)
    for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities",
              "grad_means2d_abs", "grad_backgrounds"):
        if a[k] is None:
            continue
        x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
        scale = np.abs(x).max() + 1e-30
        np.testing.assert_allclose(y, x, rtol=1e-4, atol=1e-6 * scale, err_msg=k)


@pytest.mark.parametrize("cutoff,thr", [(0.0, 1e-4), (1.0 / 255.0, 0.0), (1.0 / 255.0, 0.999),
                                        (0.3, 0.5), (-1.0, 1e-4)])
def test_cutoff_and_threshold_extremes(cutoff, thr):
    # a zero or negative cutoff takes every pair with s >= 0 (alpha 0 included,
    # so last ids move on pairs that add nothing); threshold 0 never stops a
    # pixel, 0.999 stops it at its first composite; the trace-driven backward
    # must agree with the recomputing one under each setting
    s = scenes.random_small(11, C=2, N=1500, W=80, H=56, sigma=(0.5, 9.0))
    s.alpha_cutoff = np.float32(cutoff)
    s.transmittance_threshold = np.float32(thr)
    iso, ref = _oracle_forward(s)
    d = scene_to_dev(s)
    compare_forward(ref, gpu_forward(s, d), s)
    rb, got, excluded = _bwd_case(s, absgrad=False)
    if cutoff > 0:
        _compare_grads(rb, got, excluded)
    else:
        # without a positive cutoff every pixel of a splat's tile rectangle adds
        # a term, out to s of 20 and more, where the exponential's relative
        # error (2.4e-7 + 1e-7 s) reaches 1e-5 of a term: sums of |terms| near
        # 1e3 for results near 1 then carry errors of about 2e-5 of the sum
        _compare_grads(rb, got, excluded, cancel_rel=1e-3, loose_rel=4e-5)
    f, tr = _gpu_fwd_with_trace(s, d)
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=3)
    outs = []
    for trace in (None, tr):
        outs.append(gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                                        d["backgrounds"], None, s.width, s.height, 16,
                                        f["offsets"], f["flatten_ids"], s.alpha_cutoff,
                                        f["render_alphas"], f["last_ids"], to_dev(g_rgb),
                                        to_dev(g_a), trace=trace))
    torch.cuda.synchronize()
    for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities"):
        x, y = outs[0][k].cpu().numpy(), outs[1][k].cpu().numpy()
        np.testing.assert_allclose(y, x, rtol=1e-4, atol=1e-6 * (np.abs(x).max() + 1e-30),
                                   err_msg=k)
