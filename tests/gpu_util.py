"""Helpers shared by the GPU parity tests: move a scene to the device, run
the library's path through the binding, and compare with the oracle."""

from __future__ import annotations

import os

import numpy as np
import torch

from tile_gaussian_splat_gb300 import binding as gs

DEV = "cuda:0"

# near-tie margins: at pixels where the oracle took a skip/stop decision
# within this relative distance of its threshold, the decision may go the
# other way on the GPU, so those pixels are held to the bound such a flip
# allows (tie_bound) instead of exactly.  alpha vs the cutoff: libm expf and
# the GPU's ex2-based exponential differ by a few ulp (< 1e-6 relative) and s
# is computed in the same rounding order on both sides.  T vs the threshold:
# T carries every 1 - alpha, whose relative error is alpha / (1 - alpha) times
# alpha's (1e-4 for alpha = 0.99).
TIE_ALPHA = 1e-5
TIE_T = 1e-3
RGBA_ATOL = 1e-5


def to_dev(a, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV)


def scene_to_dev(s):
    return {k: to_dev(v) for k, v in s.arrays().items()}


def u64(t):
    """int64 tensor holding uint64 bits -> numpy uint64."""
    return t.cpu().numpy().view(np.uint64)


def gpu_isect(s, d, sort=True, status=None):
    return gs.gs_isect_tiles(d["means2d"], d["radii"], d["depths"], s.tile_size, s.tile_width,
                             s.tile_height, sort=sort, d_status=status)


def gpu_forward(s, d, masks=None, status=None):
    st = status if status is not None else gs.new_status(DEV)
    tpg, keys, ids = gpu_isect(s, d, status=st)
    offsets = gs.gs_tile_offsets(keys, s.C, s.tile_width, s.tile_height, d_status=st)
    rgb, alpha, last = gs.gs_rasterize_fwd(
        d["means2d"], d["conics"], d["colors"], d["opacities"], d["backgrounds"],
        None if masks is None else to_dev(masks), s.width, s.height, s.tile_size, offsets, ids,
        s.alpha_cutoff, s.transmittance_threshold, d_status=st)
    gs.check_status(st)
    return dict(tiles_per_gauss=tpg, keys=keys, flatten_ids=ids, offsets=offsets,
                render_colors=rgb, render_alphas=alpha, last_ids=last)


# What the parity tests left out or checked at a looser bound, one record per
# comparison; printed at the end of the run (tests/conftest.py).
PARITY_LOG = []


def log_parity(**rec):
    rec["test"] = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    PARITY_LOG.append(rec)


def tie_bound(scene, n_ties):
    """Largest RGBA difference that n_ties flipped decisions can make at one
    pixel.  A flipped cutoff decision at pair j (alpha_j within TIE_ALPHA of
    the cutoff) adds or drops T_j alpha_j colour_j and scales everything
    behind it by 1 - alpha_j: at most 2 cutoff M with M the largest colour or
    background magnitude (T <= 1); it can also move the stop, which changes at
    most the T < threshold remainder: threshold M.  A flipped stop decision (T
    within TIE_T of the threshold) changes only that remainder."""
    cut = max(float(scene.alpha_cutoff), 0.0)
    thr = max(float(scene.transmittance_threshold), 0.0)
    M = max(1.0, float(np.abs(scene.colors).max()) if scene.colors.size else 1.0,
            float(np.abs(scene.backgrounds).max()) if scene.backgrounds is not None else 0.0)
    per = (2.0 * cut * (1.0 + TIE_ALPHA) + (1.0 + TIE_T) * thr) * M
    return n_ties.astype(np.float64) * per + RGBA_ATOL


def compare_forward(ref, got, scene, pixels=None, tie=None):
    """Exact last_ids and RGBA within 1e-5 at every pixel without a near tie.
    At a pixel where the oracle took n decisions within the tie margins, RGBA
    is held to tie_bound(n) and the last id to a position of the tile's list
    (or -1).  Returns the number of near-tie pixels."""
    rgb = got["render_colors"].cpu().numpy()
    alpha = got["render_alphas"].cpu().numpy()
    last = got["last_ids"].cpu().numpy()
    tie = ref["near_tie"] if tie is None else tie
    sel = np.ones(tie.shape, bool)
    if pixels is not None:
        sel = np.zeros(tie.size, bool)
        sel[pixels] = True
        sel = sel.reshape(tie.shape)
    ok = (tie == 0) & sel
    near = (tie > 0) & sel
    assert ok.sum() > 0
    np.testing.assert_array_equal(last[ok], ref["last_ids"][ok])
    err_rgb = np.abs(rgb[ok] - ref["render_colors"][ok]).max()
    err_a = np.abs(alpha[..., 0][ok] - ref["render_alphas"][..., 0][ok]).max()
    assert err_rgb <= RGBA_ATOL, f"rgb max abs err {err_rgb}"
    assert err_a <= RGBA_ATOL, f"alpha max abs err {err_a}"
    worst, worst_bound = 0.0, 0.0
    if near.any():
        bound = tie_bound(scene, tie[near])
        e = np.maximum(np.abs(rgb[near] - ref["render_colors"][near]).max(axis=-1),
                       np.abs(alpha[..., 0][near] - ref["render_alphas"][..., 0][near]))
        assert (e <= bound).all(), (f"near-tie pixel off by {e[e > bound].max()} > bound "
                                    f"{bound[e > bound].min()}")
        worst, worst_bound = float(e.max()), float(bound[np.argmax(e)])
        if "offsets" in got and "flatten_ids" in got:
            offs = got["offsets"].cpu().numpy().reshape(-1).astype(np.int64)
            n = got["flatten_ids"].numel()
            ends = np.append(offs[1:], n)
            C, H, W = tie.shape
            cc, yy, xx = np.nonzero(near)
            t = (cc * ((H + 15) // 16) + yy // 16) * ((W + 15) // 16) + xx // 16
            lv = last[near]
            assert ((lv == -1) | ((lv >= offs[t]) & (lv < ends[t]))).all()
    log_parity(kind="forward", pixels=int(sel.sum()), near_tie_pixels=int(near.sum()),
               near_tie_max_err=worst, near_tie_bound_there=worst_bound)
    return int(near.sum())


def grad_tolerance_check(name, got, ref, rtol=1e-3, atol=1e-6, mask=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    err = np.abs(got - ref)
    bad = err > rtol * np.abs(ref) + atol
    assert not bad.any(), (f"{name}: {bad.sum()} of {bad.size} outside {rtol} rel + {atol}; "
                           f"worst err {err[bad].max()} at ref {ref[bad][np.argmax(err[bad])]}")


_FNV_BASIS = 14695981039346656037
_FNV_PRIME = 1099511628211


def gpu_comp_hash(trace, offsets, last_ids, pixels, width, height):
    """For each flat pixel index p = (c H + y) W + x in `pixels`, the FNV-1a
    hash (the oracle's comp_hash) of the list positions the GPU forward
    composited there, read from its trace: word 4 (q / 32) + y % 4 of entry
    j, bit q % 32, with q = 16 ((y % 16) / 4) + x % 16 (the layout
    gs_rasterize_fwd documents).  Only entries up to the pixel's last id are
    read (later words may be unwritten)."""
    TW, TH = (width + 15) // 16, (height + 15) // 16
    offs = offsets.reshape(-1).cpu().numpy().astype(np.int64)
    last = last_ids.reshape(-1).cpu().numpy()
    out = {}
    for p in np.asarray(pixels, np.int64).tolist():
        c, rem = divmod(p, width * height)
        y, x = divmod(rem, width)
        t = (c * TH + y // 16) * TW + x // 16
        start, lj = int(offs[t]), int(last[p])
        h = _FNV_BASIS
        if lj >= start:
            rows = trace[start:lj + 1].cpu().numpy().view(np.uint32)
            q = 16 * ((y % 16) // 4) + x % 16
            bits = (rows[:, 4 * (q // 32) + (y % 16) % 4] >> np.uint32(q % 32)) & np.uint32(1)
            for j in (start + np.nonzero(bits)[0]).tolist():
                h = ((h ^ j) * _FNV_PRIME) % (1 << 64)
        out[p] = h
    return out


def flipped_pixels(ref, rb, trace, got, width, height):
    """Pixels to leave out of a GPU-forward -> GPU-backward comparison: those
    flagged near a decision by the oracle's forward or backward where the
    GPU's composited positions (from its trace) differ from the oracle's
    (comp_hash), and those with a pair near the 0.99 clamp in the oracle's
    backward (high bits of its near_tie), where the clamp's gradient switch
    may flip.  Returns (pixels, flagged count, flipped count)."""
    flagged = np.nonzero(((rb["near_tie"] > 0) | (ref["near_tie"] > 0)).reshape(-1))[0]
    gh = gpu_comp_hash(trace, got["offsets"], got["last_ids"], flagged, width, height)
    rh = ref["comp_hash"].reshape(-1)
    flipped = np.array([p for p in flagged.tolist() if gh[p] != int(rh[p])], np.int64)
    clamp = np.nonzero((rb["near_tie"].reshape(-1) >> 4) > 0)[0]
    return np.union1d(flipped, clamp), int(flagged.size), int(flipped.size)
