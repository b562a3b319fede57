"""Helpers shared by the GPU parity tests: move a scene to the device, run
the library's path through the binding, and compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

from tile_gaussian_splat_gb300 import binding as gs

DEV = "cuda:0"

# near-tie margins: pixels where the oracle took a skip/stop decision within
# this relative distance of its threshold are left out of the exact
# comparisons.  alpha vs the cutoff: libm expf and __expf differ by a few ulp
# (< 1e-6 relative) and s is computed in the same rounding order on both
# sides.  T vs the threshold: T carries every 1 - alpha, whose relative error
# is alpha / (1 - alpha) times alpha's (1e-4 for alpha = 0.99).
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


def compare_forward(ref, got, pixels=None, tie=None):
    """Exact last_ids and 1e-5 RGBA on pixels without a near tie.  Returns the
    number of near-tie pixels left out."""
    rgb = got["render_colors"].cpu().numpy()
    alpha = got["render_alphas"].cpu().numpy()
    last = got["last_ids"].cpu().numpy()
    tie = ref["near_tie"] if tie is None else tie
    ok = tie == 0
    if pixels is not None:
        sel = np.zeros(ok.size, bool)
        sel[pixels] = True
        ok = ok & sel.reshape(ok.shape)
    assert ok.sum() > 0
    np.testing.assert_array_equal(last[ok], ref["last_ids"][ok])
    err_rgb = np.abs(rgb[ok] - ref["render_colors"][ok]).max()
    err_a = np.abs(alpha[..., 0][ok] - ref["render_alphas"][..., 0][ok]).max()
    assert err_rgb <= RGBA_ATOL, f"rgb max abs err {err_rgb}"
    assert err_a <= RGBA_ATOL, f"alpha max abs err {err_a}"
    return int((~(tie == 0)).sum())


def grad_tolerance_check(name, got, ref, rtol=1e-3, atol=1e-6, mask=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    err = np.abs(got - ref)
    bad = err > rtol * np.abs(ref) + atol
    assert not bad.any(), (f"{name}: {bad.sum()} of {bad.size} outside {rtol} rel + {atol}; "
                           f"worst err {err[bad].max()} at ref {ref[bad][np.argmax(err[bad])]}")
