"""The forward's per-entry composite masks (the trace gs_rasterize_fwd writes
for gs_rasterize_bwd) against the oracle's composited list positions.

For every pixel away from a near-tie decision, the bits of the entries up to
its last id are exactly the pairs the oracle composited there.  A warp (8
rows of a tile, trace words 4h .. 4h + 3) writes the words of every entry of
the 32-entry chunks it walked and no others: the words of entries after the
chunk in which all its pixels had stopped keep what the buffer held, and a
warp with no pixel inside the image, or in a masked tile, writes nothing."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, TIE_ALPHA, TIE_T, gpu_forward, log_parity, scene_to_dev, to_dev
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A5A5A  # what the buffer holds before the forward
CHUNK = 32             # entries a warp gathers at a time


def _expected_and_check(s, masks=None):
    d = scene_to_dev(s)
    f = gpu_forward(s, d, masks=masks)
    n = f["flatten_ids"].numel()
    trace = torch.full((n, 8), SENTINEL, dtype=torch.int32, device=DEV)
    gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"], d["backgrounds"],
                        None if masks is None else to_dev(masks), s.width, s.height, 16,
                        f["offsets"], f["flatten_ids"], s.alpha_cutoff,
                        s.transmittance_threshold, trace=trace,
                        out=(f["render_colors"], f["render_alphas"], f["last_ids"]))
    torch.cuda.synchronize()
    got = trace.cpu().numpy().view(np.uint32)
    offs = f["offsets"].cpu().numpy().reshape(-1).astype(np.int64)
    ids = f["flatten_ids"].cpu().numpy()
    TH, TW = s.tile_height, s.tile_width
    ntiles = s.C * TH * TW
    ends = np.append(offs[1:], n)
    max_list = int((ends - offs).max()) if ntiles else 0
    # the oracle's composited positions per pixel, in order (its step records)
    tpg, keys, o_ids = oracle.isect_tiles(s.means2d, s.radii, s.depths, s.tile_size, TW, TH)
    iso = dict(offsets=oracle.tile_offsets(keys, s.C, TW, TH), flatten_ids=o_ids)
    assert np.array_equal(iso["offsets"].reshape(-1), offs)
    assert np.array_equal(iso["flatten_ids"], ids)
    ref = oracle.rasterize_fwd(s.means2d, s.conics, s.colors, s.opacities, s.backgrounds, masks,
                               s.width, s.height, s.tile_size, iso["offsets"], iso["flatten_ids"],
                               s.alpha_cutoff, s.transmittance_threshold, tie_rel=TIE_ALPHA,
                               tie_rel_T=TIE_T, max_steps=max(max_list, 1))
    assert (ref["step_count"] <= max(max_list, 1)).all()
    near = ref["near_tie"] > 0
    gpu_last = f["last_ids"].cpu().numpy()
    assert np.array_equal(gpu_last[~near], ref["last_ids"][~near])
    T_final = 1.0 - ref["render_alphas"][..., 0]
    stats = dict(halves=0, halves_with_ties=0, entries_checked=0, unwritten_checked=0)
    for t in range(ntiles):
        c, rem = divmod(t, TH * TW)
        ty, tx = divmod(rem, TW)
        start, end = int(offs[t]), int(ends[t])
        masked = masks is not None and masks[c, ty, tx] == 0
        for h in range(2):
            words = got[start:end, 4 * h:4 * h + 4]
            ys = [y for y in range(16 * ty + 8 * h, 16 * ty + 8 * h + 8) if y < s.height]
            xs = [x for x in range(16 * tx, 16 * tx + 16) if x < s.width]
            if masked or not ys or not xs or end == start:
                # nothing walked: every word keeps the buffer's value
                assert (words == SENTINEL).all(), (t, h)
                continue
            stats["halves"] += 1
            exp = np.zeros((end - start, 4), np.uint32)
            keep = np.zeros(4, np.uint32)  # bits of pixels away from near ties
            stops, nonnear_last, has_tie = [], start - 1, False
            for y in ys:
                for x in xs:
                    q = 16 * ((y % 16) // 4) + x % 16
                    w, b = (y % 16) % 4, q % 32
                    cnt = int(ref["step_count"][c, y, x])
                    pos = ref["step_pos"][:cnt, c, y, x].astype(np.int64)
                    assert ((pos >= start) & (pos < end)).all()
                    if near[c, y, x]:
                        has_tie = True
                        continue
                    keep[w] |= np.uint32(1 << b)
                    exp[pos - start, w] |= np.uint32(1 << b)
                    last = int(ref["last_ids"][c, y, x])
                    nonnear_last = max(nonnear_last, last)
                    # the pixel stops at its last composite if T fell below the
                    # threshold there; else it walks the whole list
                    stopped = cnt > 0 and T_final[c, y, x] < s.transmittance_threshold
                    stops.append(last if stopped else end - 1)
            if has_tie:
                stats["halves_with_ties"] += 1
                # the warp walked at least to every other pixel's last composite
                upto = nonnear_last + 1
            else:
                s_max = max(stops)
                upto = min(end, start + CHUNK * ((s_max - start) // CHUNK + 1))
                assert (words[upto - start:] == SENTINEL).all(), (t, h, upto)
                stats["unwritten_checked"] += end - upto
            sel = slice(0, upto - start)
            assert np.array_equal(words[sel] & keep, exp[sel] & keep), (t, h)
            stats["entries_checked"] += upto - start
    log_parity(kind="trace", **stats)
    return stats


def test_trace_dense_stack_stops_early():
    # heavy overlap: most pixels stop early, so most warps leave a tail of
    # their list unwritten
    s = scenes.random_small(6, C=1, N=6000, W=64, H=64, sigma=(3.0, 12.0), opacity=(0.5, 0.99))
    st = _expected_and_check(s)
    assert st["unwritten_checked"] > 0 and st["entries_checked"] > 0


def test_trace_ragged_masks_two_cameras():
    # ragged image (the last tile row's second half lies outside), masked
    # tiles, background
    s = scenes.random_small(3, C=2, N=4000, W=150, H=90, sigma=(0.5, 10.0))
    masks = np.random.default_rng(1).integers(0, 2, (2, 6, 10)).astype(np.int32)
    st = _expected_and_check(s, masks=masks)
    assert st["entries_checked"] > 0


def test_trace_threshold_never_stops():
    # threshold 0: no pixel stops, every warp walks and writes its whole list
    s = scenes.random_small(11, C=1, N=1500, W=80, H=56, sigma=(0.5, 9.0))
    s.transmittance_threshold = np.float32(0.0)
    st = _expected_and_check(s)
    assert st["unwritten_checked"] == 0 and st["entries_checked"] > 0
