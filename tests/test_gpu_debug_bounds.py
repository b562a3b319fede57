"""The range-checking build (GS_DEBUG_BOUNDS, libgs_splat_gb300_debug.so):
on valid inputs it gives the release build's results bit for bit and keeps
the status word at 0; where an index read from the inputs is out of range
(a flatten id beyond C*N, a tile range past n_isects) it skips the access,
as every build does, and also reports GS_ERR_OUT_OF_BOUNDS -- nothing traps."""

import numpy as np
import pytest
import torch

from gpu_util import DEV, gpu_forward, scene_to_dev, to_dev
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import build, scenes

pytestmark = pytest.mark.gpu


def _fwd(s, d, offsets, ids, status):
    return gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                               d["backgrounds"], None, s.width, s.height, 16, offsets, ids,
                               s.alpha_cutoff, s.transmittance_threshold, d_status=status)


def test_range_checking_build():
    build.build()
    s = scenes.random_small(4, C=2, N=2000, W=96, H=64, sigma=(0.5, 10.0))
    d = scene_to_dev(s)
    ref = gpu_forward(s, d)
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=1)
    bwd_args = lambda f: (d["means2d"], d["conics"], d["colors"], d["opacities"],
                          d["backgrounds"], None, s.width, s.height, 16, f["offsets"],
                          f["flatten_ids"], s.alpha_cutoff, f["render_alphas"], f["last_ids"],
                          to_dev(g_rgb), to_dev(g_a))
    rb = gs.gs_rasterize_bwd(*bwd_args(ref))
    bad_ids = ref["flatten_ids"].clone()
    bad_ids[5] = s.C * s.N + 7
    bad_offs = ref["offsets"].clone()
    bad_offs.view(-1)[1] = ref["flatten_ids"].numel() + 100
    with gs.library(gs.LIB_DEBUG_PATH):
        st = gs.new_status(DEV)
        got = gpu_forward(s, d, status=st)  # raises on a nonzero status
        for k in ("tiles_per_gauss", "keys", "flatten_ids", "offsets", "render_colors",
                  "render_alphas", "last_ids"):
            assert torch.equal(got[k], ref[k]), k
        gb = gs.gs_rasterize_bwd(*bwd_args(got), d_status=st)
        gs.check_status(st)
        for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities"):
            x, y = rb[k].cpu().numpy(), gb[k].cpu().numpy()
            np.testing.assert_allclose(y, x, rtol=1e-4, atol=1e-6 * np.abs(x).max(), err_msg=k)
        for offs, ids in ((ref["offsets"], bad_ids), (bad_offs, ref["flatten_ids"])):
            st = gs.new_status(DEV)
            _fwd(s, d, offs, ids, st)
            assert int(st.item()) == 9  # GS_ERR_OUT_OF_BOUNDS
    # the release build skips the same accesses without a report
    for offs, ids in ((ref["offsets"], bad_ids), (bad_offs, ref["flatten_ids"])):
        st = gs.new_status(DEV)
        _fwd(s, d, offs, ids, st)
        assert int(st.item()) == 0
