"""Channel counts other than 3 (gs_rasterize_fwd / gs_rasterize_bwd take any
`channels`): parity against the oracle for 1, 2, 4 (one launch, chunk width
= channels) and 5, 7, 16, 33 (chunks of 4 plus a ragged chunk), and the
invariant that compositing decisions do not depend on the colours."""

import numpy as np
import pytest
import torch

from gpu_util import DEV, compare_forward, gpu_forward, scene_to_dev, to_dev
from test_gpu_raster import _bwd_case, _compare_grads, _gpu_fwd_with_trace, _oracle_forward
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu


def _scene(ch, seed=21, C=2, W=100, H=70, N=3000):
    return scenes.random_small(seed, C=C, N=N, W=W, H=H, sigma=(0.5, 10.0), channels=ch)


@pytest.mark.parametrize("ch", [1, 2, 4, 5, 7, 16, 33, 1024])
def test_forward_channels(ch):
    s = _scene(ch)
    iso, ref = _oracle_forward(s)
    got = gpu_forward(s, scene_to_dev(s))
    assert got["render_colors"].shape == (s.C, s.height, s.width, ch)
    compare_forward(ref, got, s)


def test_forward_decisions_independent_of_channels():
    # alphas, last ids, pair counts and the trace come from the geometry and
    # opacities only: a 7-channel render (two launches) and a 1-channel render
    # of the same splats must agree bit for bit on them
    s7 = _scene(7, seed=22)
    s1 = _scene(7, seed=22)
    s1.colors = np.ascontiguousarray(s7.colors[..., :1])
    s1.backgrounds = np.ascontiguousarray(s7.backgrounds[..., :1])
    out = []
    for s in (s7, s1):
        d = scene_to_dev(s)
        f = gpu_forward(s, d)
        # zeroed: words of entries after a tile has stopped are not written
        tr = torch.zeros((f["flatten_ids"].numel(), 8), dtype=torch.int32, device=DEV)
        counts = torch.empty((s.C, s.height, s.width, 3), dtype=torch.int32, device=DEV)
        gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"],
                            d["backgrounds"], None, s.width, s.height, 16, f["offsets"],
                            f["flatten_ids"], s.alpha_cutoff, s.transmittance_threshold,
                            pair_counts=counts, trace=tr,
                            out=(f["render_colors"], f["render_alphas"], f["last_ids"]))
        torch.cuda.synchronize()
        out.append((f, tr, counts))
    (f7, t7, c7), (f1, t1, c1) = out
    assert torch.equal(f7["render_alphas"], f1["render_alphas"])
    assert torch.equal(f7["last_ids"], f1["last_ids"])
    assert torch.equal(c7, c1)
    assert torch.equal(t7, t1)
    err = (f7["render_colors"][..., :1] - f1["render_colors"]).abs().max().item()
    assert err <= 1e-6


@pytest.mark.parametrize("ch,absgrad", [(1, True), (2, True), (4, True), (5, True),
                                        (7, True), (16, False), (16, True), (130, True)])
def test_backward_channels(ch, absgrad):
    # above 4 channels absgrad comes from its own full-channel pass
    s = _scene(ch, seed=23)
    rb, got, excluded = _bwd_case(s, absgrad=absgrad)
    _compare_grads(rb, got, excluded)
    assert got["grad_colors"].shape == (s.C, s.N, ch)
    # background gradient: a sum of g_rgb (1 - render_alpha) over every pixel
    gb = got["grad_backgrounds"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(gb, rb["grad_backgrounds"], rtol=1e-4,
                               atol=1e-6 * s.width * s.height)
    if absgrad:
        a = got["grad_means2d_abs"].cpu().numpy()[~excluded]
        r = rb["grad_means2d_abs"][~excluded]
        np.testing.assert_allclose(a, r, rtol=1e-3, atol=1e-6)


@pytest.mark.parametrize("ch", [2, 7])
def test_backward_channels_trace_equals_recompute(ch):
    # absgrad included: above 4 channels its full-channel pass reads the trace too
    s = _scene(ch, seed=24)
    d = scene_to_dev(s)
    f, tr = _gpu_fwd_with_trace(s, d)
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, channels=ch, seed=2)
    args = (d["means2d"], d["conics"], d["colors"], d["opacities"], d["backgrounds"], None,
            s.width, s.height, 16, f["offsets"], f["flatten_ids"], s.alpha_cutoff,
            f["render_alphas"], f["last_ids"], to_dev(g_rgb), to_dev(g_a))
    a = gs.gs_rasterize_bwd(*args, absgrad=True)
    b = gs.gs_rasterize_bwd(*args, absgrad=True, trace=tr)
    for k in ("grad_means2d", "grad_conics", "grad_colors", "grad_opacities",
              "grad_backgrounds", "grad_means2d_abs"):
        x, y = a[k].cpu().numpy(), b[k].cpu().numpy()
        scale = np.abs(x).max() + 1e-30
        np.testing.assert_allclose(y, x, rtol=1e-4, atol=1e-6 * scale, err_msg=k)


def test_channel_argument_errors():
    s = _scene(5, seed=25, C=1, W=32, H=32, N=50)
    d = scene_to_dev(s)
    f = gpu_forward(s, d)
    # more channels than GS_MAX_CHANNELS
    wide = torch.zeros((1, s.N, 1025), dtype=torch.float32, device=DEV)
    with pytest.raises(gs.GsError) as e:
        gs.gs_rasterize_fwd(d["means2d"], d["conics"], wide, d["opacities"], None, None, 32, 32,
                            16, f["offsets"], f["flatten_ids"], s.alpha_cutoff,
                            s.transmittance_threshold)
    assert e.value.code == 1
