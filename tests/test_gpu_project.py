"""GPU parity of gs_project (EWA projection) against the oracle: every output
bit for bit (both sides evaluate the same IEEE single-precision operations
in the same order), on an edge-case scene, both camera models, and at the
full 4-camera x 1M-Gaussian size the bench times; then the projected
splats through the whole raster path against the oracle's."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, TIE_ALPHA, TIE_T, compare_forward, gpu_forward, to_dev
from tile_gaussian_splat_gb300 import binding as gs
from tile_gaussian_splat_gb300 import scenes

pytestmark = pytest.mark.gpu


def _same_bits(got, ref, name):
    """Bitwise equal, except that any NaN matches any NaN (payloads differ
    between CPUs and GPUs)."""
    g = np.ascontiguousarray(got)
    r = np.ascontiguousarray(ref)
    assert g.shape == r.shape, name
    if g.dtype == np.float32:
        nan = np.isnan(g) & np.isnan(r)
        gb, rb = g.view(np.uint32), r.view(np.uint32)
        bad = (gb != rb) & ~nan
    else:
        bad = g != r
    assert not bad.any(), (f"{name}: {bad.sum()} of {bad.size} differ; first at "
                           f"{np.argwhere(bad)[0]}: {g[bad][0]!r} vs {r[bad][0]!r}")


def _gpu_project(s, **kw):
    return gs.gs_project(to_dev(s.means), to_dev(s.covars), to_dev(s.viewmats),
                         to_dev(s.intrinsics), s.width, s.height, eps2d=s.eps2d,
                         near_plane=s.near_plane, far_plane=s.far_plane,
                         radius_clip=s.radius_clip, **kw)


def _check(s, orthographic=False, **params):
    for k, v in params.items():
        setattr(s, k, v)
    got = _gpu_project(s, compensation=True, orthographic=orthographic, radii_float=True)
    torch.cuda.synchronize()
    ref = oracle.project(s.means, s.covars, s.viewmats, s.intrinsics, s.width, s.height,
                         eps2d=s.eps2d, near_plane=s.near_plane, far_plane=s.far_plane,
                         radius_clip=s.radius_clip, compensation=True, orthographic=orthographic)
    for k in ("radii", "means2d", "depths", "conics", "compensations"):
        _same_bits(got[k].cpu().numpy(), ref[k], k)
    _same_bits(got["radii_float"].cpu().numpy(), ref["radii"].astype(np.float32), "radii_float")
    return ref


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("orthographic", [False, True])
def test_project_edge_cases_bit_exact(seed, orthographic):
    s = scenes.scene3d_edge(seed=seed)
    ref = _check(s, orthographic=orthographic)
    if not orthographic:
        vis = ref["radii"][..., 0] > 0
        assert 0.3 < vis.mean() < 0.95        # both visible and culled pairs
        assert (ref["radii"] == 2**31 - 1).any()  # the saturating branch ran
        assert np.isnan(ref["conics"]).any()      # an overflowing determinant too


@pytest.mark.parametrize("params", [dict(eps2d=0.0), dict(radius_clip=3.0),
                                    dict(near_plane=2.5, far_plane=6.0)])
def test_project_parameters_bit_exact(params):
    _check(scenes.scene3d_edge(seed=3, N=3000), **params)


def test_project_ragged_and_many_cameras():
    # N not a multiple of the block, more cameras than one shared-memory chunk
    base = scenes.scene3d(seed=4, C=37, N=1001, W=320, H=240, focal=280.0)
    _check(base)


def test_project_empty_and_errors():
    s = scenes.scene3d_edge(seed=0, N=64)
    d = {k: to_dev(getattr(s, k)) for k in ("means", "covars", "viewmats", "intrinsics")}
    empty = gs.gs_project(d["means"][:0], d["covars"][:0], d["viewmats"], d["intrinsics"],
                          s.width, s.height)
    assert empty["radii"].shape == (2, 0, 2)
    # means2d must be 8-byte aligned (float2 stores)
    out = dict(radii=torch.empty((2, 64, 2), dtype=torch.int32, device=DEV),
               means2d=torch.empty(2 * 64 * 2 + 1, device=DEV)[1:].view(2, 64, 2),
               depths=torch.empty((2, 64), device=DEV),
               conics=torch.empty((2, 64, 3), device=DEV), compensations=None, radii_float=None)
    with pytest.raises(gs.GsError) as e:
        gs.gs_project(d["means"], d["covars"], d["viewmats"], d["intrinsics"], s.width,
                      s.height, out=out)
    assert e.value.code == 1


@pytest.mark.slow
def test_project_full_size_bit_exact():
    # the configuration the bench times: 4 cameras x 1M Gaussians, 1920x1080
    _check(scenes.scene3d())


def test_projected_scene_through_the_raster_path():
    s = scenes.scene3d(seed=6, C=2, N=20_000, W=320, H=200, focal=330.0)
    rng = np.random.default_rng(6)
    colors = np.ascontiguousarray(np.broadcast_to(rng.uniform(0, 1, (1, s.N, 3)), (s.C, s.N, 3)),
                                  dtype=np.float32)
    opac = np.ascontiguousarray(np.broadcast_to(rng.uniform(0.05, 0.95, (1, s.N)), (s.C, s.N)),
                                dtype=np.float32)
    got = _gpu_project(s, radii_float=True)
    ref = oracle.project(s.means, s.covars, s.viewmats, s.intrinsics, s.width, s.height,
                         eps2d=s.eps2d, near_plane=s.near_plane, far_plane=s.far_plane,
                         radius_clip=s.radius_clip)
    scene2d = scenes.Scene(name="projected", C=s.C, N=s.N, width=s.width, height=s.height,
                           tile_size=16, means2d=ref["means2d"],
                           radii=ref["radii"].astype(np.float32), depths=ref["depths"],
                           conics=ref["conics"], colors=colors, opacities=opac, backgrounds=None)
    # the GPU path consumes the GPU projection's own outputs
    d = dict(means2d=got["means2d"], radii=got["radii_float"], depths=got["depths"],
             conics=got["conics"], colors=to_dev(colors), opacities=to_dev(opac),
             backgrounds=None)
    out = gpu_forward(scene2d, d)
    iso, fwd = oracle.render(scene2d, tie_rel=TIE_ALPHA, tie_rel_T=TIE_T)
    np.testing.assert_array_equal(out["flatten_ids"].cpu().numpy(), iso["flatten_ids"])
    np.testing.assert_array_equal(out["offsets"].cpu().numpy(), iso["offsets"])
    compare_forward(fwd, out, scene2d)
    assert (fwd["render_alphas"] > 0.5).mean() > 0.05  # the scene covers the images
