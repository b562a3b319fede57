"""Pins of the oracle's EWA projection (gsplat 1.0.0,
data/ext/gsplat_native/projection.c, gs_project_one) against what the
mathematics fixes, independently of the oracle's own formulas:

  * the pinhole map K p / p.z of the camera-space mean (any K, any pose);
  * the linearisation: the covariance of many sampled 3D points pushed
    through the exact pinhole map approaches J S J^T for small Gaussians
    (pins R Sigma R^T against R^T Sigma R, the view-matrix layout, and the
    Jacobian's entries and signs);
  * closed forms on the optical axis (isotropic, and rotated about the
    axis for the conic's off-diagonal sign), at the frustum clip and for the
    orthographic camera; compensation as the square root of a determinant
    ratio;
  * invariance under a rigid motion applied to the world and the camera;
  * the visibility rules (near/far, radius_clip, image overlap, det <= 0)
    and the saturating radius reading.
"""

import math

import numpy as np
import pytest

import oracle
from tile_gaussian_splat_gb300 import scenes


def _K(fx, fy, cx, cy, skew=0.0):
    return np.array([[fx, skew, cx], [0.0, fy, cy], [0.0, 0.0, 1.0]], np.float64)


def _V(R=None, t=(0.0, 0.0, 0.0)):
    V = np.eye(4)
    if R is not None:
        V[:3, :3] = R
    V[:3, 3] = t
    return V


def _proj(means, covars, V, K, W=640, H=480, **kw):
    return oracle.project(np.atleast_2d(means), np.asarray(covars).reshape(-1, 3, 3),
                          np.asarray(V)[None], np.asarray(K)[None], W, H, **kw)


def _cov2d(out, eps2d):
    """Covariance (with eps2d) recovered from the conic, and without it."""
    a, b, c = (out["conics"][0, :, i].astype(np.float64) for i in range(3))
    det = a * c - b * b
    cov = np.stack([c / det, -b / det, -b / det, a / det], -1).reshape(-1, 2, 2)
    return cov, cov - eps2d * np.eye(2)


@pytest.mark.parametrize("z,s,fx,fy,eps", [(5.0, 0.1, 1000.0, 800.0, 0.3),
                                           (2.0, 0.02, 500.0, 500.0, 0.0),
                                           (40.0, 1.5, 1200.0, 900.0, 0.1)])
def test_on_axis_isotropic_closed_form(z, s, fx, fy, eps):
    # a Gaussian on the optical axis: centre at the principal point, 2D
    # covariance diag((fx s / z)^2, (fy s / z)^2) + eps2d
    K = _K(fx, fy, 320.0, 240.0)
    out = _proj([0.0, 0.0, z], np.eye(3) * s * s, _V(), K, eps2d=eps, compensation=True)
    np.testing.assert_array_equal(out["means2d"][0, 0], [320.0, 240.0])
    assert out["depths"][0, 0] == np.float32(z)
    vx, vy = (fx * s / z) ** 2 + eps, (fy * s / z) ** 2 + eps
    np.testing.assert_allclose(out["conics"][0, 0], [1 / vx, 0.0, 1 / vy], rtol=2e-6, atol=1e-12)
    for v, r in ((vx, out["radii"][0, 0, 0]), (vy, out["radii"][0, 0, 1])):
        exact = 3.33 * math.sqrt(v)
        assert abs(exact - round(exact)) > 1e-3  # not at a rounding boundary
        assert r == math.ceil(exact)
    comp = math.sqrt(((fx * s / z) ** 2 * (fy * s / z) ** 2) / (vx * vy))
    assert out["compensations"][0, 0] == pytest.approx(comp, rel=1e-5)


def test_means2d_is_the_pinhole_map():
    rng = np.random.default_rng(0)
    n = 500
    R = scenes.random_rotations(rng, 1)[0]
    V = _V(R, rng.uniform(-1, 1, 3) + [0, 0, 6])
    K = _K(700.0, 650.0, 300.0, 200.0, skew=3.0)
    K[1, 0] = 0.0
    means = rng.uniform(-1.5, 1.5, (n, 3))
    out = _proj(means, np.tile(np.eye(3) * 1e-4, (n, 1, 1)), V, K)
    p = means @ R.T + V[:3, 3]
    uv = (p @ K.T)[:, :2] / p[:, 2:3]
    np.testing.assert_allclose(out["means2d"][0], uv, rtol=1e-5, atol=1e-3)
    np.testing.assert_allclose(out["depths"][0], p[:, 2], rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_covariance_is_the_linearised_pinhole_map(seed):
    # sample the 3D Gaussian, push every sample through the exact pinhole map
    # and compare the samples' 2D covariance with the oracle's (eps2d = 0)
    rng = np.random.default_rng(seed)
    R = scenes.random_rotations(rng, 1)[0]
    V = _V(R, [0.3, -0.2, 5.0])
    K = _K(900.0, 800.0, 320.0, 240.0)
    mean = rng.uniform(-0.4, 0.4, 3)
    A = rng.standard_normal((3, 3)) * 0.01          # anisotropic, rotated
    Sigma = A @ A.T
    out = _proj(mean, Sigma, V, K, eps2d=0.0)
    _, cov = _cov2d(out, 0.0)
    x = rng.multivariate_normal(mean, Sigma, 400_000)
    p = x @ R.T + V[:3, 3]
    uv = np.stack([K[0, 0] * p[:, 0] / p[:, 2] + K[0, 2], K[1, 1] * p[:, 1] / p[:, 2] + K[1, 2]], 1)
    emp = np.cov(uv.T)
    # sampling error ~ sqrt(2 / n) = 0.2 %, linearisation error ~ sigma / z
    scale = math.sqrt(emp[0, 0] * emp[1, 1])
    np.testing.assert_allclose(cov[0], emp, rtol=0, atol=0.02 * scale)
    # the transposed rotation gives a different covariance: the pin has power
    wrong = _proj(mean, R.T @ R.T @ Sigma @ R @ R, V, K, eps2d=0.0)
    assert np.abs(_cov2d(wrong, 0.0)[1][0] - emp).max() > 0.1 * scale


@pytest.mark.parametrize("theta", [0.3, 1.2, 2.5])
def test_conic_of_rotated_on_axis_gaussian(theta):
    # on the optical axis with fx = fy = f, a Gaussian rotated about z by
    # theta projects to (f/z)^2 R2 diag(a^2, b^2) R2^T + eps2d I; the conic is
    # its inverse as (a, b, c) of [[a, b], [b, c]]
    f, z, sa, sb, sc, eps = 600.0, 4.0, 0.08, 0.02, 0.05, 0.3
    ct, st = math.cos(theta), math.sin(theta)
    Rz = np.array([[ct, -st, 0.0], [st, ct, 0.0], [0.0, 0.0, 1.0]])
    Sigma = Rz @ np.diag([sa * sa, sb * sb, sc * sc]) @ Rz.T
    out = _proj([0.0, 0.0, z], Sigma, _V(), _K(f, f, 320.0, 240.0), eps2d=eps)
    cov = (f / z) ** 2 * (Rz[:2, :2] @ np.diag([sa * sa, sb * sb]) @ Rz[:2, :2].T) + eps * np.eye(2)
    inv = np.linalg.inv(cov)
    np.testing.assert_allclose(out["conics"][0, 0], [inv[0, 0], inv[0, 1], inv[1, 1]],
                               rtol=1e-5, atol=1e-7)


def test_frustum_clip_closed_form():
    # beyond the widened image edge the Jacobian uses the clamped x/z:
    # cov_xx = (fx / z)^2 s_x^2 + (fx L / z)^2 s_z^2 with L the clamp limit
    W, H, fx, fy, cx, cy = 640, 480, 500.0, 500.0, 320.0, 240.0
    z, sx, sz = 4.0, 0.05, 0.2
    L = (W - cx) / fx + 0.15 * W / fx
    Sigma = np.diag([sx * sx, 1e-4, sz * sz])
    for x in (L * z * 1.5, L * z * 0.5):
        out = _proj([x, 0.0, z], Sigma, _V(), _K(fx, fy, cx, cy), W, H, eps2d=0.0)
        _, cov = _cov2d(out, 0.0)
        u = min(x / z, L)
        want = (fx / z) ** 2 * sx * sx + (fx * u / z) ** 2 * sz * sz
        assert cov[0, 0, 0] == pytest.approx(want, rel=1e-4)
    # and on the low side
    Lo = -(cx / fx + 0.15 * W / fx)
    out = _proj([Lo * z * 2.0, 0.0, z], Sigma, _V(), _K(fx, fy, cx, cy), W, H, eps2d=0.0)
    _, cov = _cov2d(out, 0.0)
    want = (fx / z) ** 2 * sx * sx + (fx * Lo / z) ** 2 * sz * sz
    assert cov[0, 0, 0] == pytest.approx(want, rel=1e-4)


def test_orthographic_closed_form():
    rng = np.random.default_rng(7)
    n = 200
    R = scenes.random_rotations(rng, 1)[0]
    V = _V(R, [0.1, 0.2, 3.0])
    K = _K(120.0, 110.0, 320.0, 240.0)
    means = rng.uniform(-1, 1, (n, 3))
    A = rng.standard_normal((n, 3, 3)) * 0.05
    Sigma = A @ np.transpose(A, (0, 2, 1))
    out = oracle.project(means, Sigma, V[None], K[None], 640, 480, eps2d=0.0,
                         orthographic=True)
    p = means @ R.T + V[:3, 3]
    np.testing.assert_allclose(out["means2d"][0], p[:, :2] * [120.0, 110.0] + [320.0, 240.0],
                               rtol=1e-5, atol=1e-3)
    J = np.array([[120.0, 0, 0], [0, 110.0, 0]])
    want = J @ R @ Sigma @ R.T @ J.T
    _, cov = _cov2d(out, 0.0)
    np.testing.assert_allclose(cov, want, rtol=2e-3, atol=1e-3 * np.abs(want).max())


def test_rigid_motion_invariance():
    # moving the world by Q and the camera with it changes nothing but rounding
    rng = np.random.default_rng(9)
    s = scenes.scene3d(seed=3, C=2, N=3000, W=320, H=200, focal=300.0)
    Q = scenes.random_rotations(rng, 1)[0]
    T = np.eye(4)
    T[:3, :3] = Q
    T[:3, 3] = rng.uniform(-2, 2, 3)
    means2 = s.means.astype(np.float64) @ Q.T + T[:3, 3]
    covars2 = Q @ s.covars.astype(np.float64) @ Q.T
    views2 = s.viewmats.astype(np.float64) @ np.linalg.inv(T)
    a = oracle.project(s.means, s.covars, s.viewmats, s.intrinsics, s.width, s.height)
    b = oracle.project(means2, covars2, views2, s.intrinsics, s.width, s.height)
    np.testing.assert_allclose(b["means2d"], a["means2d"], rtol=0, atol=5e-3)
    np.testing.assert_allclose(b["depths"], a["depths"], rtol=1e-5)
    np.testing.assert_allclose(b["conics"], a["conics"], rtol=2e-2, atol=1e-4)
    same = (a["radii"] == b["radii"]).mean()
    assert same > 0.97  # radii move only where ceil sits at a rounding boundary


def test_visibility_rules():
    K = _K(500.0, 500.0, 320.0, 240.0)
    S = np.eye(3) * 0.01
    cases = {
        "ok": ([0.0, 0.0, 5.0], {}),
        "behind_near": ([0.0, 0.0, 0.005], {}),
        "at_near": ([0.0, 0.0, 0.01], {}),
        "beyond_far": ([0.0, 0.0, 50.0], {"far_plane": 20.0}),
        "clipped_radius": ([0.0, 0.0, 5.0], {"radius_clip": 1000.0}),
        "left_of_image": ([-40.0, 0.0, 5.0], {}),
        "below_image": ([0.0, 30.0, 5.0], {}),
    }
    for name, (m, kw) in cases.items():
        out = _proj(m, S, _V(), K, **kw)
        r = out["radii"][0, 0]
        if name == "ok":
            assert (r > 0).all(), name
        else:
            assert (r == 0).all(), name
        # means2d, depths and conics are written whether visible or not
        assert out["depths"][0, 0] == np.float32(m[2])
    # det <= 0 (zero covariance, no eps2d): invisible, conic from the 1e-10 stand-in
    out = _proj([0.0, 0.0, 5.0], np.zeros((3, 3)), _V(), K, eps2d=0.0, compensation=True)
    assert (out["radii"] == 0).all()
    np.testing.assert_array_equal(out["conics"][0, 0], [0.0, 0.0, 0.0])
    assert out["compensations"][0, 0] == 0.0
    # a splat straddling the image edge still overlaps it
    out = _proj([-3.3, 0.0, 5.0], S, _V(), K)
    assert (out["radii"][0, 0] > 0).all()


def test_radius_saturates():
    out = _proj([0.0, 0.0, 5.0], np.eye(3) * 1e16, _V(), _K(500.0, 500.0, 320.0, 240.0))
    # 3.33 * sqrt((500 / 5)^2 1e16) = 3.3e10 > 2^31 - 1
    assert (out["radii"][0, 0] == 2**31 - 1).all()


def test_camera_major_layout():
    s = scenes.scene3d_edge(seed=2, N=500)
    both = oracle.project(s.means, s.covars, s.viewmats, s.intrinsics, s.width, s.height,
                          compensation=True)
    for c in range(2):
        one = oracle.project(s.means, s.covars, s.viewmats[c:c + 1], s.intrinsics[c:c + 1],
                             s.width, s.height, compensation=True)
        for k in ("radii", "means2d", "depths", "conics", "compensations"):
            np.testing.assert_array_equal(both[k][c], one[k][0], err_msg=k)
