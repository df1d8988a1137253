"""Pins for the oracle's projection (c1): closed forms, a library rotation routine, a Monte-Carlo
estimate of the projected covariance, invariances, culling and the tile-span brute force of the
learn-gs notebook "11 - Tiles" (claim 2).  CPU only."""
import math

import numpy as np
import pytest

from gaussian_splatting_tile_gb300 import scenes


def one_gaussian(mean, scale, quat, opacity=0.5, dc=(1.0, 0.0, 0.0)):
    sh = np.zeros((3, 1), np.float32)
    sh[:, 0] = np.asarray(dc, np.float32) / np.float32(0.28209479177387814)
    return scenes.Gaussians(means=np.asarray(mean, np.float32).reshape(3, 1),
                            scales=np.asarray(scale, np.float32).reshape(3, 1),
                            quats=np.asarray(quat, np.float32).reshape(4, 1),
                            opacity=np.asarray([opacity], np.float32), sh=sh, sh_degree=0)


def axis_camera(d=4.0, f=150.0, W=128, H=128):
    return scenes.look_at([0.0, 0.0, d], [0.0, 0.0, 0.0], f, f, W, H)


def test_isotropic_closed_form(orc):
    # An isotropic Gaussian of scale s at depth d on the optical axis projects to
    # Sigma_2d = ((f s / d)^2 + 0.3) I exactly; lambda_max = sigma^2 + sqrt(0.1) because of the
    # floor on the discriminant (the discriminant is 0 here).
    f, d, s = 150.0, 4.0, 0.02
    g = one_gaussian([0, 0, 0], [s, s, s], [1, 0, 0, 0])
    cam = axis_camera(d, f)
    P = orc.project(cam, g)
    I = orc.project_intermediates(cam, g)
    s32 = float(np.float32(s))
    sig2 = (f * s32 / d) ** 2 + 0.3
    assert I["cov2d"][:, 0] == pytest.approx([sig2, 0.0, sig2], abs=1e-12)
    assert sig2 == pytest.approx(0.8625, abs=1e-7)
    assert P["conic"][:, 0] == pytest.approx([1 / sig2, 0.0, 1 / sig2], rel=1e-12)
    assert P["means2d"][:, 0] == pytest.approx([64.0, 64.0], abs=1e-12)
    assert P["depth"][0] == pytest.approx(d, rel=1e-12)
    lam = sig2 + math.sqrt(0.1)
    assert lam == pytest.approx(1.178728, abs=1e-6)
    assert P["radius"][0] == math.ceil(3 * math.sqrt(lam)) == 4
    # span: floor((64 -+ 4)/16) = 3 .. floor(68/16)+1 = 5 on both axes -> 2x2 tiles
    assert list(P["rect"][:, 0]) == [3, 5, 3, 5]
    assert P["tiles_touched"][0] == 4
    # degree-0 colour is Y_0 times the DC coefficient
    assert P["color"][:, 0] == pytest.approx([1.0, 0.0, 0.0], rel=1e-6)


def test_anisotropic_axis_aligned_radius(orc):
    # q = identity and a camera on the axis: Sigma_2d = diag((f sx/d)^2, (f sy/d)^2) + 0.3 I,
    # lambda_max = mid + max(sqrt(0.1), |a - c|/2) and r = ceil(3 sqrt(lambda_max)).
    f, d = 150.0, 4.0
    for sx, sy in [(0.05, 0.02), (0.02, 0.11), (0.3, 0.01)]:
        g = one_gaussian([0, 0, 0], [sx, sy, 0.03], [1, 0, 0, 0])
        cam = axis_camera(d, f)
        P = orc.project(cam, g)
        I = orc.project_intermediates(cam, g)
        a = (f * float(np.float32(sx)) / d) ** 2 + 0.3
        c = (f * float(np.float32(sy)) / d) ** 2 + 0.3
        assert I["cov2d"][:, 0] == pytest.approx([a, 0.0, c], rel=1e-12)
        lam = 0.5 * (a + c) + max(math.sqrt(0.1), abs(a - c) / 2)
        assert P["radius"][0] == math.ceil(3 * math.sqrt(lam))


def test_camera_transform_orientation(orc):
    # A point right of the target in world x lands right of centre (u > cx); a point above it
    # (world +y, y-up world) lands above centre (v < cy); depth is the distance along the axis.
    cam = axis_camera(5.0, 100.0, 64, 64)
    for mean, su, sv in [([0.5, 0, 0], 1, 0), ([0, 0.5, 0], 0, -1), ([-0.5, 0, 0], -1, 0)]:
        g = one_gaussian(mean, [0.01] * 3, [1, 0, 0, 0])
        P = orc.project(cam, g)
        I = orc.project_intermediates(cam, g)
        assert I["pcam"][2, 0] == pytest.approx(5.0, rel=1e-7)
        du = P["means2d"][0, 0] - 32.0
        dv = P["means2d"][1, 0] - 32.0
        assert np.sign(round(du, 9)) == su and np.sign(round(dv, 9)) == sv
        assert abs(du) + abs(dv) == pytest.approx(100.0 * 0.5 / 5.0, rel=1e-6)


def test_cov3d_matches_scipy_rotation(orc):
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(3)
    n = 64
    q = rng.standard_normal((4, n)) * rng.uniform(0.2, 3.0, n)  # non-unit on purpose
    s = np.exp(rng.uniform(-3, 0, (3, n)))
    g = scenes.Gaussians(means=np.zeros((3, n), np.float32), scales=s.astype(np.float32),
                         quats=q.astype(np.float32), opacity=np.full(n, 0.5, np.float32),
                         sh=np.zeros((3, n), np.float32), sh_degree=0)
    I = orc.project_intermediates(axis_camera(), g)
    for i in range(n):
        w, x, y, z = g.quats[:, i].astype(np.float64)
        Rm = Rotation.from_quat([x, y, z, w]).as_matrix()  # scipy takes scalar-last
        S3 = Rm @ np.diag(g.scales[:, i].astype(np.float64) ** 2) @ Rm.T
        ref = [S3[0, 0], S3[0, 1], S3[0, 2], S3[1, 1], S3[1, 2], S3[2, 2]]
        assert I["cov3d"][:, i] == pytest.approx(ref, abs=1e-12)


def test_projected_covariance_monte_carlo(orc):
    # Independent of the Jacobian formula: sample world points from N(m, Sigma_3d), push them
    # through the exact pinhole, and compare the sample covariance of (u, v) with
    # Sigma_2d - 0.3 I.  Small Gaussians far from the camera keep the linearisation tight.
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(5)
    cam = scenes.look_at([1.0, 0.7, 4.0], [0.1, -0.2, 0.0], 300.0, 280.0, 256, 200)
    means = np.array([[0.2, -0.3, 0.1], [0.6, 0.4, -0.5], [-0.4, 0.1, 0.3]]).T
    scales = np.array([[0.02, 0.005, 0.01], [0.004, 0.015, 0.02], [0.01, 0.01, 0.002]]).T
    quats = rng.standard_normal((4, 3))
    g = scenes.Gaussians(means=means.astype(np.float32), scales=scales.astype(np.float32),
                         quats=quats.astype(np.float32), opacity=np.full(3, 0.5, np.float32),
                         sh=np.zeros((3, 3), np.float32), sh_degree=0)
    I = orc.project_intermediates(cam, g)
    R = cam.R.astype(np.float64)
    t = cam.t.astype(np.float64)
    for i in range(3):
        w, x, y, z = g.quats[:, i].astype(np.float64)
        Rm = Rotation.from_quat([x, y, z, w]).as_matrix()
        L = Rm @ np.diag(g.scales[:, i].astype(np.float64))
        pts = g.means[:, i].astype(np.float64)[:, None] + L @ rng.standard_normal((3, 400_000))
        pc = R @ pts + t[:, None]
        u = cam.fx * pc[0] / pc[2] + cam.cx
        v = cam.fy * pc[1] / pc[2] + cam.cy
        C = np.cov(np.stack([u, v]))
        a, b, c = I["cov2d"][:, i]
        ref = np.array([[a - 0.3, b], [b, c - 0.3]])
        scale = np.sqrt(np.diag(ref))
        assert np.abs((C - ref) / np.outer(scale, scale)).max() < 0.02


def test_jacobian_clamp_off_axis(orc):
    # A point far off-axis: x/z beyond 1.3 * (W/2)/fx.  J is built at the clamped tx = lim * z,
    # so J[0,2] = -fx * lim / z while u stays unclamped.
    W, H, f = 64, 64, 50.0
    cam = axis_camera(2.0, f, W, H)
    lim = 1.3 * (W / 2) / f
    x = 3.0  # camera z = 2, x/z = 1.5 > lim = 0.832
    g = one_gaussian([x, 0.0, 0.0], [0.3, 0.3, 0.3], [1, 0, 0, 0])
    I = orc.project_intermediates(cam, g)
    z = I["pcam"][2, 0]
    assert I["pcam"][0, 0] == pytest.approx(3.0)
    assert I["jac"][0, 0] == pytest.approx(f / z)
    assert I["jac"][2, 0] == pytest.approx(-f * (lim * z) / z ** 2, rel=1e-6)
    assert I["jac"][5, 0] == pytest.approx(0.0, abs=1e-12)  # y = 0: unclamped, -fy*0/z^2
    P = orc.project(cam, g)
    if P["radius"][0] > 0:
        assert P["means2d"][0, 0] == pytest.approx(f * x / z + W / 2)
    # the unclamped J against a numerical Jacobian of the pinhole at an on-axis-ish point
    g2 = one_gaussian([0.2, -0.1, 0.3], [0.05] * 3, [1, 0, 0, 0])
    I2 = orc.project_intermediates(cam, g2)
    p = I2["pcam"][:, 0]
    h = 1e-6
    num = np.zeros((2, 3))
    for k in range(3):
        dp = np.zeros(3)
        dp[k] = h
        uvp = np.array([f * (p + dp)[0] / (p + dp)[2], f * (p + dp)[1] / (p + dp)[2]])
        uvm = np.array([f * (p - dp)[0] / (p - dp)[2], f * (p - dp)[1] / (p - dp)[2]])
        num[:, k] = (uvp - uvm) / (2 * h)
    assert I2["jac"][:, 0].reshape(2, 3) == pytest.approx(num, rel=1e-7, abs=1e-7)


def test_quaternion_norm_invariance(orc):
    g, cam = scenes.tiny_scene(seed=1, n=300)
    P1 = orc.project(cam, g)
    # powers of two scale the quaternion exactly, so only the normalisation is exercised
    for f in (2.0, 0.25, 8.0):
        g2 = scenes.Gaussians(means=g.means, scales=g.scales, quats=(g.quats * np.float32(f)),
                              opacity=g.opacity, sh=g.sh, sh_degree=g.sh_degree)
        P2 = orc.project(cam, g2)
        assert np.array_equal(P1["radius"], P2["radius"])
        for k in ("means2d", "depth", "conic", "color"):
            np.testing.assert_allclose(P1[k], P2[k], rtol=1e-12, atol=1e-12)


def test_z_rotation_swaps_scales(orc):
    c = math.cos(math.pi / 4)
    g = one_gaussian([0, 0, 0], [0.3, 0.1, 0.05], [c, 0, 0, c])
    I = orc.project_intermediates(axis_camera(), g)
    s = g.scales[:, 0].astype(np.float64)
    ref = [s[1] ** 2, 0, 0, s[0] ** 2, 0, s[2] ** 2]
    assert I["cov3d"][:, 0] == pytest.approx(ref, abs=1e-7)


def test_culling(orc):
    cam = axis_camera(4.0, 150.0)
    cases = {
        "behind near plane": ([0, 0, 3.96], [0.02] * 3, [1, 0, 0, 0]),   # z = 0.04
        "behind camera": ([0, 0, 6.0], [0.02] * 3, [1, 0, 0, 0]),
        "off screen": ([50.0, 0, 0], [0.02] * 3, [1, 0, 0, 0]),
        "zero quaternion": ([0, 0, 0], [0.02] * 3, [0, 0, 0, 0]),
        "nan mean": ([float("nan"), 0, 0], [0.02] * 3, [1, 0, 0, 0]),
    }
    for name, (m, s, q) in cases.items():
        P = orc.project(cam, one_gaussian(m, s, q))
        assert P["radius"][0] == 0, name
        assert P["tiles_touched"][0] == 0, name
        assert not np.any(P["conic"][:, 0]) and not np.any(P["means2d"][:, 0]), name
    # just in front of the near plane is kept
    P = orc.project(cam, one_gaussian([0, 0, 3.9], [0.001] * 3, [1, 0, 0, 0]))
    assert P["radius"][0] > 0


def test_span_matches_brute_force_overlap(orc):
    # learn-gs "11 - Tiles", claim 2: a tile is listed exactly when its square overlaps the
    # splat's bounding square [u - r, u + r] x [v - r, v + r]; checked in float32.
    rng = np.random.default_rng(11)
    n = 400
    cam = scenes.look_at([0, 0, 3.0], [0, 0, 0], 60.0, 60.0, 64, 64)
    g = scenes.Gaussians(means=rng.uniform(-2.5, 2.5, (3, n)).astype(np.float32),
                         scales=np.exp(rng.uniform(-4, -1, (3, n))).astype(np.float32),
                         quats=rng.standard_normal((4, n)).astype(np.float32),
                         opacity=np.full(n, 0.5, np.float32),
                         sh=np.zeros((3, n), np.float32), sh_degree=0)
    P = orc.project(cam, g, prec=32)
    TX = TY = 4
    seen = 0
    for i in range(n):
        if P["radius"][i] == 0:
            continue
        seen += 1
        u, v = np.float32(P["means2d"][0, i]), np.float32(P["means2d"][1, i])
        r = np.float32(P["radius"][i])
        xl, xh, yl, yh = P["rect"][:, i]
        for tx in range(TX):
            for ty in range(TY):
                overlap = (np.float32(tx * 16) <= u + r and np.float32((tx + 1) * 16) > u - r and
                           np.float32(ty * 16) <= v + r and np.float32((ty + 1) * 16) > v - r)
                listed = xl <= tx < xh and yl <= ty < yh
                assert overlap == listed
        assert P["tiles_touched"][i] == (xh - xl) * (yh - yl)
    assert seen > 50


def test_fp32_and_fp64_take_the_same_decisions(orc):
    g, cam = scenes.tiny_scene(seed=0)
    P32 = orc.project(cam, g, prec=32, margin=1e-5)
    P64 = orc.project(cam, g, prec=64, margin=1e-5)
    clear = P64["ambig"] == 0
    assert clear.mean() > 0.99
    assert np.array_equal(P32["radius"][clear], P64["radius"][clear])
    assert np.array_equal(P32["rect"][:, clear], P64["rect"][:, clear])
    vis = clear & (P64["radius"] > 0)
    np.testing.assert_allclose(P32["means2d"][:, vis], P64["means2d"][:, vis], rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(P32["conic"][:, vis], P64["conic"][:, vis], rtol=1e-4, atol=1e-6)
