"""Pins for the oracle's backward passes (c4, c5, c7): central finite differences of the oracle's
own double-precision forwards (which the forward pins fix independently), hand-derived two-splat
gradients, the zero gradient through a clamped alpha (rigel "Deliberate differences"), the
quaternion-gradient invariant dq . q = 0, and the off-axis clamp branch.  CPU only."""
import numpy as np
import pytest

import oracle
from gaussian_splatting_tile_gb300 import scenes


def random_projected(seed, n, W, H):
    rng = np.random.default_rng(seed)
    u = rng.uniform(-4, W + 4, n)
    v = rng.uniform(-4, H + 4, n)
    s1 = rng.uniform(1.5, 6.0, n)
    s2 = rng.uniform(1.5, 6.0, n)
    th = rng.uniform(0, np.pi, n)
    c, s = np.cos(th), np.sin(th)
    a = c * c * s1 ** 2 + s * s * s2 ** 2
    b = c * s * (s1 ** 2 - s2 ** 2)
    cc = s * s * s1 ** 2 + c * c * s2 ** 2
    det = a * cc - b * b
    conic = np.stack([cc / det, -b / det, a / det])
    lam = 0.5 * (a + cc) + np.sqrt(np.maximum(0.1, (0.5 * (a + cc)) ** 2 - det))
    radius = np.ceil(3 * np.sqrt(lam)).astype(np.int32)
    opac = rng.uniform(0.1, 0.95, n)
    color = rng.uniform(0, 1, (3, n))
    depth = rng.uniform(1, 5, n)
    # round to float32 so the binning (float decisions) and the double maths see the same values
    f = lambda x: x.astype(np.float32).astype(np.float64)
    return f(np.stack([u, v])), f(conic), f(opac), f(color), f(depth), radius


def loss(orc, cam, m2, con, op, col, B, G, bg):
    F = orc.raster_fwd(cam, m2, con, op, col, B["ranges"], B["point_list"], bg=bg, margin=1e-7)
    return float(np.sum(F["image"] * G)), F


def test_raster_backward_finite_differences(orc):
    W, H, n = 40, 28, 60
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 50.0, 50.0, W, H)
    m2, con, op, col, dep, rad = random_projected(0, n, W, H)
    op[0] = 1.0  # its centre pixel (if any) is clamped at 0.99
    B = orc.bin(cam, m2.astype(np.float32), dep.astype(np.float32), rad)
    G = np.random.default_rng(1).standard_normal((3, H, W))
    bg = (0.2, 0.1, 0.3)
    L0, F0 = loss(orc, cam, m2, con, op, col, B, G, bg)
    assert (F0["n_contrib"] > 0).mean() > 0.5
    assert (F0["final_T"] < 0.5).mean() > 0.05  # overlapping splats, some pixels saturate
    an = orc.raster_bwd(cam, m2, con, op, col, B["ranges"], B["point_list"], F0["n_contrib"], G, bg=bg)
    rng = np.random.default_rng(2)
    checked = 0
    params = {"dmeans2d": m2, "dconic": con, "dopacity": op, "dcolor": col}
    for name, arr in params.items():
        flat = arr.reshape(-1)
        grad = an[name].reshape(-1)
        for idx in rng.choice(flat.size, size=min(40, flat.size), replace=False):
            h = 1e-6 * max(1.0, abs(flat[idx]))
            old = flat[idx]
            fds = []
            for step in (h, 2 * h):
                flat[idx] = old + step
                Lp, Fp = loss(orc, cam, m2, con, op, col, B, G, bg)
                flat[idx] = old - step
                Lm, Fm = loss(orc, cam, m2, con, op, col, B, G, bg)
                fds.append((Lp - Lm) / (2 * step))
            flat[idx] = old
            # a guard (skip, clamp, stop) flipping inside +-2h puts a jump into the loss, and the
            # two step sizes then disagree: such a sample says nothing about the derivative
            if abs(fds[0] - fds[1]) > 1e-6 * max(1.0, abs(fds[0])):
                continue
            assert fds[0] == pytest.approx(grad[idx], rel=1e-5, abs=1e-7), (name, idx)
            checked += 1
    assert checked > 120


def test_two_splat_gradients(orc):
    # L = sum over channels of C with C = a1 c1 + (1 - a1) a2 c2 (c1 red, c2 blue, bg black):
    # dL/da1 = 1 - a2 = 0.6, dL/da2 = 1 - a1 = 0.5, dL/dc1 = a1 T1 = 0.5, dL/dc2 = a2 T2 = 0.2.
    # Both centred on the pixel, so exp(power) = 1: dL/do = dL/da, and the mean gradient is 0.
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 50.0, 50.0, 16, 16)
    m2 = np.array([[8.0, 8.0], [8.0, 8.0]])
    con = np.array([[1.0, 1.0], [0.0, 0.0], [1.0, 1.0]])
    op = np.array([0.5, 0.4])
    col = np.array([[1.0, 0.0], [0.0, 0.0], [0.0, 1.0]])
    dep = np.array([1.0, 2.0])
    rad = np.array([64, 64], np.int32)
    B = orc.bin(cam, m2.astype(np.float32), dep.astype(np.float32), rad)
    F = orc.raster_fwd(cam, m2, con, op, col, B["ranges"], B["point_list"])
    G = np.zeros((3, 16, 16))
    G[:, 8, 8] = 1.0
    g = orc.raster_bwd(cam, m2, con, op, col, B["ranges"], B["point_list"], F["n_contrib"], G)
    assert g["dopacity"] == pytest.approx([0.6, 0.5], abs=1e-15)
    assert g["dcolor"][:, 0] == pytest.approx([0.5, 0.5, 0.5], abs=1e-15)
    assert g["dcolor"][:, 1] == pytest.approx([0.2, 0.2, 0.2], abs=1e-15)
    assert not g["dmeans2d"].any() and not g["dconic"].any()


def test_clamped_alpha_has_no_alpha_gradient(orc):
    # Opacity 1 at the splat's centre: o exp(0) = 1 > 0.99, alpha is the constant 0.99 there.
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 50.0, 50.0, 16, 16)
    m2 = np.array([[8.0], [8.0]])
    con = np.array([[0.5], [0.0], [0.5]])
    op = np.array([1.0])
    col = np.array([[0.3], [0.6], [0.9]])
    B = orc.bin(cam, m2.astype(np.float32), np.array([1.0], np.float32), np.array([64], np.int32))
    F = orc.raster_fwd(cam, m2, con, op, col, B["ranges"], B["point_list"])
    G = np.zeros((3, 16, 16))
    G[:, 8, 8] = 1.0
    g = orc.raster_bwd(cam, m2, con, op, col, B["ranges"], B["point_list"], F["n_contrib"], G)
    assert g["dopacity"][0] == 0.0 and not g["dconic"].any() and not g["dmeans2d"].any()
    assert g["dcolor"][:, 0] == pytest.approx([0.99] * 3)
    # one pixel over, exp(-0.25) < 0.99: the gradient flows
    G2 = np.zeros((3, 16, 16))
    G2[:, 8, 9] = 1.0
    g2 = orc.raster_bwd(cam, m2, con, op, col, B["ranges"], B["point_list"], F["n_contrib"], G2)
    assert g2["dopacity"][0] == pytest.approx(np.exp(-0.25) * col.sum())


def project_loss(orc, cam, g, w):
    P = orc.project(cam, g, margin=1e-7)
    L = float(np.sum(P["means2d"] * w["m2"]) + np.sum(P["conic"] * w["con"]) +
              np.sum(P["color"] * w["col"]))
    return L, P


def off_axis_set(cam, n, rng):
    # Gaussians well outside the 1.3x frustum on x or y but large enough to still touch the image.
    z = rng.uniform(1.5, 3.0, n)
    lim_x = 1.3 * (cam.width / 2) / cam.fx
    xz = rng.choice([-1, 1], n) * lim_x * rng.uniform(1.1, 1.6, n)
    yz = rng.uniform(-0.3, 0.3, n)
    pc = np.stack([xz * z, yz * z, z])
    Rt = cam.R.astype(np.float64).T
    return Rt @ (pc - cam.t.astype(np.float64)[:, None])


@pytest.mark.parametrize("degree", [3, -1])
def test_project_backward_finite_differences(orc, degree):
    rng = np.random.default_rng(9)
    cam = scenes.look_at([0.3, 0.4, 3.0], [0, 0, 0], 80.0, 90.0, 96, 80)
    n_in, n_off = 30, 12
    means = np.concatenate([rng.uniform(-1, 1, (3, n_in)), off_axis_set(cam, n_off, rng)], axis=1)
    n = n_in + n_off
    scales = np.exp(rng.uniform(-3.5, -1.0, (3, n)))
    scales[:, n_in:] = np.exp(rng.uniform(-0.5, 0.3, (3, n_off)))
    quats = rng.standard_normal((4, n)) * rng.uniform(0.5, 2.0, n)  # non-unit on purpose
    K = 16 if degree == 3 else 0
    g = scenes.Gaussians(means=means.astype(np.float32), scales=scales.astype(np.float32),
                         quats=quats.astype(np.float32), opacity=np.full(n, 0.5, np.float32),
                         sh=rng.normal(0, 0.5, (3 * K, n)).astype(np.float32) if K else None,
                         sh_degree=degree,
                         colors=None if K else rng.uniform(0, 1, (3, n)).astype(np.float32))
    for k in ("means", "scales", "quats", "sh"):
        a = getattr(g, k)
        if a is not None:
            setattr(g, k, a.astype(np.float64))
    w = dict(m2=rng.standard_normal((2, n)), con=rng.standard_normal((3, n)),
             col=rng.standard_normal((3, n)))
    L0, P0 = project_loss(orc, cam, g, w)
    vis = P0["radius"] > 0
    assert vis[:n_in].sum() > 20 and vis[n_in:].sum() >= 4
    an = orc.project_bwd(cam, g, P0["radius"], w["m2"], w["con"], w["col"])
    assert np.all(an["dmeans"][:, ~vis] == 0)
    # the forward normalises q, so the gradient has no radial component
    dots = np.sum(an["dquats"] * g.quats, axis=0)
    assert np.abs(dots).max() < 1e-9 * max(1.0, np.abs(an["dquats"]).max())
    checked = 0
    pairs = [("means", "dmeans"), ("scales", "dscales"), ("quats", "dquats")]
    if K:
        pairs.append(("sh", "dsh"))
    for attr, gname in pairs:
        arr = getattr(g, attr)
        for i in np.nonzero(vis)[0]:
            for r in range(arr.shape[0]):
                old = arr[r, i]
                h = 1e-6 * max(1.0, abs(old))
                arr[r, i] = old + h
                Lp, Pp = project_loss(orc, cam, g, w)
                arr[r, i] = old - h
                Lm, Pm = project_loss(orc, cam, g, w)
                arr[r, i] = old
                if Pp["ambig"][i] or Pm["ambig"][i] or Pp["radius"][i] == 0 or Pm["radius"][i] == 0:
                    continue
                fd = (Lp - Lm) / (2 * h)
                assert fd == pytest.approx(an[gname][r, i], rel=1e-5, abs=1e-6), (attr, r, i)
                checked += 1
    assert checked > 200


def test_appearance_mlp(orc):
    rng = np.random.default_rng(4)
    n, L, H = 25, 8, 16
    cam = scenes.look_at([0.5, 1.0, 4.0], [0, 0, 0], 100, 100, 64, 64)
    means = rng.uniform(-1, 1, (3, n))
    lat = rng.standard_normal((L, n))
    W1 = rng.uniform(-0.5, 0.5, (H, L + 3))
    b1 = rng.uniform(-0.2, 0.2, H)
    W2 = rng.uniform(-0.5, 0.5, (3, H))
    b2 = rng.uniform(-0.2, 0.2, 3)
    # closed form: a zero output layer gives sigmoid(b2) for every Gaussian
    c0 = orc.appearance_fwd(cam, means, lat, W1, b1, np.zeros((3, H)), b2)
    np.testing.assert_allclose(c0, np.repeat((1 / (1 + np.exp(-b2)))[:, None], n, 1), rtol=1e-15)
    G = rng.standard_normal((3, n))
    an = orc.appearance_bwd(cam, means, lat, W1, b1, W2, b2, G)
    params = dict(dlatents=lat, dW1=W1, db1=b1, dW2=W2, db2=b2)

    def Lf():
        return float(np.sum(orc.appearance_fwd(cam, means, lat, W1, b1, W2, b2) * G))

    for name, arr in params.items():
        flat = arr.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            h = 1e-6
            flat[idx] = old + h
            Lp = Lf()
            flat[idx] = old - h
            Lm = Lf()
            flat[idx] = old
            assert (Lp - Lm) / (2 * h) == pytest.approx(an[name].reshape(-1)[idx], rel=1e-6, abs=1e-8)


def test_magnitude_sums_bound_the_gradients():
    """The compositing backward's magnitude sums (the rounding scale of the gradient sums) are at
    least the gradients' magnitudes (triangle inequality) and vanish where nothing was added."""
    g, cam = scenes.tiny_scene(seed=3, n=300)
    P = oracle.project(cam, g)
    B = oracle.bin(cam, P["means2d"].astype(np.float32), P["depth"].astype(np.float32), P["radius"])
    F = oracle.raster_fwd(cam, P["means2d"], P["conic"], g.opacity, P["color"], B["ranges"], B["point_list"])
    O = oracle.raster_bwd(cam, P["means2d"], P["conic"], g.opacity, P["color"], B["ranges"], B["point_list"],
                          F["n_contrib"], scenes.image_grad(cam))
    for k in ("dmeans2d", "dconic", "dopacity", "dcolor"):
        assert (O["abs_" + k] >= np.abs(O[k]) * (1 - 1e-12)).all(), k
        assert (O["abs_" + k] > 0).any()
    absent = np.ones(g.n, bool)
    absent[B["point_list"]] = False  # in no tile's list: nothing is added for them
    absent[:5] = True
    P["means2d"][:, :5] = -1e4  # five Gaussians moved far off the image keep their list entries
    O2 = oracle.raster_bwd(cam, P["means2d"], P["conic"], g.opacity, P["color"], B["ranges"], B["point_list"],
                           F["n_contrib"], scenes.image_grad(cam))
    assert not O2["abs_dconic"][:, absent].any() and not O2["abs_dcolor"][:, absent].any()
