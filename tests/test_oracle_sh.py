"""Pins for the oracle's SH basis (c6): orthonormality on the sphere by exact quadrature, and
the signs/normalisation against scipy's complex spherical harmonics in the real form of Sloan's
"Stupid Spherical Harmonics (SH) Tricks", Appendix A2 (the table the viewer page prints in
2.2.3).  CPU only."""
import numpy as np
import pytest

from gaussian_splatting_tile_gb300 import scenes


def quadrature(nt=16, nphi=32):
    # Gauss-Legendre in cos(theta) x uniform in phi: exact for polynomials of degree <= 2*nt-1
    # in cos(theta) and trigonometric degree < nphi in phi; products of two degree-3 SH are
    # degree 6.
    x, w = np.polynomial.legendre.leggauss(nt)
    phi = (np.arange(nphi) + 0.5) * 2 * np.pi / nphi
    ct, ph = np.meshgrid(x, phi, indexing="ij")
    st = np.sqrt(1 - ct ** 2)
    dirs = np.stack([st * np.cos(ph), st * np.sin(ph), ct]).reshape(3, -1)
    wts = (w[:, None] * np.full(nphi, 2 * np.pi / nphi)[None, :]).reshape(-1)
    return dirs, wts


def test_orthonormal(orc):
    dirs, wts = quadrature()
    Y = orc.sh_basis(dirs)
    gram = (Y * wts) @ Y.T
    np.testing.assert_allclose(gram, np.eye(16), atol=1e-12)


def real_sh_from_scipy(l, m, dirs):
    import scipy.special as sp
    theta = np.arccos(np.clip(dirs[2], -1, 1))
    phi = np.arctan2(dirs[1], dirs[0])
    if hasattr(sp, "sph_harm_y"):
        Ylm = sp.sph_harm_y(l, abs(m), theta, phi)
    else:  # older scipy: sph_harm(m, n, azimuth, polar)
        Ylm = sp.sph_harm(abs(m), l, phi, theta)
    # scipy's associated Legendre functions carry the Condon-Shortley phase; Sloan's real form is
    # sqrt(2) Re for m > 0, sqrt(2) Im of the |m| function for m < 0, and Y_l^0 for m = 0.
    if m > 0:
        return np.sqrt(2) * Ylm.real
    if m < 0:
        return np.sqrt(2) * Ylm.imag
    return Ylm.real


def test_matches_scipy_real_form(orc):
    rng = np.random.default_rng(0)
    d = rng.standard_normal((3, 500))
    d /= np.linalg.norm(d, axis=0, keepdims=True)
    Y = orc.sh_basis(d)
    for l in range(4):
        for m in range(-l, l + 1):
            k = l * l + l + m
            np.testing.assert_allclose(Y[k], real_sh_from_scipy(l, m, d), atol=1e-12,
                                       err_msg=f"l={l} m={m}")


def test_degree0_colour_is_view_independent(orc):
    g, _ = scenes.tiny_scene(seed=2, n=200)
    cams = [scenes.look_at(e, [0, 0, 0], 150, 150, 128, 128)
            for e in ([0, 0, 4], [3, 1, 2], [-2, -2, 3])]
    Y0 = 0.5 / np.sqrt(np.pi)
    for cam in cams:
        P = orc.project(cam, g)
        vis = P["radius"] > 0
        np.testing.assert_allclose(P["color"][:, vis], Y0 * g.sh[:, vis].astype(np.float64),
                                   rtol=1e-12)


def test_sh_colour_is_sum_over_basis(orc):
    # colour_ch = sum_k sh[k*3+ch] Y_k(d) with d from the camera centre to the mean: checked by
    # evaluating the basis on the directions computed here from the camera's centre -R^T t.
    g = scenes.procedural_scene(seed=4, n_sphere=300, n_helix=100, n_plane=100)
    cam = scenes.procedural_camera(160, 120, azimuth=0.7)
    P = orc.project(cam, g)
    C = -(cam.R.astype(np.float64).T @ cam.t.astype(np.float64))
    d = g.means.astype(np.float64) - C[:, None]
    d /= np.linalg.norm(d, axis=0, keepdims=True)
    Y = orc.sh_basis(d)
    sh = g.sh.astype(np.float64).reshape(16, 3, -1)
    ref = np.einsum("kcn,kn->cn", sh, Y)
    vis = P["radius"] > 0
    assert vis.sum() > 100
    np.testing.assert_allclose(P["color"][:, vis], ref[:, vis], rtol=1e-10, atol=1e-12)
