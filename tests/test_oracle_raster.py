"""Pins for the oracle's forward compositing (c3): the closed-form image of one isotropic
Gaussian, a two-splat hand example, the invariant accumulated alpha = 1 - final_T (rigel
"Gallery"), contributor counting, and brute-force all-pixels x all-splats rendering where the
3-sigma radius cannot bind (learn-gs "11 - Tiles", tiled vs naive).  CPU only."""
import math

import numpy as np
import pytest

from gaussian_splatting_tile_gb300 import scenes


def manual_splats(cam, rows):
    """rows: (u, v, A, B, C, opacity, r, g, b, depth).  Binned by the oracle with a radius large
    enough to cover the whole image, so every splat is in every tile's list."""
    a = np.asarray(rows, np.float64)
    n = a.shape[0]
    means2d, conic, opac, color, depth = a[:, 0:2].T, a[:, 2:5].T, a[:, 5], a[:, 6:9].T, a[:, 9]
    radius = np.full(n, 4 * max(cam.width, cam.height), np.int32)
    return means2d, conic, opac, color, depth, radius


def test_two_splat_worked_example(orc):
    # Front splat alpha 0.5 red, back splat alpha 0.4 blue, both centred on pixel (8, 8) so that
    # exp(power) = 1 there; background black.  C = 0.5 red + 0.5 * 0.4 blue = (0.5, 0, 0.2),
    # final_T = 0.5 * 0.6 = 0.3, two contributors, accumulated alpha 0.7.
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 50.0, 50.0, 16, 16)
    m2, con, op, col, dep, rad = manual_splats(cam, [
        (8, 8, 1, 0, 1, 0.5, 1, 0, 0, 1.0),
        (8, 8, 1, 0, 1, 0.4, 0, 0, 1, 2.0)])
    B = orc.bin(cam, m2.astype(np.float32), dep.astype(np.float32), rad)
    assert list(B["point_list"]) == [0, 1]
    F = orc.raster_fwd(cam, m2, con, op, col, B["ranges"], B["point_list"])
    assert F["image"][:, 8, 8] == pytest.approx([0.5, 0.0, 0.2], abs=1e-15)
    assert F["final_T"][8, 8] == pytest.approx(0.3, abs=1e-15)
    assert F["n_contrib"][8, 8] == 2
    # background enters as T_final * bg
    F = orc.raster_fwd(cam, m2, con, op, col, B["ranges"], B["point_list"], bg=(1.0, 1.0, 1.0))
    assert F["image"][:, 8, 8] == pytest.approx([0.8, 0.3, 0.5], abs=1e-15)


def test_isotropic_gaussian_image(orc):
    # One isotropic Gaussian (sigma^2 = (f s/d)^2 + 0.3 = 0.8625) with opacity 0.5 centred on
    # pixel (64, 64): image = colour * alpha(rho) with alpha = 0.5 exp(-rho^2 / (2 sigma^2)):
    # alpha(0) = 0.5, alpha(1) = 0.280030, alpha(2) = 0.049194, alpha(3) = 0.0027 < 1/255 (skipped).
    sh = (np.array([[1.0], [0.5], [0.25]]) / 0.28209479177387814).astype(np.float32)
    g = scenes.Gaussians(means=np.zeros((3, 1), np.float32), scales=np.full((3, 1), 0.02, np.float32),
                         quats=np.array([[1], [0], [0], [0]], np.float32),
                         opacity=np.array([0.5], np.float32), sh=sh, sh_degree=0)
    cam = scenes.look_at([0, 0, 4.0], [0, 0, 0], 150.0, 150.0, 128, 128)
    P, B, F = orc.render(cam, g)
    sig2 = (150.0 * float(np.float32(0.02)) / 4.0) ** 2 + 0.3
    expect = {0: 0.5, 1: 0.280030, 2: 0.049194}
    for rho, a in expect.items():
        a_exact = 0.5 * math.exp(-rho * rho / (2 * sig2))
        assert a_exact == pytest.approx(a, abs=1e-6)
        for (dx, dy) in [(rho, 0), (0, rho), (-rho, 0), (0, -rho)]:
            px = F["image"][:, 64 + dy, 64 + dx]
            assert P["color"][:, 0] == pytest.approx([1.0, 0.5, 0.25], rel=1e-7)
            assert px == pytest.approx(P["color"][:, 0] * a_exact, rel=1e-12)
            assert F["final_T"][64 + dy, 64 + dx] == pytest.approx(1 - a_exact, rel=1e-12)
    assert 0.5 * math.exp(-9 / (2 * sig2)) < 1 / 255
    assert not F["image"][:, 64, 67].any() and F["final_T"][64, 67] == 1.0
    assert F["n_contrib"][64, 67] == 1          # inside the span: examined, skipped
    # outside the 4-pixel radius square the tiles (3..4 on each axis) do not list the splat
    assert F["n_contrib"][10, 10] == 0 and F["n_contrib"][64, 80] == 0
    assert F["n_contrib"][64, 79] == 1


def test_accumulated_alpha_invariant(orc):
    # With every colour 1 and a black background, each channel equals sum_i alpha_i T_i,
    # which telescopes to 1 - final_T.
    g, cam = scenes.tiny_scene(seed=3)
    g.sh[:] = np.float32(1.0 / 0.28209479177387814)
    P, B, F = orc.render(cam, g)
    for ch in range(3):
        np.testing.assert_allclose(F["image"][ch], 1.0 - F["final_T"], atol=1e-12)
    lens = (B["ranges"][:, 1] - B["ranges"][:, 0]).astype(np.int64)
    TX = cam.tiles_x
    H, W = cam.height, cam.width
    tile_of = (np.arange(H)[:, None] // 16) * TX + (np.arange(W)[None, :] // 16)
    assert np.all(F["n_contrib"] <= lens[tile_of])
    assert np.all((F["final_T"] > 0) & (F["final_T"] <= 1))


def test_stops_after_transmittance_falls_below_threshold(orc):
    # Ten opaque splats (alpha 0.99) at one pixel: T = 0.01, then 1e-4 (not < 1e-4: exactly the
    # threshold in exact arithmetic, rounding decides), then 1e-6 < 1e-4 -> stop at three.
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 50.0, 50.0, 16, 16)
    rows = [(8, 8, 1, 0, 1, 1.0, 1, 1, 1, 1.0 + k) for k in range(10)]
    m2, con, op, col, dep, rad = manual_splats(cam, rows)
    B = orc.bin(cam, m2.astype(np.float32), dep.astype(np.float32), rad)
    F = orc.raster_fwd(cam, m2, con, op, col, B["ranges"], B["point_list"])
    T2 = (1 - 0.99) * (1 - 0.99)
    expected_n = 2 if T2 < 1e-4 else 3
    assert F["n_contrib"][8, 8] == expected_n
    assert F["final_T"][8, 8] < 1e-4
    # a pixel far from every centre never stops: it examines the whole list
    F2 = orc.raster_fwd(cam, m2, con * 50, op, col, B["ranges"], B["point_list"])
    assert F2["n_contrib"][0, 0] == 10 and F2["final_T"][0, 0] == 1.0


def brute_force_render(cam, P, opacity, bg):
    """Every pixel composites every visible splat in (depth, index) order, no tiles."""
    H, W = cam.height, cam.width
    vis = np.nonzero(P["radius"] > 0)[0]
    order = vis[np.lexsort((vis, P["depth"][vis].astype(np.float32)))]
    py, px = np.meshgrid(np.arange(H, dtype=np.float64), np.arange(W, dtype=np.float64), indexing="ij")
    T = np.ones((H, W))
    C = np.zeros((3, H, W))
    live = np.ones((H, W), bool)
    for g in order:
        dx = px - P["means2d"][0, g]
        dy = py - P["means2d"][1, g]
        A, B_, Cc = P["conic"][:, g]
        power = -0.5 * (A * dx * dx + Cc * dy * dy) - B_ * dx * dy
        alpha = np.minimum(0.99, float(opacity[g]) * np.exp(power))
        use = live & (alpha >= 1 / 255)
        for ch in range(3):
            C[ch] = np.where(use, C[ch] + P["color"][ch, g] * alpha * T, C[ch])
        T = np.where(use, T * (1 - alpha), T)
        live &= ~(use & (T < 1e-4))
    return C + T[None] * np.asarray(bg)[:, None, None], T


@pytest.mark.parametrize("seed", [0, 1])
def test_tiled_equals_brute_force_when_radius_cannot_bind(orc, seed):
    # With opacity <= 0.35 < e^4.5/255 no splat can reach alpha >= 1/255 outside its 3-sigma
    # square, so skipping it there (the tiles) and evaluating it (brute force) agree exactly.
    g, cam = scenes.tiny_scene(seed=seed, opacity_cap=0.35)
    bg = (0.1, 0.2, 0.3)
    P, B, F = orc.render(cam, g, bg=bg)
    img, T = brute_force_render(cam, P, g.opacity, bg)
    np.testing.assert_allclose(F["image"], img, atol=1e-13, rtol=0)
    np.testing.assert_allclose(F["final_T"], T, atol=1e-13, rtol=0)


def test_fp32_variant_agrees(orc):
    g, cam = scenes.tiny_scene(seed=0)
    P, B, F64 = orc.render(cam, g, prec=64)
    F32 = orc.raster_fwd(cam, P["means2d"], P["conic"], g.opacity, P["color"], B["ranges"],
                         B["point_list"], prec=32)
    np.testing.assert_allclose(F32["image"], F64["image"], atol=1e-5)
    assert (F32["n_contrib"] == F64["n_contrib"]).mean() > 0.999
