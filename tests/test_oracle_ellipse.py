"""Pins of the oracle's ellipse-tile test (c2', the pages' next binning step), CPU only.

The oracle keeps a tile of a splat's radius square when the minimum of q(d) = d^T Q d over the
tile's pixel-centre square is at most k.  It is pinned against things that do not share its
arithmetic:
  - its rectangle minimum against scipy's bounded least squares (q = |L^T d|^2 with Q = L L^T, a
    library routine) and against the closed form of an axis-aligned ellipse;
  - its decisions against brute force over the integer pixel centres (every tile holding a pixel
    centre inside the ellipse is kept), against the ellipse's closed-form bounding box (no tile
    outside it is kept), and, tile by tile, against the bounded least-squares minimum;
  - its binning: the square binning's per-tile lists with entries removed, order kept."""
import numpy as np
from scipy.optimize import lsq_linear

import oracle
from gaussian_splatting_tile_gb300 import scenes


def lsq_min(A, B, C, x0, x1, y0, y1):
    """min of A x^2 + 2 B x y + C y^2 over a rectangle by bounded least squares."""
    Lc = np.linalg.cholesky(np.array([[A, B], [B, C]], np.float64))  # Q = Lc Lc^T
    if x0 == x1 and y0 == y1:
        d = np.array([x0, y0])
        return float(d @ np.array([[A, B], [B, C]]) @ d)
    r = lsq_linear(Lc.T, np.zeros(2), bounds=([x0, y0], [x1, y1]), method="bvls", tol=1e-14)
    return 2.0 * r.cost


def random_splats(rng, count, cam):
    for _ in range(count):
        u, v = rng.uniform(-20, cam.width + 20), rng.uniform(-20, cam.height + 20)
        th = rng.uniform(0, np.pi)
        s1, s2 = np.exp(rng.uniform(np.log(0.6), np.log(60), 2))
        Rm = np.array([[np.cos(th), -np.sin(th)], [np.sin(th), np.cos(th)]])
        cov = Rm @ np.diag([s1 * s1, s2 * s2]) @ Rm.T + 0.3 * np.eye(2)
        Q = np.linalg.inv(cov).astype(np.float32)
        o = rng.uniform(0.01, 1.0)
        k = np.float32(2.002 * np.log(255 * o)) if 255 * o > 1 else np.float32(0)
        yield np.float32(u), np.float32(v), Q[0, 0], Q[0, 1], Q[1, 1], k


def test_rectangle_minimum_against_bounded_least_squares():
    rng = np.random.default_rng(1)
    for _ in range(3000):
        M = rng.normal(size=(2, 2))
        Q = M @ M.T + 0.05 * np.eye(2)
        A, B, C = Q[0, 0], Q[0, 1], Q[1, 1]
        x0, y0 = rng.uniform(-30, 30, 2)
        x1, y1 = x0 + rng.uniform(0, 20), y0 + rng.uniform(0, 20)
        got = oracle.quad_min_rect(A, B, C, x0, x1, y0, y1)
        ref = lsq_min(A, B, C, x0, x1, y0, y1)
        assert abs(got - ref) <= 1e-9 * max(1.0, ref), (A, B, C, x0, x1, y0, y1, got, ref)


def test_rectangle_minimum_closed_form_axis_aligned():
    # B = 0: the minimum is A dist(0, [x0, x1])^2 + C dist(0, [y0, y1])^2
    dist = lambda a, b: 0.0 if a <= 0 <= b else min(abs(a), abs(b))
    rng = np.random.default_rng(2)
    for _ in range(500):
        A, C = rng.uniform(0.01, 3, 2)
        x0, y0 = rng.uniform(-30, 30, 2)
        x1, y1 = x0 + rng.uniform(0, 20), y0 + rng.uniform(0, 20)
        ref = A * dist(x0, x1) ** 2 + C * dist(y0, y1) ** 2
        assert abs(oracle.quad_min_rect(A, 0.0, C, x0, x1, y0, y1) - ref) <= 1e-12 * max(1, ref)
    # a hand case: unit circle scaled by 1/sigma^2 = 1/25 at (8, 8); tile (1, 0) starts at x = 16,
    # 8 px away: q = 64 / 25 = 2.56, kept for k = 2.56 (1 + 2e-5) and dropped for k = 2.56 (1 - 2e-5)
    cam = scenes.procedural_camera(64, 64)
    for k, kept in ((2.56 * (1 + 2e-5), 1), (2.56 * (1 - 2e-5), 0)):
        rect, codes = oracle.ellipse_tiles(cam, 8.0, 8.0, 0.04, 0.0, 0.04, k, 1 << 20, widen=0.0)
        xl, xh, yl, yh = rect
        assert codes[0 - yl, 1 - xl] & 1 == kept and codes[0 - yl, 1 - xl] & 2 == 0


def test_decisions_against_pixel_centres_bounding_box_and_least_squares():
    rng = np.random.default_rng(0)
    cam = scenes.procedural_camera(200, 136)
    TX, TY = (cam.width + 15) // 16, (cam.height + 15) // 16
    px, py = np.meshgrid(np.arange(16 * TX, dtype=np.float64), np.arange(16 * TY, dtype=np.float64))
    n_amb = n_dec = 0
    for u, v, A, B, C, k in random_splats(rng, 250, cam):
        rect, codes = oracle.ellipse_tiles(cam, u, v, A, B, C, k, 1 << 20)  # the square does not bind
        assert rect == (0, TX, 0, TY)
        kept, amb = (codes & 1) != 0, (codes & 2) != 0
        n_amb += int(amb.sum())
        n_dec += codes.size
        Ad, Bd, Cd, kd = float(A), float(B), float(C), float(k)
        # every tile holding a pixel centre inside the ellipse is kept
        dx, dy = px - float(u), py - float(v)
        inside = (Ad * dx * dx + 2 * Bd * dx * dy + Cd * dy * dy) <= kd * (1 - 1e-5)
        hit = inside.reshape(TY, 16, TX, 16).any(axis=(1, 3))
        assert not (hit & ~kept & ~amb).any()
        # nothing outside the ellipse's bounding box |dx| <= sqrt(k C / det), |dy| <= sqrt(k A / det)
        det = Ad * Cd - Bd * Bd
        ex, ey = (np.sqrt(kd * Cd / det), np.sqrt(kd * Ad / det)) if kd > 0 else (-1.0, -1.0)
        for ty in range(TY):
            for tx in range(TX):
                x0, x1 = 16 * tx - float(u), 16 * tx + 15 - float(u)
                y0, y1 = 16 * ty - float(v), 16 * ty + 15 - float(v)
                if x1 < -ex - 1e-9 or x0 > ex + 1e-9 or y1 < -ey - 1e-9 or y0 > ey + 1e-9:
                    assert not kept[ty, tx]
                    continue
                if amb[ty, tx]:
                    continue
                m = lsq_min(Ad, Bd, Cd, x0, x1, y0, y1)
                assert kept[ty, tx] == (m <= kd), (u, v, A, B, C, k, ty, tx, m)
    assert n_amb <= 0.01 * n_dec


def test_radius_square_bounds_the_kept_tiles():
    rng = np.random.default_rng(3)
    cam = scenes.procedural_camera(200, 136)
    TX, TY = (cam.width + 15) // 16, (cam.height + 15) // 16
    for u, v, A, B, C, k in random_splats(rng, 200, cam):
        (_, _, _, _), full = oracle.ellipse_tiles(cam, u, v, A, B, C, k, 1 << 20)
        r = int(rng.integers(3, 40))
        (xl, xh, yl, yh), sub = oracle.ellipse_tiles(cam, u, v, A, B, C, k, r)
        assert (xl, xh) == (int(np.clip(np.floor((u - r) / 16), 0, TX)), int(np.clip(np.floor((u + r) / 16) + 1, 0, TX)))
        assert (yl, yh) == (int(np.clip(np.floor((v - r) / 16), 0, TY)), int(np.clip(np.floor((v + r) / 16) + 1, 0, TY)))
        assert np.array_equal(sub, full[yl:yh, xl:xh])


def test_binning_is_the_square_binning_restricted_to_kept_tiles():
    g, cam = scenes.tiny_scene(seed=0)
    P = oracle.project(cam, g, prec=32)
    m2, dp, rd = P["means2d"].astype(np.float32), P["depth"].astype(np.float32), P["radius"]
    con = P["conic"].astype(np.float32)
    o = g.opacity.astype(np.float64)
    k = np.where(255 * o > 1, 2.002 * np.log(np.maximum(255 * o, 1)), 0).astype(np.float32)
    Bs = oracle.bin(cam, m2, dp, rd)
    Be = oracle.bin_ellipse(cam, m2, dp, rd, con, k)
    assert 0 < Be["n_entries"] < Bs["n_entries"]
    # per tile: the ellipse list is the square list with some Gaussians removed, in the same order
    for t in range(cam.n_tiles):
        s0, s1 = Bs["ranges"][t]
        e0, e1 = Be["ranges"][t]
        sq = list(Bs["point_list"][s0:s1])
        el = list(Be["point_list"][e0:e1])
        it = iter(sq)
        assert all(x in it for x in el)  # subsequence
    # each Gaussian's count is the number of tiles the test keeps for it, and its knife edges are
    # the ones listed
    amb = {(int(i), int(t)) for i, t in Be["ambiguous"]}
    for i in np.flatnonzero(rd > 0)[:300]:
        (xl, xh, yl, yh), codes = oracle.ellipse_tiles(cam, m2[0, i], m2[1, i], con[0, i], con[1, i], con[2, i],
                                                       k[i], rd[i])
        assert Be["tiles_touched"][i] == int((codes & 1).sum())
        listed = {t for j, t in amb if j == i}
        assert listed == {(yl + a) * cam.tiles_x + xl + b for a, b in zip(*np.nonzero(codes & 2))}
        assert Be["ambiguous_gaussian"][i] == bool(listed)
