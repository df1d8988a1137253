"""Pins of the oracle's exact ellipse-tile test (c2', the pages' next binning step), CPU only.

For random splats the tiles the test keeps are compared with brute force in double precision:
every tile holding a pixel centre with d^T Q d <= k must be kept (the test is conservative),
and every kept tile must come within 0.02 px (the widening) of the ellipse with k x (1 + 1e-6)
(the test is tight); with a finite radius the kept tiles lie inside the radius square.  The
binning built on it keeps the (tile, depth) order of the square test's entries restricted to the
kept tiles."""
import numpy as np

import oracle
from gaussian_splatting_tile_gb300 import scenes


def brute_min_over_rect(A, B, C, x0, x1, y0, y1):
    """min of A x^2 + 2 B x y + C y^2 over the rectangle [x0, x1] x [y0, y1] (double)."""
    if x0 <= 0 <= x1 and y0 <= 0 <= y1:
        return 0.0
    best = np.inf
    for X in (x0, x1):
        y = np.clip(-B * X / C, y0, y1)
        best = min(best, A * X * X + 2 * B * X * y + C * y * y)
    for Y in (y0, y1):
        x = np.clip(-B * Y / A, x0, x1)
        best = min(best, A * x * x + 2 * B * x * Y + C * Y * Y)
    return best


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


def test_conservative_and_tight_against_brute_force():
    rng = np.random.default_rng(0)
    cam = scenes.procedural_camera(200, 136)
    TX, TY = (cam.width + 15) // 16, (cam.height + 15) // 16
    for u, v, A, B, C, k in random_splats(rng, 400, cam):
        rows = oracle.ellipse_tiles(cam, u, v, A, B, C, k, 1 << 20)  # the square does not bind
        kept = {(ty, tx) for ty, lo, hi in rows for tx in range(lo, hi + 1)}
        r = int(rng.integers(3, 40))
        sq = lambda p, n: (int(np.clip(np.floor((p - r) / 16), 0, n)), int(np.clip(np.floor((p + r) / 16) + 1, 0, n)))
        (xl, xh), (yl, yh) = sq(float(u), TX), sq(float(v), TY)
        kept_r = {(ty, tx) for ty, lo, hi in oracle.ellipse_tiles(cam, u, v, A, B, C, k, r) for tx in range(lo, hi + 1)}
        assert kept_r == {(ty, tx) for ty, tx in kept if yl <= ty < yh and xl <= tx < xh}
        Ad, Bd, Cd, kd = float(A), float(B), float(C), float(k)
        for ty in range(TY):
            for tx in range(TX):
                x0, x1 = 16 * tx - float(u), 16 * tx + 15 - float(u)
                y0, y1 = 16 * ty - float(v), 16 * ty + 15 - float(v)
                m = brute_min_over_rect(Ad, Bd, Cd, x0, x1, y0, y1)
                if kd > 0 and m <= kd * (1 - 1e-6):
                    assert (ty, tx) in kept, (u, v, A, B, C, k, ty, tx)
                if (ty, tx) in kept:
                    mw = brute_min_over_rect(Ad, Bd, Cd, x0 - 0.02, x1 + 0.02, y0 - 0.02, y1 + 0.02)
                    assert mw <= kd * (1 + 1e-6), (u, v, A, B, C, k, ty, tx, mw)


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
    # and each Gaussian's count is the number of tiles the test keeps for it
    for i in np.flatnonzero(rd > 0)[:200]:
        rows = oracle.ellipse_tiles(cam, m2[0, i], m2[1, i], con[0, i], con[1, i], con[2, i], k[i], rd[i])
        assert Be["tiles_touched"][i] == sum(max(0, hi - lo + 1) for _, lo, hi in rows)
