"""Pins of the oracle's L1 + D-SSIM loss (c11), CPU only: the gradient against central
differences of the oracle's own loss, SSIM(x, x) = 1 with a vanishing SSIM gradient, the
closed form of SSIM between constant images away from the border, symmetry, and lambda = 0
reducing to the L1 term."""
import numpy as np

import oracle


def test_gradient_matches_central_differences():
    rng = np.random.default_rng(0)
    img = rng.uniform(0, 1, (2, 9, 13))
    tgt = rng.uniform(0, 1, (2, 9, 13))
    g, L0, _ = oracle.l1_dssim(img, tgt, 0.2, 1.0)
    h = 1e-6
    for idx in [(0, 0, 0), (0, 4, 6), (1, 8, 12), (1, 2, 11), (0, 7, 1)]:
        e = np.zeros_like(img)
        e[idx] = h
        _, Lp, _ = oracle.l1_dssim(img + e, tgt, 0.2, 1.0)
        _, Lm, _ = oracle.l1_dssim(img - e, tgt, 0.2, 1.0)
        assert abs(img[idx] - tgt[idx]) > 10 * h  # away from the L1 kink
        assert abs((Lp - Lm) / (2 * h) - g[idx]) < 1e-7


def test_identity_and_symmetry():
    rng = np.random.default_rng(1)
    x = rng.uniform(0, 1, (3, 12, 10))
    y = rng.uniform(0, 1, (3, 12, 10))
    g, L, s = oracle.l1_dssim(x, x, 1.0, 1.0)
    assert np.allclose(s, 1.0, atol=1e-12) and abs(L) < 1e-12 and np.abs(g).max() < 1e-12
    _, _, s1 = oracle.l1_dssim(x, y)
    _, _, s2 = oracle.l1_dssim(y, x)
    assert np.allclose(s1, s2, atol=1e-14)


def test_constant_images_closed_form():
    a, b = 0.7, 0.3
    x = np.full((1, 15, 17), a)
    y = np.full((1, 15, 17), b)
    _, _, s = oracle.l1_dssim(x, y)
    C1 = 0.01 ** 2
    inner = s[0, 5:-5, 5:-5]  # windows entirely inside the image: zero variances
    assert np.allclose(inner, (2 * a * b + C1) / (a * a + b * b + C1), rtol=1e-12)


def test_lambda_zero_is_the_l1_term():
    rng = np.random.default_rng(2)
    x = rng.uniform(0, 1, (2, 6, 7))
    y = rng.uniform(0, 1, (2, 6, 7))
    g, L, _ = oracle.l1_dssim(x, y, 0.0, 3.0)
    g1, L1 = oracle.l1_loss_grad(x, y, 3.0 / x.size)
    assert np.allclose(g, g1, rtol=1e-14, atol=0) and abs(L - L1) < 1e-14
