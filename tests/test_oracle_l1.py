"""Pins of the oracle's L1 loss term (c8; rigel README, training: "L1 + D-SSIM"), CPU only.

The gradient is checked against one-sided finite differences of the oracle's own loss value
away from ties (|d| is linear there, so the difference quotient is exact up to rounding), and
the loss and gradient against a hand-worked example."""
import numpy as np

import oracle


def test_hand_example():
    img = np.array([0.5, 0.2, 0.3, -1.0])
    tgt = np.array([0.2, 0.2, 0.7, 1.0])
    g, loss = oracle.l1_loss_grad(img, tgt, 0.25)
    # |d| = 0.3, 0, 0.4, 2.0 -> 0.25 * 2.7; signs +, 0 (tie), -, -
    assert np.allclose(loss, 0.675, rtol=0, atol=1e-15)
    assert np.array_equal(g, [0.25, 0.0, -0.25, -0.25])


def test_gradient_is_the_difference_quotient_of_the_loss():
    rng = np.random.default_rng(3)
    img = rng.standard_normal((3, 7, 5))
    tgt = rng.standard_normal((3, 7, 5))
    scale = 1.0 / img.size
    g, L0 = oracle.l1_loss_grad(img, tgt, scale)
    h = 1e-7  # far below every |image - target| of this sample
    assert np.abs(img - tgt).min() > 10 * h
    for idx in [(0, 0, 0), (1, 3, 2), (2, 6, 4), (0, 5, 1)]:
        e = np.zeros_like(img)
        e[idx] = h
        _, L1 = oracle.l1_loss_grad(img + e, tgt, scale)
        assert abs((L1 - L0) / h - g[idx]) < 1e-6 * scale + 1e-12
    assert g.shape == img.shape


def test_zero_at_equality_and_symmetry():
    x = np.array([1.0, -2.0, 3.5])
    g, loss = oracle.l1_loss_grad(x, x, 1.0)
    assert loss == 0.0 and not g.any()
    g1, l1 = oracle.l1_loss_grad(x, -x, 2.0)
    g2, l2 = oracle.l1_loss_grad(-x, x, 2.0)
    assert l1 == l2 and np.array_equal(g1, -g2)
