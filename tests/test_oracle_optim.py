"""Pins of the oracle's Adam step (c9) and densification statistics (c10), CPU only.

Adam is checked against torch.optim.Adam (an independent implementation) in float64 over
several steps, with the activation's chain rule taken by autograd; the statistics against a
hand example."""
import numpy as np
import pytest
import torch

import oracle


@pytest.mark.parametrize("activation", [0, 1, 2])
def test_adam_matches_torch_over_steps(activation):
    rng = np.random.default_rng(activation)
    n, lr, b1, b2, eps = 257, 0.01, 0.9, 0.999, 1e-15
    p0 = rng.standard_normal(n) * (0.5 if activation else 1.0)
    p = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([p], lr=lr, betas=(b1, b2), eps=eps)
    act = {0: lambda x: x, 1: torch.exp, 2: torch.sigmoid}[activation]
    mine, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for step in range(1, 5):
        g_act = rng.standard_normal(n)  # gradient w.r.t. the activated value
        opt.zero_grad()
        (act(p) * torch.from_numpy(g_act)).sum().backward()  # autograd applies act'(p)
        opt.step()
        mine, m, v, a = oracle.adam_step(mine, g_act, m, v, lr, activation, b1, b2, eps, step)
        ref = p.detach().numpy()
        assert np.allclose(mine, ref, rtol=1e-12, atol=1e-14)
        assert np.allclose(a, act(p).detach().numpy(), rtol=1e-12, atol=1e-14)


def test_adam_first_step_moves_by_lr_times_sign():
    # with zero moments the bias-corrected first step is lr * g / (|g| + eps)
    g = np.array([2.0, -0.5, 0.0, 1e-3])
    p, m, v, _ = oracle.adam_step(np.zeros(4), g, np.zeros(4), np.zeros(4), 0.1, eps=1e-12)
    assert np.allclose(p, [-0.1, 0.1, 0.0, -0.1], atol=1e-9)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)


def test_densify_stats_hand_example():
    dm2 = np.array([[3.0, 1.0, 0.0], [4.0, 0.0, 2.0]])
    radius = np.array([5, 0, 1], np.int32)
    a, c = oracle.densify_stats(dm2, radius, np.array([1.0, 1.0, 1.0]), np.array([2.0, 2.0, 2.0]))
    assert np.array_equal(a, [6.0, 1.0, 3.0]) and np.array_equal(c, [3.0, 2.0, 3.0])
