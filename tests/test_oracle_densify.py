"""Pins of the oracle's densification (c12: clone, split, prune; rigel README "GaussianModel:
activations, densify/prune"; criteria of 3D Gaussian Splatting's adaptive density control), CPU
only: a hand-built example through every branch with its output order written out; split offsets
in closed form for the identity and a 90-degree rotation; the children's sample covariance
against the projection's 3D covariance (itself pinned against scipy's Rotation); and the rule of
the rigel README's model tests: every parameter array and its Adam moments come out the same
length."""
import numpy as np

import oracle
from gaussian_splatting_tile_gb300 import scenes

TAU, DENSE, MIN_OP, MAX_SC = 2e-4, 0.05, 0.005, 0.5
LOGIT = lambda o: np.log(o / (1 - o))


def hand_case():
    # i: 0 keep (small gradient); 1 clone (large gradient, small); 2 split (large gradient, large);
    #    3 removed (faint); 4 removed (large gradient but faint: its clone or children would be);
    #    5 removed (larger than max_scale); 6 split whose children (s / 1.6) are still too large;
    #    7 no views (count 0): kept; 8 clone; 9 split
    accum = np.array([1e-4, 9e-4, 9e-4, 0, 9e-4, 0, 9e-4, 5.0, 6e-4, 1e-3])
    count = np.array([1, 3, 3, 1, 3, 1, 1, 0, 2, 4], float)
    big = np.log(0.2)  # > dense (0.05), and 0.2 / 1.6 < max_scale
    small = np.log(0.01)
    huge = np.log(0.7)  # > max_scale
    top = np.log(0.9)   # split, children 0.9 / 1.6 = 0.5625 > 0.5
    ls_max = [small, small, big, small, small, huge, top, small, small, big]
    log_scales = np.full((3, 10), np.log(0.001))
    log_scales[1] = ls_max  # the largest of the three
    logits = np.full(10, LOGIT(0.5))
    logits[[3, 4]] = LOGIT(0.001)
    return accum, count, log_scales, logits


def test_hand_example_every_branch_and_order():
    accum, count, log_scales, logits = hand_case()
    action, amb, counts = oracle.densify_classify(accum, count, log_scales, logits, TAU, DENSE, MIN_OP, MAX_SC)
    assert action.tolist() == [1, 2, 3, 0, 0, 0, 0, 1, 2, 3]
    assert not amb.any()
    assert counts == dict(n_out=4 + 2 + 4, kept=4, cloned=2, split=2, removed=4)
    # order: kept originals (0, 1, 7, 8), clones (1, 8), first children (2, 9), second children (2, 9)
    ids = np.arange(10, dtype=np.float64)[None]
    out, _, _ = oracle.densify_group(action, ids)
    assert out[0].tolist() == [0, 1, 7, 8, 1, 8, 2, 9, 2, 9]


def test_moments_follow_the_originals_and_start_at_zero_for_new_gaussians():
    accum, count, log_scales, logits = hand_case()
    action, _, counts = oracle.densify_classify(accum, count, log_scales, logits, TAU, DENSE, MIN_OP, MAX_SC)
    p = np.arange(20, dtype=np.float64).reshape(2, 10)
    m, v = p + 100, p + 200
    po, mo, vo = oracle.densify_group(action, p, m, v)
    assert po.shape == mo.shape == vo.shape == (2, counts["n_out"])
    assert mo[:, :4].tolist() == m[:, [0, 1, 7, 8]].tolist() and vo[:, :4].tolist() == v[:, [0, 1, 7, 8]].tolist()
    assert not mo[:, 4:].any() and not vo[:, 4:].any()


def test_split_offsets_closed_form():
    n = 2
    action = np.array([3, 3], np.int32)
    means = np.array([[1.0, -2.0], [0.5, 0.0], [3.0, 1.0]])
    log_scales = np.log(np.array([[0.1, 0.2], [0.3, 0.05], [0.02, 0.4]]))
    # Gaussian 0: identity; Gaussian 1: 90 degrees about z, q = (cos 45, 0, 0, sin 45) (scaled by 3:
    # any norm)
    c = np.cos(np.pi / 4)
    quats = np.array([[1.0, 3 * c], [0.0, 0.0], [0.0, 0.0], [0.0, 3 * c]])
    z = np.random.default_rng(0).standard_normal((2, 3, n))
    out, _, _ = oracle.densify_group(action, means, kind=1, quats=quats, log_scales=log_scales, noise=z)
    s = np.exp(log_scales)
    for ch in range(2):
        o0 = out[:, ch * 2 + 0] - means[:, 0]
        assert np.allclose(o0, s[:, 0] * z[ch, :, 0], rtol=0, atol=1e-15)
        # R_z(90) (a, b, c) = (-b, a, c)
        a, b, cc = s[:, 1] * z[ch, :, 1]
        assert np.allclose(out[:, ch * 2 + 1] - means[:, 1], [-b, a, cc], rtol=0, atol=1e-14)
    lo, _, _ = oracle.densify_group(action, log_scales, kind=2)
    assert np.allclose(np.exp(lo[:, [0, 2]]), s[:, [0, 0]] / 1.6, rtol=1e-14)


def test_children_sample_the_gaussians_3d_covariance():
    g, _ = scenes.tiny_scene(seed=4, n=3)
    n_draw = 200_000
    i = 1
    means = np.repeat(g.means[:, i:i + 1].astype(np.float64), n_draw, axis=1)
    quats = np.repeat(g.quats[:, i:i + 1].astype(np.float64), n_draw, axis=1)
    log_scales = np.repeat(np.log(g.scales[:, i:i + 1].astype(np.float64)), n_draw, axis=1)
    z = np.random.default_rng(1).standard_normal((2, 3, n_draw))
    out, _, _ = oracle.densify_group(np.full(n_draw, 3, np.int32), means, kind=1, quats=quats,
                                     log_scales=log_scales, noise=z)
    d = out - means[:, :1]
    cov = d @ d.T / d.shape[1]
    cov3 = oracle.project_intermediates(scenes.look_at([0, 0, 4.0], [0, 0, 0], 100, 100, 64, 64), g)["cov3d"][:, i]
    ref = np.array([[cov3[0], cov3[1], cov3[2]], [cov3[1], cov3[3], cov3[4]], [cov3[2], cov3[4], cov3[5]]])
    # the sample covariance of 400k draws: relative error ~ sqrt(2 / 4e5) = 0.2% of the diagonal
    assert np.allclose(cov, ref, rtol=0, atol=0.01 * np.abs(np.diag(ref)).max())


def test_every_parameter_and_its_moments_keep_one_length():
    rng = np.random.default_rng(2)
    n = 5000
    accum = rng.exponential(3e-4, n)
    count = rng.integers(0, 5, n).astype(float)
    log_scales = rng.uniform(np.log(1e-3), np.log(0.8), (3, n))
    logits = rng.normal(0, 3, n)
    quats = rng.standard_normal((4, n))
    means = rng.standard_normal((3, n))
    action, amb, counts = oracle.densify_classify(accum, count, log_scales, logits, TAU, DENSE, MIN_OP, MAX_SC)
    assert counts["kept"] > 0 and counts["cloned"] > 0 and counts["split"] > 0 and counts["removed"] > 0
    assert counts["n_out"] == counts["kept"] + counts["cloned"] + 2 * counts["split"]
    assert counts["kept"] + counts["split"] + counts["removed"] == n
    z = rng.standard_normal((2, 3, n))
    groups = [(means, 1), (log_scales, 2), (quats, 0), (logits[None], 0), (rng.standard_normal((3, n)), 0),
              (rng.standard_normal((45, n)), 0)]
    for p, kind in groups:
        po, mo, vo = oracle.densify_group(action, p, p * 0 + 1, p * 0 + 2, kind=kind, quats=quats,
                                          log_scales=log_scales, noise=z)
        assert po.shape[1] == mo.shape[1] == vo.shape[1] == counts["n_out"]
