"""GPU parity of the fused Adam step (rs_adam_step) and the densification statistics
(rs_densify_stats) against the oracle, through the C ABI.

Tolerances: the kernel runs float32, the oracle float64 on the same float32 inputs, each side
carrying its own state across steps.  A step moves a parameter by at most lr and is computed to
about 1e-6 of itself in float32, and each step rounds the stored parameter to float32 (half an
ulp, 6e-8 relative); after 5 steps |p - p_ref| <= 1e-3 lr + 4e-7 |p_ref|.  The first moment is
a running sum of gradients of order one that can cancel, so it agrees to 2e-6 absolute (a few
float32 ulps of its terms) + rel 1e-5; the second moment (positive terms) to rel 1e-5."""
import numpy as np
import pytest
import torch

import oracle
from gaussian_splatting_tile_gb300 import rs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gaussian_splatting_tile_gb300 import build_lib
    build_lib.build()


def test_adam_matches_oracle_over_steps():
    rng = np.random.default_rng(11)
    specs = [(3 * 1007, 1.6e-4, rs.RS_ACT_IDENTITY), (3 * 1007, 5e-3, rs.RS_ACT_EXP),
             (1007, 5e-2, rs.RS_ACT_SIGMOID), (48 * 1007 - 5, 1.25e-4, rs.RS_ACT_IDENTITY), (0, 1e-3, 0)]
    host = []
    groups = []
    for k, lr, act in specs:
        p0 = (rng.standard_normal(k) * (0.5 if act else 1.0) - (3.0 if act == rs.RS_ACT_EXP else 0.0)).astype(np.float32)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
        gr = rs.AdamGroup(t(p0), torch.zeros(k, device="cuda"), torch.zeros(k, device="cuda"),
                          torch.zeros(k, device="cuda"), lr, act,
                          torch.full((k,), float("nan"), device="cuda") if act else None)
        groups.append(gr)
        host.append(dict(p=p0.astype(np.float64), m=np.zeros(k), v=np.zeros(k), lr=lr, act=act))
    for step in range(1, 6):
        for gr, h in zip(groups, host):
            g = rng.standard_normal(gr.param.numel()).astype(np.float32)
            gr.grad.copy_(torch.from_numpy(g))
            h["g"] = g
        rs.rs_adam_step(groups, step, 0.9, 0.999, 1e-15)
        for h in host:
            h["p"], h["m"], h["v"], h["a"] = oracle.adam_step(h["p"], h["g"], h["m"], h["v"], h["lr"], h["act"],
                                                             0.9, 0.999, 1e-15, step)
    torch.cuda.synchronize()
    for gr, h in zip(groups, host):
        if gr.param.numel() == 0:
            continue
        assert np.allclose(gr.param.cpu().numpy(), h["p"], rtol=4e-7, atol=1e-3 * h["lr"])
        assert np.allclose(gr.m.cpu().numpy(), h["m"], rtol=1e-5, atol=2e-6)
        assert np.allclose(gr.v.cpu().numpy(), h["v"], rtol=1e-5, atol=1e-9)
        if gr.activated is not None:
            assert np.allclose(gr.activated.cpu().numpy(), h["a"], rtol=1e-5, atol=1e-7)


def test_densify_stats_match_oracle():
    rng = np.random.default_rng(12)
    n = 5003
    dm2 = rng.standard_normal((2, n)).astype(np.float32)
    radius = np.where(rng.uniform(size=n) < 0.2, 0, rng.integers(1, 40, n)).astype(np.int32)
    acc0 = rng.uniform(0, 1, n).astype(np.float32)
    cnt0 = rng.integers(0, 5, n).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    acc, cnt = t(acc0), t(cnt0)
    rs.rs_densify_stats(t(dm2), t(radius), acc, cnt)
    torch.cuda.synchronize()
    a_ref, c_ref = oracle.densify_stats(dm2, radius, acc0, cnt0)
    assert np.allclose(acc.cpu().numpy(), a_ref, rtol=1e-6, atol=1e-7)
    assert np.array_equal(cnt.cpu().numpy(), c_ref.astype(np.float32))
