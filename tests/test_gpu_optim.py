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


def densify_inputs(n, seed):
    rng = np.random.default_rng(seed)
    f = lambda a: np.ascontiguousarray(a, np.float32)
    return dict(accum=f(rng.exponential(3e-4, n)), count=f(rng.integers(0, 5, n)),
                log_scales=f(rng.uniform(np.log(1e-3), np.log(0.8), (3, n))), logits=f(rng.normal(0, 3, n)),
                quats=f(rng.standard_normal((4, n))), means=f(rng.standard_normal((3, n))),
                sh=f(rng.standard_normal((48, n))), noise=f(rng.standard_normal((2, 3, n))),
                m=[f(rng.standard_normal((r, n))) for r in (3, 3, 4, 1, 48)],
                v=[f(rng.exponential(1.0, (r, n))) for r in (3, 3, 4, 1, 48)])


@pytest.mark.parametrize("n", [100_003, 1])
def test_densify_matches_oracle(n):
    """rs_densify_plan + rs_densify_apply over five parameter groups (means, log-scales,
    quaternions, opacity logits, 48 SH coefficients) with their Adam moments, against the oracle:
    the same fate for every Gaussian whose decisions are not knife edges (at knife edges the GPU's
    fate is given to the oracle: either is correct); every array and its moments of one length;
    copies and moments bit for bit; split children's means within float32 rounding of R(q) (s * z)
    and log-scales within one float32 step of log(s / 1.6)."""
    TAU, DENSE, MIN_OP, MAX_SC = 2e-4, 0.05, 0.005, 0.5
    h = densify_inputs(n, seed=3)
    d = {k: torch.from_numpy(v).cuda() for k, v in h.items() if k not in ("m", "v")}
    dm = [torch.from_numpy(x).cuda() for x in h["m"]]
    dv = [torch.from_numpy(x).cuda() for x in h["v"]]
    ws = torch.empty(rs.rs_densify_workspace_size(n), dtype=torch.uint8, device="cuda")
    act = torch.full((n,), 255, dtype=torch.uint8, device="cuda")
    counts = rs.rs_densify_plan(d["accum"], d["count"], d["log_scales"], d["logits"], TAU, DENSE, MIN_OP, MAX_SC, ws,
                                act)
    oa, amb, oc = oracle.densify_classify(h["accum"], h["count"], h["log_scales"], h["logits"], TAU, DENSE, MIN_OP,
                                          MAX_SC)
    ga = act.cpu().numpy().astype(np.int32)
    assert np.array_equal(ga[~amb], oa[~amb])
    assert amb.mean() < 1e-3
    action = np.where(amb, ga, oa).astype(np.int32)
    n_out = counts["n_out"]
    assert n_out == int(((action == 1) | (action == 2)).sum() + (action == 2).sum() + 2 * (action == 3).sum())
    if not amb.any():
        assert counts == oc
    params = [(d["means"], rs.RS_DENSIFY_MEANS), (d["log_scales"], rs.RS_DENSIFY_LOG_SCALES),
              (d["quats"], rs.RS_DENSIFY_COPY), (d["logits"], rs.RS_DENSIFY_COPY), (d["sh"], rs.RS_DENSIFY_COPY)]
    groups = []
    for (p, kind), m, v in zip(params, dm, dv):
        rows = p.numel() // n
        o = lambda: torch.full((rows, max(n_out, 1)), float("nan"), device="cuda")
        groups.append(rs.DensifyGroup(p.contiguous(), o(), m, v, o(), o(), kind))
    rs.rs_densify_apply(n, ws, d["quats"], d["log_scales"], d["noise"], groups, n_out)
    torch.cuda.synchronize()
    host_params = [h["means"], h["log_scales"], h["quats"], h["logits"][None], h["sh"]]
    for k, (gr, p, m, v) in enumerate(zip(groups, host_params, h["m"], h["v"])):
        po, mo, vo = oracle.densify_group(action, p, m, v, kind=gr.kind, quats=h["quats"],
                                          log_scales=h["log_scales"], noise=h["noise"])
        gp, gm, gv = (x.cpu().numpy()[:, :n_out].astype(np.float64) for x in (gr.param_out, gr.m_out, gr.v_out))
        assert gp.shape == po.shape == gm.shape == gv.shape  # one length for every array and its moments
        assert np.array_equal(gm, mo) and np.array_equal(gv, vo), k
        new = np.zeros(n_out, bool)
        new[int(((action == 1) | (action == 2)).sum()):] = True
        split_part = np.zeros(n_out, bool)
        split_part[n_out - 2 * int((action == 3).sum()):] = True
        if gr.kind == rs.RS_DENSIFY_COPY:
            assert np.array_equal(gp, po), k
        else:
            assert np.array_equal(gp[:, ~split_part], po[:, ~split_part]), k
            tol = 1e-6 * (np.abs(po[:, split_part]) + 1.0)
            assert (np.abs(gp[:, split_part] - po[:, split_part]) <= tol).all(), k
