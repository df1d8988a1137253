"""GPU parity of the appearance MLP, the L1 loss term and the training-shaped step (the
five-stage step of rigel's appearance-MLP model: MLP forward, rasteriser forward, L1 loss,
rasteriser backward, MLP backward) against the oracle, through the C ABI.

Tolerances:
  - MLP colours: |c - c_ref| <= 1e-5 + 1e-4 |c_ref|.  The products run in TF32 with split
    operands (relative error about 2^-21 per product); the second layer sums 64 terms of order
    one, and the sigmoid's slope is at most 1/4.
  - gradients: rel 1e-3 / abs 1e-5 as everywhere else.  In the training step dL/dimage is
    +-scale, and the sign of (image - target) is spatially coherent, so a Gaussian's upstream
    sums grow with its pixel count instead of its square root as they do for dL/dimage ~ N(0,1);
    fp32 rounding grows with them.  There the absolute part is 1e-5 x the largest |reference|
    of each output array (and at least 1e-5 x scale).
  - relu knife edges: a hidden pre-activation within 1e-4 of zero may switch the relu's slope
    between the two sides (both are correct); the colour gradient of such a Gaussian is set to
    zero on both sides before the MLP backward.
  - L1: the sign of a float difference is exact, so dL/dimage is bit-exact; the loss is a float
    sum with rel 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
from gaussian_splatting_tile_gb300 import pipeline, rs, scenes

from .parity import (GRAD_ATOL, GRAD_RTOL, allclose_report, check_binning, check_forward,
                     check_project_backward, check_projection, check_raster_backward, gpu_state)

pytestmark = pytest.mark.gpu

KNIFE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    from gaussian_splatting_tile_gb300 import build_lib
    build_lib.build()


def camera_centre(cam):
    R = np.asarray(cam.R, np.float64).reshape(3, 3)
    return -R.T @ np.asarray(cam.t, np.float64).reshape(3)


def relu_knife_edges(cam, means, latents, W1, b1):
    """Gaussians with a hidden pre-activation within KNIFE of zero (double precision)."""
    d = np.asarray(means, np.float64) - camera_centre(cam)[:, None]
    d /= np.linalg.norm(d, axis=0, keepdims=True)
    x = np.concatenate([np.asarray(latents, np.float64), d], axis=0)
    z1 = np.asarray(W1, np.float64) @ x + np.asarray(b1, np.float64)[:, None]
    return (np.abs(z1) < KNIFE).any(axis=0)


def mlp_params(rng, L, H, bias=0.1):
    a1 = np.sqrt(6.0 / (L + 3 + H))
    a2 = np.sqrt(6.0 / (H + 3))
    return dict(W1=rng.uniform(-a1, a1, (H, L + 3)).astype(np.float32),
                b1=(bias * rng.standard_normal(H)).astype(np.float32),
                W2=rng.uniform(-a2, a2, (3, H)).astype(np.float32),
                b2=(bias * rng.standard_normal(3)).astype(np.float32))


@pytest.mark.parametrize("n,L,H,seed", [(1007, 8, 64, 0), (333, 29, 32, 1), (17, 1, 64, 2), (64, 13, 32, 3)])
def test_mlp_matches_oracle(n, L, H, seed):
    rng = np.random.default_rng(seed)
    cam = scenes.procedural_camera(64, 48)
    means = rng.uniform(-1.5, 1.5, (3, n)).astype(np.float32)
    latents = rng.standard_normal((L, n)).astype(np.float32)
    p = mlp_params(rng, L, H)
    dcol = rng.standard_normal((3, n)).astype(np.float32)
    knife = relu_knife_edges(cam, means, latents, p["W1"], p["b1"])
    dcol[:, knife] = 0.0
    mlp = rs.DeviceMLP.from_numpy(p)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    colors = torch.full((3, n), float("nan"), device="cuda")
    rs.rs_appearance_fwd(cam, t(means), t(latents), mlp, colors)
    dlat = torch.full((L, n), float("nan"), device="cuda")
    grads = rs.DeviceMLPGrads.like(mlp)
    for v in (grads.dW1, grads.db1, grads.dW2, grads.db2):
        v.fill_(float("nan"))  # the call zeroes its weight gradients itself
    rs.rs_appearance_bwd(cam, t(means), t(latents), mlp, t(dcol), dlat, grads)
    torch.cuda.synchronize()
    ref = oracle.appearance_fwd(cam, means, latents, p["W1"], p["b1"], p["W2"], p["b2"])
    allclose_report("colors", colors.cpu().numpy(), ref, 1e-4, 1e-5)
    O = oracle.appearance_bwd(cam, means, latents, p["W1"], p["b1"], p["W2"], p["b2"], dcol)
    allclose_report("dlatents", dlat.cpu().numpy(), O["dlatents"], GRAD_RTOL, GRAD_ATOL)
    for k in ("dW1", "db1", "dW2", "db2"):
        allclose_report(k, getattr(grads, k).cpu().numpy(), O[k], GRAD_RTOL, GRAD_ATOL)


@pytest.mark.parametrize("H", [64, 32])
def test_mlp_many_tiles_per_block(H):
    # 300k Gaussians: more 128-row tiles than the forward launches blocks, so each block walks
    # several tiles (tensor memory and the completion barrier are reused across them)
    n, L = 300_000, 8
    rng = np.random.default_rng(11 + H)
    cam = scenes.procedural_camera(64, 48, azimuth=0.7)
    means = rng.uniform(-1.5, 1.5, (3, n)).astype(np.float32)
    latents = rng.standard_normal((L, n)).astype(np.float32)
    p = mlp_params(rng, L, H)
    dcol = rng.standard_normal((3, n)).astype(np.float32)
    dcol[:, relu_knife_edges(cam, means, latents, p["W1"], p["b1"])] = 0.0
    mlp = rs.DeviceMLP.from_numpy(p)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    colors = torch.full((3, n), float("nan"), device="cuda")
    rs.rs_appearance_fwd(cam, t(means), t(latents), mlp, colors)
    dlat = torch.full((L, n), float("nan"), device="cuda")
    grads = rs.DeviceMLPGrads.like(mlp)
    rs.rs_appearance_bwd(cam, t(means), t(latents), mlp, t(dcol), dlat, grads)
    torch.cuda.synchronize()
    ref = oracle.appearance_fwd(cam, means, latents, p["W1"], p["b1"], p["W2"], p["b2"])
    allclose_report("colors", colors.cpu().numpy(), ref, 1e-4, 1e-5)
    O = oracle.appearance_bwd(cam, means, latents, p["W1"], p["b1"], p["W2"], p["b2"], dcol)
    allclose_report("dlatents", dlat.cpu().numpy(), O["dlatents"], GRAD_RTOL, GRAD_ATOL)
    # weight gradients are sums over 300k Gaussians: the absolute part scales with the largest sum
    for k in ("dW1", "db1", "dW2", "db2"):
        allclose_report(k, getattr(grads, k).cpu().numpy(), O[k], GRAD_RTOL, GRAD_ATOL, atol_of_max=1e-5)
    # no block gave up waiting for its tensor-core products
    assert rs.rs_device_error() == rs.RS_OK


def test_mlp_empty():
    cam = scenes.procedural_camera(64, 48)
    p = mlp_params(np.random.default_rng(5), 8, 64)
    mlp = rs.DeviceMLP.from_numpy(p)
    e = torch.empty(3, 0, device="cuda")
    grads = rs.DeviceMLPGrads.like(mlp)
    for v in (grads.dW1, grads.db1, grads.dW2, grads.db2):
        v.fill_(1.0)
    rs.rs_appearance_fwd(cam, e, torch.empty(8, 0, device="cuda"), mlp, e)
    rs.rs_appearance_bwd(cam, e, torch.empty(8, 0, device="cuda"), mlp, e, torch.empty(8, 0, device="cuda"), grads)
    torch.cuda.synchronize()
    for v in (grads.dW1, grads.db1, grads.dW2, grads.db2):
        assert not v.any()


def test_l1_matches_oracle():
    rng = np.random.default_rng(7)
    img = rng.uniform(0, 1, (3, 123, 77)).astype(np.float32)
    tgt = rng.uniform(0, 1, (3, 123, 77)).astype(np.float32)
    tgt[:, ::5, ::3] = img[:, ::5, ::3]  # exact ties: gradient 0
    scale = 1.0 / img.size
    dimg = torch.full(img.shape, float("nan"), device="cuda")
    loss = torch.full((1,), float("nan"), device="cuda")
    rs.rs_l1_loss_grad(torch.from_numpy(img).cuda(), torch.from_numpy(tgt).cuda(), scale, dimg, loss)
    torch.cuda.synchronize()
    g_ref, l_ref = oracle.l1_loss_grad(img, tgt, scale)
    assert np.array_equal(dimg.cpu().numpy(), g_ref.astype(np.float32))
    assert abs(float(loss.item()) - l_ref) <= 1e-5 * abs(l_ref)


def test_training_shaped_step():
    """250,000 Gaussians (sphere / helix / plane), 8 views of 400x400, MLP 11 -> 64 -> 3,
    L1 loss against the oracle's render of the same Gaussians with their procedural colours,
    scale 1 / (3 H W V).  Every stage of every view is checked against the oracle (each oracle
    stage fed the GPU's upstream outputs)."""
    g, cams, p = scenes.training_scene()
    V = len(cams)
    H, W = cams[0].height, cams[0].width
    scale = 1.0 / (3 * H * W * V)
    atol = GRAD_ATOL * scale
    frac = GRAD_ATOL
    dg = rs.DeviceGaussians.from_numpy(g)
    mlp = rs.DeviceMLP.from_numpy(p)
    lat = torch.from_numpy(p["latents"]).cuda()
    step = pipeline.AppearanceStep(cams[0], dg, mlp, lat)
    bg = (0.0, 0.0, 0.0)
    for v, cam in enumerate(cams):
        target = oracle.render(cam, g)[2]["image"].astype(np.float32)
        F = step.forward(cam, torch.from_numpy(target).cuda(), scale, bg=bg)
        torch.cuda.synchronize()
        G = gpu_state(step.R, step.gc, F)
        colors = step.colors.cpu().numpy()
        # MLP forward, then projection with the oracle's own colours
        ref = oracle.appearance_fwd(cam, g.means, p["latents"], p["W1"], p["b1"], p["W2"], p["b2"])
        allclose_report(f"view {v} colors", colors, ref, 1e-4, 1e-5)
        gref = scenes.Gaussians(g.means, g.scales, g.quats, g.opacity, None, -1, ref)
        check_projection(cam, gref, G)
        check_binning(cam, G)
        fwd = check_forward(cam, g, G, bg)
        # L1: bit-exact gradient, loss as a float sum
        d_ref, l_ref = oracle.l1_loss_grad(G["image"], target, scale)
        dimg = step.dL_dimage.cpu().numpy()
        assert np.array_equal(dimg, d_ref.astype(np.float32)), f"view {v}: L1 gradient"
        assert abs(float(step.loss.item()) - l_ref) <= 1e-5 * abs(l_ref) + 1e-9
        # compositing and projection backward from the GPU's L1 gradient
        check_raster_backward(cam, g, G, bg, fwd, dimg, atol=atol, atol_of_max=frac)
        gcol = scenes.Gaussians(g.means, g.scales, g.quats, g.opacity, None, -1, colors)
        check_project_backward(cam, gcol, G, atol=atol, atol_of_max=frac)
        # MLP backward from the GPU's colour gradient (zero at relu knife edges on both sides)
        dcol = np.array(G["dcolor"], np.float32)
        dcol[:, relu_knife_edges(cam, g.means, p["latents"], p["W1"], p["b1"])] = 0.0
        step.mlp_backward(torch.from_numpy(dcol).cuda())
        torch.cuda.synchronize()
        O = oracle.appearance_bwd(cam, g.means, p["latents"], p["W1"], p["b1"], p["W2"], p["b2"], dcol)
        allclose_report(f"view {v} dlatents", step.dL_dlatents.cpu().numpy(), O["dlatents"], GRAD_RTOL, atol,
                        atol_of_max=frac)
        for k in ("dW1", "db1", "dW2", "db2"):
            allclose_report(f"view {v} {k}", getattr(step.mlp_grads, k).cpu().numpy(), O[k], GRAD_RTOL, atol,
                            atol_of_max=frac)


@pytest.mark.parametrize("shape,lam", [((3, 37, 53), 0.2), ((3, 400, 400), 0.2), ((1, 5, 3), 0.5), ((2, 16, 16), 1.0)])
def test_l1_dssim_matches_oracle(shape, lam):
    """L1 + D-SSIM: gradient |g - g_ref| <= 1e-3 |g_ref| + 1e-5 max|g_ref| (float32 window sums of
    order one, the SSIM quotients and the 121-tap adjoint), loss rel 1e-5; two calls in a row on
    the same workspace give the same result."""
    rng = np.random.default_rng(sum(shape))
    img = rng.uniform(0, 1, shape).astype(np.float32)
    tgt = np.clip(img + 0.2 * rng.standard_normal(shape), 0, 1).astype(np.float32)
    scale = 0.125
    ws = torch.empty(rs.rs_l1_dssim_workspace_size(*shape), dtype=torch.uint8, device="cuda")
    t = lambda a: torch.from_numpy(a).cuda()
    out = []
    for _ in range(2):
        d = torch.full(shape, float("nan"), device="cuda")
        loss = torch.full((1,), float("nan"), device="cuda")
        rs.rs_l1_dssim_loss_grad(t(img), t(tgt), lam, scale, d, loss, ws)
        torch.cuda.synchronize()
        out.append((d.cpu().numpy(), float(loss.item())))
    g_ref, l_ref, _ = oracle.l1_dssim(img, tgt, lam, scale)
    for d, loss in out:
        allclose_report("dL/dimage", d, g_ref, 1e-3, 1e-5 * float(np.abs(g_ref).max()))
        assert abs(loss - l_ref) <= 1e-5 * abs(l_ref)
