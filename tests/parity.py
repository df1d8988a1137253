"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, then the oracle on the
same seeded inputs, stage by stage (each oracle stage consumes the GPU's upstream outputs, so a
stage is judged on its own arithmetic), and compare.

Tolerances (rigel README "Numbers"; the target the tests hold the path to):
  - binning: keys, point lists and tile ranges bit-exact given identical projected inputs;
  - forward compositing: n_contrib equal on >= 99.9% of pixels; image and final_T within
    max-abs 1e-4 on every pixel whose decisions (skip at 1/255, stop at T < 1e-4) are not
    within a relative 1e-5 of their thresholds in double precision;
  - gradients: |g - g_ref| <= 1e-5 + 1e-3 |g_ref| for every Gaussian, with the upstream
    gradient set to zero (on both sides) at the few knife-edge pixels, where either decision
    is correct and the two sides may legitimately differ.  The compositing backward's outputs
    are sums over pixels of terms that can cancel; no float32 computation of such a sum is more
    accurate than a small multiple of eps32 x (the sum of the terms' magnitudes), which the
    oracle reports, so that bound (SUM_EPS x the magnitude sum) is added to the tolerance.
  - projection values: |x - x_ref| <= 1e-5 + 2e-4 |x_ref| (fp32 arithmetic over a few dozen
    operations on quantities with condition numbers up to a few hundred); for the pixel
    position u = fx x/z + cx the rounding scales with the summed terms, not the result, so
    |u - u_ref| <= 1e-5 + 2e-4 |u_ref| + 1e-6 (|u_ref| + max(cx, cy)); integer outputs
    (cull, radius, tiles) exact where no decision is within 1e-5 of its threshold.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gaussian_splatting_tile_gb300 import pipeline, rs, scenes

MARGIN = 1e-5
GRAD_RTOL, GRAD_ATOL = 1e-3, 1e-5
SUM_EPS = 32 * 2.0 ** -24  # float32 rounding of a cancelling sum, per unit of its magnitude sum
IMG_ATOL = 1e-4


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def renderer_state(R, dg, E):
    """Host copies of the forward outputs a renderer's buffers hold (E entries), with the renderer
    and Gaussians for the backward.  `keys` is None when the renderer does not keep the keys."""
    P = R.proj
    keys = None if R.keys_sorted is None else R.keys_sorted[:E].cpu().numpy().view(np.uint64)
    return dict(renderer=R, dg=dg, n_entries=E,
                means2d=P.means2d.cpu().numpy(), depth=P.depth.cpu().numpy(),
                conic=P.conic.cpu().numpy(), color=P.color.cpu().numpy(),
                radius=P.radius.cpu().numpy(), tiles_touched=u32(P.tiles_touched),
                keys=keys, point_list=u32(R.point_list[:E]), ranges=u32(R.tile_ranges),
                image=R.image.cpu().numpy(), final_T=R.final_T.cpu().numpy(),
                n_contrib=u32(R.n_contrib))


def gpu_state(R, dg, F):
    """Host copies of a forward's outputs, with the renderer and Gaussians for the backward."""
    return renderer_state(R, dg, F.n_entries)


def grads_into(G, grads):
    """Host copies of a renderer's gradient buffers into G."""
    G.update({k: getattr(grads, k).cpu().numpy() for k in
              ("dmeans2d", "dconic", "dopacity", "dcolor", "dmeans", "dscales", "dquats")})
    G["dsh"] = None if grads.dsh is None else grads.dsh.cpu().numpy()
    return G


def run_gpu(g, cam, bg=(0.0, 0.0, 0.0)):
    """Forward through the C ABI; returns host copies plus the renderer for the backward."""
    dg = rs.DeviceGaussians.from_numpy(g)
    R = pipeline.Renderer(cam, g.n)
    F = R.forward(dg, bg=bg)
    torch.cuda.synchronize()
    return gpu_state(R, dg, F)


def run_gpu_backward(G, dL):
    """Backward through the C ABI with upstream gradient dL [3,H,W]; fills G's gradients."""
    R = G["renderer"]
    B = R.backward(G["dg"], torch.from_numpy(np.ascontiguousarray(dL, np.float32)).cuda())
    torch.cuda.synchronize()
    grads_into(G, B)
    G["dL"] = dL
    return G


def allclose_report(name, got, ref, rtol, atol, mask=None, extra=None, atol_of_max=0.0):
    """|got - ref| <= atol + rtol |ref| (+ extra) elementwise; with atol_of_max the absolute part
    is at least atol_of_max x max |ref| over the array."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if atol_of_max and ref.size:
        atol = max(atol, atol_of_max * float(np.abs(ref).max()))
    if extra is not None:
        extra = np.broadcast_to(np.asarray(extra, np.float64), ref.shape)
    if mask is not None:
        got, ref = got[..., mask], ref[..., mask]
        if extra is not None:
            extra = extra[..., mask]
    err = np.abs(got - ref)
    tol = atol + rtol * np.abs(ref) + (0.0 if extra is None else extra)
    bad = err > tol
    if bad.any():
        w = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside |d| <= {atol} + {rtol}|ref| (+ extra); "
                             f"worst |d| = {err.max():.3e}; worst relative to its tolerance at {w}: got "
                             f"{got[w]:.9g}, ref {ref[w]:.9g}, tol {tol[w]:.3e}")
    return float(err.max()) if err.size else 0.0


def check_projection(cam, g, G, min_clear=0.995):
    """min_clear: the share of Gaussians with no knife-edge decision the check insists on.  The
    tile-span decisions compare (u +- r) / 16 with integers at a margin relative to u, so at the
    same scene density their knife-edge share grows with the image's pixel coordinates (0.4% of
    the Gaussians at 1080p, 0.8% at 3840 x 2160, 1.2% at 4608 x 4096)."""
    O64 = oracle.project(cam, g, prec=64, margin=MARGIN)
    O32 = oracle.project(cam, g, prec=32)
    clear = O64["ambig"] == 0
    assert clear.mean() > min_clear
    # integer decisions: exact where not at a knife edge (taken in float, the kernel's precision)
    assert np.array_equal(G["radius"][clear], O32["radius"][clear])
    assert np.array_equal(G["tiles_touched"][clear], O32["tiles_touched"][clear])
    assert (G["radius"] == O32["radius"]).mean() >= 0.999
    vis = clear & (G["radius"] > 0) & (O64["radius"] > 0)
    r = {}
    centre = max(abs(float(cam.cx)), abs(float(cam.cy)))
    r["means2d"] = allclose_report("means2d", G["means2d"], O64["means2d"], 2e-4, 1e-5, vis,
                                   extra=1e-6 * (np.abs(O64["means2d"]) + centre))
    for k in ("depth", "conic", "color"):
        r[k] = allclose_report(k, G[k], O64[k], 2e-4, 1e-5, vis)
    culled = G["radius"] == 0
    assert not G["conic"][:, culled].any() and not G["tiles_touched"][culled].any()
    return r


def check_binning(cam, G):
    B = oracle.bin(cam, G["means2d"].astype(np.float32), G["depth"].astype(np.float32), G["radius"])
    assert G["n_entries"] == B["n_entries"]
    assert np.array_equal(G["tiles_touched"], B["tiles_touched"])
    if G["keys"] is not None:  # renderers that do not keep the keys write only the point list
        assert np.array_equal(G["keys"], B["keys_sorted"])
    assert np.array_equal(G["point_list"], B["point_list"])
    assert np.array_equal(G["ranges"].reshape(-1, 2), B["ranges"])
    return B


def forward_oracle(cam, g, G, bg, tile_mask=None, prec=64):
    return oracle.raster_fwd(cam, G["means2d"], G["conic"], g.opacity, G["color"],
                             G["ranges"].reshape(-1, 2), G["point_list"], bg=bg, prec=prec,
                             margin=MARGIN, tile_mask=tile_mask)


def pixel_mask_of_tiles(cam, tile_mask):
    TX = cam.tiles_x
    ty = np.arange(cam.height)[:, None] // 16
    tx = np.arange(cam.width)[None, :] // 16
    return tile_mask[ty * TX + tx].astype(bool)


def check_forward(cam, g, G, bg, tile_mask=None):
    O = forward_oracle(cam, g, G, bg, tile_mask)
    pm = np.ones((cam.height, cam.width), bool) if tile_mask is None else pixel_mask_of_tiles(cam, tile_mask)
    eq = (G["n_contrib"] == O["n_contrib"])[pm]
    assert eq.mean() >= 0.999, f"n_contrib equal on {eq.mean():.5f} of pixels"
    clear = pm & (O["ambig"] == 0)
    assert np.array_equal(G["n_contrib"][clear], O["n_contrib"][clear])
    img_err = np.abs(G["image"] - O["image"])[:, clear].max() if clear.any() else 0.0
    t_err = np.abs(G["final_T"] - O["final_T"])[clear].max() if clear.any() else 0.0
    assert img_err <= IMG_ATOL and t_err <= IMG_ATOL, (img_err, t_err)
    return dict(O=O, n_contrib_equal=float(eq.mean()), image_err=float(img_err),
                final_T_err=float(t_err), ambiguous_pixels=int((pm & (O["ambig"] != 0)).sum()))


def check_raster_backward(cam, g, G, bg, fwd, dL, tile_mask=None, atol=GRAD_ATOL, atol_of_max=0.0,
                          run_backward=None):
    """Stage parity of the compositing backward: both sides walk the GPU's n_contrib, and the
    upstream gradient is zeroed at knife-edge pixels on both sides.  run_backward(G, dL) fills
    G's gradients from the GPU (default: the renderer's backward, call by call)."""
    amb = fwd["O"]["ambig"] != 0
    dL = np.array(dL, np.float32)
    dL[:, amb] = 0.0
    (run_backward or run_gpu_backward)(G, dL)
    O = oracle.raster_bwd(cam, G["means2d"], G["conic"], g.opacity, G["color"],
                          G["ranges"].reshape(-1, 2), G["point_list"], G["n_contrib"], dL, bg=bg,
                          tile_mask=tile_mask)
    res = {}
    for k in ("dmeans2d", "dconic", "dopacity", "dcolor"):
        res[k] = allclose_report(k, G[k], O[k], GRAD_RTOL, atol, atol_of_max=atol_of_max,
                                 extra=SUM_EPS * O["abs_" + k])
    return O, res


def check_project_backward(cam, g, G, atol=GRAD_ATOL, atol_of_max=0.0):
    """Stage parity of the projection backward, fed the GPU's own raster gradients."""
    O = oracle.project_bwd(cam, g, G["radius"], G["dmeans2d"], G["dconic"], G["dcolor"])
    res = {}
    for k in ("dmeans", "dscales", "dquats"):
        res[k] = allclose_report(k, G[k], O[k], GRAD_RTOL, atol, atol_of_max=atol_of_max)
    if G["dsh"] is not None:
        res["dsh"] = allclose_report("dsh", G["dsh"], O["dsh"], GRAD_RTOL, atol, atol_of_max=atol_of_max)
    return res
