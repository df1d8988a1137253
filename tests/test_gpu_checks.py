"""The compositing kernels' checks of caller data (rs.h RS_ERR_DEVICE_CHECK): a point-list entry
>= n and a tile range past the list's capacity are skipped, flagged and reported by
rs_device_error, and nothing is read outside the buffers.  A skipped entry counts as examined but
transparent: the image equals the oracle's with that entry pointing at a Gaussian of opacity 0."""
import numpy as np
import pytest
import torch

import oracle
from gaussian_splatting_tile_gb300 import pipeline, rs, scenes

from . import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gaussian_splatting_tile_gb300 import build_lib
    build_lib.build()
    oracle.build()
    assert torch.cuda.is_available()


def rendered(seed=0):
    g, cam = scenes.tiny_scene(seed=seed)
    dev = torch.device("cuda:0")
    dg = rs.DeviceGaussians.from_numpy(g, dev)
    R = pipeline.Renderer(cam, g.n, dev, keep_keys=False)
    R.forward(dg)
    torch.cuda.synchronize()
    assert rs.rs_device_error() == rs.RS_OK
    return g, cam, dg, R


def outputs_like(R):
    return torch.empty_like(R.image), torch.empty_like(R.final_T), torch.empty_like(R.n_contrib)


def test_entry_out_of_range_is_skipped_and_reported():
    g, cam, dg, R = rendered()
    ranges = R.tile_ranges.cpu().numpy().view(np.uint32).astype(np.int64)
    t = int(np.argmax(ranges[:, 1] - ranges[:, 0]))  # the longest list
    e = int(ranges[t, 0])                              # its front entry
    pl = R.point_list.clone()
    pl[e] = g.n + 5
    img, fT, nc = outputs_like(R)
    rs.rs_rasterize_fwd(cam, R.proj, g.n, R.tile_ranges, pl, (0.0, 0.0, 0.0), img, fT, nc, R.raster_ws)
    assert rs.rs_device_error() == rs.RS_ERR_DEVICE_CHECK
    assert rs.rs_device_error() == rs.RS_OK  # the flag was cleared
    # the oracle on the GPU's projection, the entry pointing at an extra Gaussian of opacity 0
    m2 = np.c_[R.proj.means2d.cpu().numpy(), np.zeros((2, 1), np.float32)]
    con = np.c_[R.proj.conic.cpu().numpy(), np.ones((3, 1), np.float32)]
    col = np.c_[R.proj.color.cpu().numpy(), np.zeros((3, 1), np.float32)]
    op = np.r_[g.opacity, np.zeros(1, np.float32)]
    plo = R.point_list[: R.n_entries].cpu().numpy().view(np.uint32).copy()
    plo[e] = g.n
    O = oracle.raster_fwd(cam, m2, con, op, col, ranges.astype(np.uint32), plo)
    clear = O["ambig"] == 0
    assert np.array_equal(nc.cpu().numpy().view(np.uint32)[clear], O["n_contrib"][clear])
    assert np.abs(img.cpu().numpy() - O["image"])[:, clear].max() <= P.IMG_ATOL
    # the list as the binning wrote it gives the unchanged image again, with no flag
    img2, fT2, nc2 = outputs_like(R)
    rs.rs_rasterize_fwd(cam, R.proj, g.n, R.tile_ranges, R.point_list, (0.0, 0.0, 0.0), img2, fT2, nc2,
                        R.raster_ws)
    assert rs.rs_device_error() == rs.RS_OK
    assert torch.equal(img2, R.image) and torch.equal(nc2, R.n_contrib)


def test_range_past_the_capacity_draws_the_tile_empty_and_is_reported():
    g, cam, dg, R = rendered(seed=1)
    ranges = R.tile_ranges.clone()
    rr = ranges.cpu().numpy().view(np.uint32)
    t = int(np.argmax(rr[:, 1].astype(np.int64) - rr[:, 0]))
    cap = R.point_list.numel()
    bad = np.array([cap - 10, cap + 100], np.uint32).view(np.int32)
    ranges[t] = torch.from_numpy(bad).to(ranges.device)
    img, fT, nc = outputs_like(R)
    rs.rs_rasterize_fwd(cam, R.proj, g.n, ranges, R.point_list, (0.0, 0.0, 0.0), img, fT, nc, R.raster_ws)
    assert rs.rs_device_error() == rs.RS_ERR_DEVICE_CHECK
    ty, tx = divmod(t, cam.tiles_x)
    ys, xs = slice(16 * ty, min(16 * ty + 16, cam.height)), slice(16 * tx, min(16 * tx + 16, cam.width))
    assert (fT[ys, xs] == 1.0).all() and (nc[ys, xs] == 0).all() and (img[:, ys, xs] == 0.0).all()
    # every other tile as before
    keep = torch.ones_like(R.final_T, dtype=torch.bool)
    keep[ys, xs] = False
    assert torch.equal(img[:, keep], R.image[:, keep]) and torch.equal(nc[keep], R.n_contrib[keep])
    # the backward over the same ranges skips the tile too and reports it
    dL = torch.from_numpy(scenes.image_grad(cam)).to(img.device)
    n = g.n
    gr = [torch.empty(k * n, dtype=torch.float32, device=img.device) for k in (2, 3, 1, 3)]
    rs.rs_rasterize_bwd(cam, R.proj, n, ranges, R.point_list, (0.0, 0.0, 0.0), fT, nc, R.raster_ws, dL, *gr)
    assert rs.rs_device_error() in (rs.RS_ERR_DEVICE_CHECK, rs.RS_OK)
    assert all(torch.isfinite(x).all() for x in gr)


def test_backward_twice_on_one_forward():
    # the backward hands out its work through a counter in the workspace that the forward zeroes;
    # the call leaves it at zero, so a second backward on the same forward state covers every
    # chunk again (the gradients agree up to the order of the atomic additions)
    g, cam, dg, R = rendered(seed=2)
    dL = torch.from_numpy(scenes.image_grad(cam)).to(R.image.device)
    n = g.n
    runs = []
    for _ in range(3):
        gr = [torch.empty(k * n, dtype=torch.float32, device=R.image.device) for k in (2, 3, 1, 3)]
        rs.rs_rasterize_bwd(cam, R.proj, n, R.tile_ranges, R.point_list, (0.0, 0.0, 0.0), R.final_T, R.n_contrib,
                            R.raster_ws, dL, *gr)
        torch.cuda.synchronize()
        assert rs.rs_device_error() == rs.RS_OK
        runs.append(gr)
    for a, b in zip(runs[0], runs[2]):
        assert torch.count_nonzero(a) > 0
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-6 * float(a.abs().max()))
