"""The graph-captured frame (pipeline.FrameGraph): replaying one view's forward + backward as a
single CUDA graph gives the eager frame's outputs -- image, final_T, n_contrib and the binning
bit for bit, the gradients up to the order of their float atomics -- for several views of one
renderer, and a replay reads the current contents of its input buffers."""
import numpy as np
import pytest
import torch

from gaussian_splatting_tile_gb300 import pipeline, rs, scenes

pytestmark = pytest.mark.gpu

GRADS = ("dmeans2d", "dconic", "dopacity", "dcolor", "dmeans", "dscales", "dquats", "dsh")


@pytest.fixture(scope="module", autouse=True)
def built():
    from gaussian_splatting_tile_gb300 import build_lib
    build_lib.build()


def snapshot(R):
    out = {k: getattr(R, k).clone() for k in ("image", "final_T", "n_contrib", "tile_ranges")}
    out["point_list"] = R.point_list[: R.n_entries].clone()
    out.update({k: getattr(R.grads, k).clone() for k in GRADS})
    return out


def eager(R, dg, dL, cam):
    R.set_camera(cam)
    R.forward(dg)
    R.backward(dg, dL)
    torch.cuda.synchronize()
    return snapshot(R)


def same(a, b):
    for k in ("image", "final_T", "n_contrib", "tile_ranges", "point_list"):
        assert torch.equal(a[k], b[k]), k
    for k in GRADS:
        x, y = a[k].double(), b[k].double()
        tol = 1e-5 * float(y.abs().max()) + 1e-12
        assert float((x - y).abs().max()) <= tol, k


def test_frame_graph_replays_the_eager_frame():
    g = scenes.procedural_scene(seed=1, n_sphere=20_000, n_helix=5_000, n_plane=5_000)
    cams = [scenes.procedural_camera(400, 304, azimuth=a) for a in (0.0, 1.3, 2.6)]
    dg = rs.DeviceGaussians.from_numpy(g)
    dL = torch.from_numpy(scenes.image_grad(cams[0])).cuda()
    R = pipeline.Renderer(cams[0], g.n)
    ref = [eager(R, dg, dL, c) for c in cams]
    graphs = pipeline.FrameGraphs(R, dg, dL, cams)
    for v in (1, 0, 2, 1):
        fg = graphs.get(v)
        fg.replay()
        torch.cuda.synchronize()
        assert fg.check() == R.n_entries > 0
        same(snapshot(R), ref[v])
    # the graph reads its inputs' current contents: halve every opacity, compare with eager
    dg.opacity.mul_(0.5)
    ref2 = eager(R, dg, dL, cams[2])
    graphs.get(2).replay()
    torch.cuda.synchronize()
    graphs.get(2).check()
    same(snapshot(R), ref2)
    assert not torch.equal(ref2["image"], ref[2]["image"])


@pytest.mark.parametrize("slots", [2, 4])
def test_streamed_frames_match_eager_frames(slots):
    """pipeline.StreamedFrames (host inputs, host gradients, copies and the slots' compute
    overlapping): the gradients that reach pinned host memory equal the eager frame's, for the
    last frame of every slot; the entry counts match."""
    g = scenes.procedural_scene(seed=2, n_sphere=15_000, n_helix=4_000, n_plane=4_000)
    cams = [scenes.procedural_camera(320, 240, azimuth=a) for a in (0.3, 1.9, 3.4)]
    dL = scenes.image_grad(cams[0])
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).pin_memory()
    host = dict(means=pin(g.means), scales=pin(g.scales), quats=pin(g.quats), opacity=pin(g.opacity),
                sh=pin(g.sh))
    S = pipeline.StreamedFrames(cams, host, g.sh_degree, pin(dL), slots=slots)
    views = [0, 1, 2, 1, 0, 2, 2, 0, 1]
    S.prepare(views)
    for v in views:
        S.frame(v)
    counts = S.finish()
    dg = rs.DeviceGaussians.from_numpy(g)
    R = pipeline.Renderer(cams[0], g.n)
    ref = {v: eager(R, dg, torch.from_numpy(dL).cuda(), cams[v]) for v in set(views)}
    assert all(c > 0 for c in counts) and len(counts) == len(views)
    for slot in range(slots):  # frame k runs in slot k % slots
        last = views[max(k for k in range(len(views)) if k % slots == slot)]
        out = S.host_out[slot]
        for k in ("dmeans", "dscales", "dquats", "dopacity", "dsh"):
            x, y = out[k].double(), ref[last][k].cpu().double()
            tol = 1e-5 * float(y.abs().max()) + 1e-12
            assert float((x - y).abs().max()) <= tol, (slot, k)
