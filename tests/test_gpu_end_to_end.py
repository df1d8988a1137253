"""The path as the benchmark runs it, checked against the oracle.

1. Graph-captured frames with several views in flight: each renderer (capacity 4 M entries, no
   keys kept, as the benchmark's headline) replays its view's CUDA graph on its own stream; the
   projection, binning, compositing and both backward passes of every replay are compared with
   the oracle stage by stage (the rigel README's "Binning" sync removed by rs_bin_async; the
   graph is the pages' next step).
2. pipeline.StreamedFrames (the end-to-end path: Gaussians and dL/dimage from pinned host
   memory, gradients back to pinned host memory, copies overlapping compute): the last frame
   of every slot against the oracle, gradients read from the host buffers.
3. The full pipeline from the raw Gaussians (the rigel README "Numbers", full-pipeline row):
   the GPU's image and gradients against the oracle's own projection, binning, compositing and
   backward, with no GPU value fed to the oracle.  Knife edges are flagged in double precision:
   tiles whose lists hold a Gaussian with a knife-edge projection decision, or whose lists differ
   only in the order of Gaussians at equal float32 depth, are left out, and pixels whose
   compositing decisions are knife edges get no upstream gradient, on both sides.
"""
import numpy as np
import pytest
import torch

import oracle
from gaussian_splatting_tile_gb300 import pipeline, rs, scenes

from . import parity as P

pytestmark = pytest.mark.gpu
BG = (0.0, 0.0, 0.0)


@pytest.fixture(scope="module", autouse=True)
def built():
    from gaussian_splatting_tile_gb300 import build_lib
    build_lib.build()
    oracle.build()
    assert torch.cuda.is_available()


def sampled_tiles(cam, count, seed):
    rng = np.random.default_rng(seed)
    tm = np.zeros(cam.n_tiles, np.uint8)
    tm[rng.choice(cam.n_tiles, min(count, cam.n_tiles), replace=False)] = 1
    return tm


def replay_in_flight(frames):
    """Replays every frame graph on a stream of its own, all joined to the current stream (the
    benchmark's headline); returns the entry counts."""
    main = torch.cuda.current_stream()
    sides = [torch.cuda.Stream() for _ in frames]
    for side, fg in zip(sides, frames):
        side.wait_stream(main)
        with torch.cuda.stream(side):
            fg.replay()
    for side in sides:
        main.wait_stream(side)
    torch.cuda.synchronize()
    return [fg.check() for fg in frames]


def precomputed_backward(grads_of):
    """run_backward for check_raster_backward when the GPU's gradients were produced already
    (by a graph replay or a streamed frame) from the upstream gradient `used`."""
    def run(G, dL):
        used, grads = grads_of(G)
        assert np.array_equal(np.asarray(dL, np.float32), used), "the GPU ran on another dL/dimage"
        G.update(grads)
        G["dL"] = dL
    return run


def test_headline_graph_frames_in_flight_against_oracle():
    g = scenes.procedural_scene(seed=0)
    dg = rs.DeviceGaussians.from_numpy(g)
    orbit = scenes.orbit_cameras(1920, 1080)
    sq720 = scenes.procedural_camera(720, 720, focal=700.0)
    setups = [(orbit, 0), (orbit, 20), (orbit, 40), ([sq720], 0)]
    runs = []
    for i, (cams, v) in enumerate(setups):
        cam = cams[v]
        tm = sampled_tiles(cam, 96, seed=10 + i)
        pm = P.pixel_mask_of_tiles(cam, tm)
        dL_host = (scenes.image_grad(cam) * pm[None]).astype(np.float32)
        dL = torch.from_numpy(dL_host).cuda()
        R = pipeline.Renderer(cam, g.n, capacity=4_000_000, keep_keys=False)
        fg = pipeline.FrameGraphs(R, dg, dL, cams).get(v)
        runs.append(dict(cam=cam, tm=tm, dL=dL, dL_host=dL_host, R=R, fg=fg))
    # first replay: forward against the oracle, and the knife-edge pixels of each view
    E = replay_in_flight([r["fg"] for r in runs])
    for r, e in zip(runs, E):
        G = P.renderer_state(r["R"], dg, e)
        P.check_projection(r["cam"], g, G)
        P.check_binning(r["cam"], G)
        r["fwd"] = P.check_forward(r["cam"], g, G, BG, tile_mask=r["tm"])
        r["G"] = G
        amb = r["fwd"]["O"]["ambig"] != 0
        r["dL_host"][:, amb] = 0.0
        r["dL"].copy_(torch.from_numpy(r["dL_host"]))
    # second replay, reading the zeroed dL/dimage: the same forward, gradients against the oracle
    E2 = replay_in_flight([r["fg"] for r in runs])
    assert E2 == E
    for r in runs:
        G = r["G"]
        assert np.array_equal(r["R"].image.cpu().numpy(), G["image"])
        grads = P.grads_into({}, r["R"].grads)
        run = precomputed_backward(lambda G, r=r, grads=grads: (r["dL_host"], grads))
        P.check_raster_backward(r["cam"], g, G, BG, r["fwd"], r["dL_host"], tile_mask=r["tm"], run_backward=run)
        P.check_project_backward(r["cam"], g, G)
    assert min(E) > 300_000


def test_streamed_frames_against_oracle():
    g = scenes.procedural_scene(seed=2, n_sphere=15_000, n_helix=4_000, n_plane=4_000)
    cams = [scenes.procedural_camera(320, 240, azimuth=a) for a in (0.3, 1.9, 3.4)]
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).pin_memory()
    host = dict(means=pin(g.means), scales=pin(g.scales), quats=pin(g.quats), opacity=pin(g.opacity),
                sh=pin(g.sh))
    dL_host = pin(scenes.image_grad(cams[0]))
    slots = 4
    S = pipeline.StreamedFrames(cams, host, g.sh_degree, dL_host, slots=slots)
    views = [0, 1, 2, 1, 0, 2, 2, 0]
    last = {s: views[max(k for k in range(len(views)) if k % slots == s)] for s in range(slots)}

    def run_all():
        S.prepare(views)
        for v in views:
            S.frame(v)
        return S.finish()

    counts = run_all()
    assert len(counts) == len(views) and min(counts) > 0
    # forward of each slot's last frame against the oracle; the knife-edge pixels of all of them
    states, amb = {}, np.zeros((cams[0].height, cams[0].width), bool)
    for s in range(slots):
        sl = S.slots[s]
        E = sl["graphs"].get(last[s]).check()  # the pinned count of the slot's last replay
        G = P.renderer_state(sl["R"], sl["dg"], E)
        cam = cams[last[s]]
        P.check_projection(cam, g, G)
        P.check_binning(cam, G)
        fwd = P.check_forward(cam, g, G, BG)
        amb |= fwd["O"]["ambig"] != 0
        states[s] = (G, fwd)
    # the frames again, dL/dimage zero at those pixels; gradients from the host buffers
    dL_host[:, torch.from_numpy(amb)] = 0.0
    run_all()
    dLz = dL_host.numpy().copy()
    for s in range(slots):
        sl = S.slots[s]
        G, fwd = states[s]
        cam = cams[last[s]]
        assert np.array_equal(sl["R"].image.cpu().numpy(), G["image"])
        grads = {k: getattr(sl["R"].grads, k).cpu().numpy() for k in ("dmeans2d", "dconic", "dcolor")}
        grads.update({k: sl["host_out"][k].numpy().copy() for k in ("dmeans", "dscales", "dquats", "dopacity", "dsh")})
        run = precomputed_backward(lambda G, grads=grads: (dLz, grads))
        P.check_raster_backward(cam, g, G, BG, fwd, dLz, run_backward=run)
        P.check_project_backward(cam, g, G)


def oracle_chain(cam, g, proj, B, n_contrib, dL, bg, keep):
    """The oracle's compositing backward and projection backward from projected values `proj`."""
    Rb = oracle.raster_bwd(cam, proj["means2d"], proj["conic"], g.opacity, proj["color"], B["ranges"],
                           B["point_list"], n_contrib, dL, bg=bg, tile_mask=keep)
    Pb = oracle.project_bwd(cam, g, proj["radius"], Rb["dmeans2d"], Rb["dconic"], Rb["dcolor"])
    return {**Rb, **Pb}


def full_pipeline_check(g, cam, bg, tile_mask=None, max_excluded=0.12):
    """The GPU path from the raw Gaussians against the oracle's own pipeline (see the module
    docstring); returns the share of tiles left out.  With a few hundred entries per tile, about
    one tile in twenty holds a Gaussian at a knife edge or two at equal float32 depth (at most
    `max_excluded` of the tiles may be left out; the stage checks cover every tile exactly).

    End to end, the GPU's stages read its own float32 projection where the oracle's read double
    values, so a gradient can differ by what that rounding moves it (the mean's gradient, a
    difference of large per-pixel terms, is the most sensitive).  The oracle measures this
    itself: it runs its compositing and backward chain again on projections rounded or perturbed
    at float32's resolution (its own float32 projection, and two random relative perturbations of
    2^-23 of its double one), and four times the largest change is added to the tolerance of the
    image, final_T and every gradient (with the float32 summation bound for the gradients)."""
    G = P.run_gpu(g, cam, bg)
    O = oracle.project(cam, g, prec=64, margin=P.MARGIN)
    B = oracle.bin(cam, O["means2d"].astype(np.float32), O["depth"].astype(np.float32), O["radius"])
    tm = np.ones(cam.n_tiles, np.uint8) if tile_mask is None else tile_mask.astype(np.uint8)
    amb_g = O["ambig"] != 0
    depth = O["depth"].astype(np.float32).astype(np.float64)
    gr, orr = G["ranges"].reshape(-1, 2), B["ranges"]
    keep = tm.copy()
    for t in np.flatnonzero(tm):
        lg = G["point_list"][gr[t, 0]:gr[t, 1]]
        lo = B["point_list"][orr[t, 0]:orr[t, 1]]
        if np.array_equal(lg, lo):
            continue
        # admissible differences: Gaussians whose projection decisions (cull, radius, span) are
        # knife edges present on one side only, or Gaussians of equal float32 depth in another order
        diff = np.setxor1d(lg, lo)
        assert amb_g[diff].all(), f"tile {t}: the lists differ in Gaussians with clear decisions"
        common = np.intersect1d(lg, lo)
        a, b = lg[np.isin(lg, common)], lo[np.isin(lo, common)]
        if not np.array_equal(a, b):
            d = depth[a]
            assert (np.diff(d) >= -2e-6 * np.abs(d[:-1])).all(), f"tile {t}: the GPU's list is out of depth order"
        keep[t] = 0
    excluded = 1.0 - keep.sum() / max(1, tm.sum())
    assert excluded <= max_excluded, excluded
    F = oracle.raster_fwd(cam, O["means2d"], O["conic"], g.opacity, O["color"], B["ranges"], B["point_list"],
                          bg=bg, prec=64, margin=P.MARGIN, tile_mask=keep)
    O32 = oracle.project(cam, g, prec=32)
    rng = np.random.default_rng(0)
    perturbed = [dict(O32, radius=O["radius"])]
    for _ in range(2):
        perturbed.append(dict(radius=O["radius"], **{
            k: O[k] * (1 + 2.0 ** -23 * rng.uniform(-1, 1, O[k].shape)) for k in ("means2d", "conic", "color")}))
    sens_img, sens_T = 0.0, 0.0
    for pp in perturbed:
        Fp = oracle.raster_fwd(cam, pp["means2d"], pp["conic"], g.opacity, pp["color"], B["ranges"],
                               B["point_list"], bg=bg, prec=64, tile_mask=keep)
        sens_img = np.maximum(sens_img, np.abs(Fp["image"] - F["image"]))
        sens_T = np.maximum(sens_T, np.abs(Fp["final_T"] - F["final_T"]))
    clear = P.pixel_mask_of_tiles(cam, keep) & (F["ambig"] == 0)
    assert clear.sum() > 0.9 * P.pixel_mask_of_tiles(cam, keep).sum()
    # the stop decision (T < 1e-4) can move with the projection's rounding: n_contrib equal on
    # >= 99.9% of the clear pixels, and the others get no upstream gradient on either side
    same_n = G["n_contrib"] == F["n_contrib"]
    assert same_n[clear].mean() >= 0.999, same_n[clear].mean()
    P.allclose_report("image", G["image"], F["image"], 0.0, P.IMG_ATOL, mask=clear, extra=4 * sens_img)
    P.allclose_report("final_T", G["final_T"], F["final_T"], 0.0, P.IMG_ATOL, mask=clear, extra=4 * sens_T)
    clear &= same_n
    dL = (scenes.image_grad(cam) * clear[None]).astype(np.float32)
    P.run_gpu_backward(G, dL)
    ref = oracle_chain(cam, g, O, B, F["n_contrib"], dL, bg, keep)
    sens = {}
    for pp in perturbed:
        ch = oracle_chain(cam, g, pp, B, F["n_contrib"], dL, bg, keep)
        for k in ("dmeans2d", "dconic", "dopacity", "dcolor", "dmeans", "dscales", "dquats", "dsh"):
            if ref.get(k) is not None:
                sens[k] = np.maximum(sens.get(k, 0.0), np.abs(ch[k] - ref[k]))
    for k in ("dmeans2d", "dconic", "dopacity", "dcolor"):
        P.allclose_report(k, G[k], ref[k], P.GRAD_RTOL, P.GRAD_ATOL, extra=4 * sens[k] + P.SUM_EPS * ref["abs_" + k])
    # the projection backward of Gaussians whose forward decisions are knife edges (cull, radius,
    # span, the clamp branch of the Jacobian) may legitimately differ
    ok = ~amb_g
    for k in ("dmeans", "dscales", "dquats") + (("dsh",) if G["dsh"] is not None else ()):
        P.allclose_report(k, G[k], ref[k], P.GRAD_RTOL, P.GRAD_ATOL, mask=ok, extra=4 * sens[k])
    return excluded


@pytest.mark.parametrize("bg", [(0.0, 0.0, 0.0), (0.25, 0.5, 1.0)])
def test_full_pipeline_tiny(bg):
    g, cam = scenes.tiny_scene(seed=0)
    full_pipeline_check(g, cam, bg)


def test_full_pipeline_sh_degree3_ragged():
    g = scenes.procedural_scene(seed=1, n_sphere=12_000, n_helix=4_000, n_plane=4_000)
    cam = scenes.procedural_camera(200, 136, azimuth=0.4)
    full_pipeline_check(g, cam, (0.1, 0.2, 0.3))


def test_full_pipeline_160k_720_sampled_tiles():
    g = scenes.procedural_scene(seed=0)
    cam = scenes.procedural_camera(720, 720, focal=700.0)
    full_pipeline_check(g, cam, BG, tile_mask=sampled_tiles(cam, 96, seed=7))
