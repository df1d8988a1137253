"""GPU parity: every stage of the CUDA path (called through the C ABI) against the CPU oracle on
the same seeded inputs.  Small scenes are compared element by element; the full-size
workloads are compared in full for projection and binning and on a random sample of tiles for
compositing and its backward (the upstream gradient is zero outside the sampled tiles, so the
GPU's per-Gaussian sums cover exactly the oracle's tiles)."""
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
    import oracle
    oracle.build()
    assert torch.cuda.is_available()


def full_check(g, cam, bg):
    G = P.run_gpu(g, cam, bg)
    P.check_projection(cam, g, G)
    P.check_binning(cam, G)
    fwd = P.check_forward(cam, g, G, bg)
    P.check_raster_backward(cam, g, G, bg, fwd, scenes.image_grad(cam))
    P.check_project_backward(cam, g, G)
    return G, fwd


@pytest.mark.parametrize("bg", [(0.0, 0.0, 0.0), (0.25, 0.5, 1.0)])
def test_tiny_config_all_stages(bg):
    g, cam = scenes.tiny_scene(seed=0)
    G, fwd = full_check(g, cam, bg)
    assert G["n_entries"] > 1000 and fwd["n_contrib_equal"] >= 0.999


def test_sh_degree3_ragged_image():
    # 200 x 136 leaves a partial tile column and row; degree-3 SH exercises the full basis
    g = scenes.procedural_scene(seed=1, n_sphere=12_000, n_helix=4_000, n_plane=4_000)
    cam = scenes.procedural_camera(200, 136, azimuth=0.4)
    full_check(g, cam, (0.1, 0.2, 0.3))


@pytest.mark.parametrize("degree", [-1, 1, 2])
def test_other_colour_sources(degree):
    g = scenes.procedural_scene(seed=2, n_sphere=3000, n_helix=1000, n_plane=1000,
                                sh_degree=max(degree, 0))
    if degree == -1:
        g.colors = np.ascontiguousarray(np.random.default_rng(0).uniform(0, 1, (3, g.n)), np.float32)
        g.sh, g.sh_degree = None, -1
    else:
        K = (degree + 1) ** 2
        g.sh = np.ascontiguousarray(g.sh[:3 * K])
        g.sh_degree = degree
    cam = scenes.procedural_camera(96, 80, azimuth=1.0)
    full_check(g, cam, (0.0, 0.0, 0.0))


def sampled_check(g, cam, n_tiles_sample, seed=0, bg=(0.0, 0.0, 0.0), min_clear=0.995):
    rng = np.random.default_rng(seed)
    tile_mask = np.zeros(cam.n_tiles, np.uint8)
    tile_mask[rng.choice(cam.n_tiles, n_tiles_sample, replace=False)] = 1
    pm = P.pixel_mask_of_tiles(cam, tile_mask)
    dL = scenes.image_grad(cam) * pm[None].astype(np.float32)
    G = P.run_gpu(g, cam, bg)
    P.check_projection(cam, g, G, min_clear=min_clear)
    P.check_binning(cam, G)
    fwd = P.check_forward(cam, g, G, bg, tile_mask=tile_mask)
    P.check_raster_backward(cam, g, G, bg, fwd, dL, tile_mask=tile_mask)
    P.check_project_backward(cam, g, G)
    return G, fwd


def test_full_size_160k_720():
    g = scenes.procedural_scene(seed=0)
    cam = scenes.procedural_camera(720, 720, focal=700.0)
    G, fwd = sampled_check(g, cam, 96)
    assert G["n_entries"] > 300_000


@pytest.mark.parametrize("view", [0, 20, 40])
def test_full_size_160k_1080p_orbit(view):
    g = scenes.procedural_scene(seed=0)
    cam = scenes.orbit_cameras(1920, 1080)[view]
    G, fwd = sampled_check(g, cam, 128, seed=view)
    assert G["n_entries"] > 1_000_000


def test_full_size_160k_720p_orbit():
    g = scenes.procedural_scene(seed=0)
    cam = scenes.orbit_cameras(1280, 720)[10]
    sampled_check(g, cam, 96, seed=3)


def test_full_size_stress_1m():
    g, cam = scenes.stress_scene(seed=0)
    G, fwd = sampled_check(g, cam, 48, seed=4)
    assert G["n_entries"] > 5_000_000


def test_4k_image_tile_ids_of_15_bits():
    # 3840 x 2160 has 32,400 tiles: the tile sort's two passes take 8-bit digits
    g = scenes.procedural_scene(seed=5, n_sphere=25_000, n_helix=7_500, n_plane=7_500)
    cam = scenes.orbit_cameras(3840, 2160)[7]
    assert 16_384 < cam.n_tiles <= 32_768
    G, fwd = sampled_check(g, cam, 64, seed=5, min_clear=0.985)
    assert G["n_entries"] > 500_000


def test_tile_ids_of_17_bits():
    # 4608 x 4096 has 73,728 tiles: three passes of 6-bit digits
    g = scenes.procedural_scene(seed=6, n_sphere=12_000, n_helix=4_000, n_plane=4_000)
    cam = scenes.procedural_camera(4608, 4096, azimuth=2.5)
    assert 65_536 < cam.n_tiles <= 131_072
    G, fwd = sampled_check(g, cam, 64, seed=6, min_clear=0.98)
    assert G["n_entries"] > 100_000


def test_empty_scene_is_background():
    g, cam = scenes.tiny_scene(seed=0, n=0)
    dg = rs.DeviceGaussians.from_numpy(g)
    R = pipeline.Renderer(cam, 0)
    F = R.forward(dg, bg=(0.5, 0.25, 0.125))
    torch.cuda.synchronize()
    assert F.n_entries == 0
    img = F.image.cpu().numpy()
    assert np.all(img[0] == 0.5) and np.all(img[1] == 0.25) and np.all(img[2] == 0.125)
    assert np.all(F.final_T.cpu().numpy() == 1.0) and not F.n_contrib.cpu().numpy().any()


def test_all_culled_and_single_gaussian():
    g, cam = scenes.tiny_scene(seed=5, n=50)
    away = scenes.look_at([0, 0, 4.0], [0, 0, 8.0], 150.0, 150.0, 128, 128)  # looking away
    G = P.run_gpu(g, away)
    assert G["n_entries"] == 0 and not G["radius"].any()
    assert np.all(G["final_T"] == 1.0)
    one = scenes.Gaussians(g.means[:, :1].copy(), g.scales[:, :1].copy(), g.quats[:, :1].copy(),
                           g.opacity[:1].copy(), g.sh[:, :1].copy(), 0)
    one.means[:] = 0.0
    one.scales[:] = 0.05
    G = P.run_gpu(one, cam)
    P.check_projection(cam, one, G)
    P.check_binning(cam, G)
    fwd = P.check_forward(cam, one, G, (0.0, 0.0, 0.0))
    P.check_raster_backward(cam, one, G, (0.0, 0.0, 0.0), fwd, scenes.image_grad(cam))
    P.check_project_backward(cam, one, G)


def test_capacity_overflow_then_retry_matches():
    g, cam = scenes.tiny_scene(seed=0)
    dg = rs.DeviceGaussians.from_numpy(g)
    R = pipeline.Renderer(cam, g.n, capacity=16)
    R.project(dg)
    with pytest.raises(rs.RsError) as e:
        rs.rs_bin(cam, R.proj, g.n, R.workspace, R.capacity, R.keys_sorted, R.point_list, R.tile_ranges)
    assert e.value.code == rs.RS_ERR_CAPACITY and e.value.n_entries > 16
    E = R.bin()  # grows and retries
    assert E == e.value.n_entries and R.capacity >= E
    ref = P.run_gpu(g, cam)
    assert np.array_equal(ref["point_list"], P.u32(R.point_list[:E]))


def test_bin_async_matches_rs_bin_and_reports_overflow():
    """rs_bin_async (no host wait) gives rs_bin's outputs and reports (E, 0) in pinned memory; on
    overflow it writes no entry, leaves every range empty (the frame renders the background) and
    reports the count, and the redone frame matches."""
    g = scenes.procedural_scene(seed=1, n_sphere=20_000, n_helix=5_000, n_plane=5_000)
    cam = scenes.procedural_camera(320, 240)
    ref = P.run_gpu(g, cam)
    dg = rs.DeviceGaussians.from_numpy(g)
    res = torch.full((2,), -1, dtype=torch.int64).pin_memory()
    R = pipeline.Renderer(cam, g.n, capacity=ref["n_entries"] + 10)
    R.forward_async(dg, res)
    torch.cuda.synchronize()
    assert R.check_async(res) == ref["n_entries"] and int(res[1]) == 0
    E = ref["n_entries"]
    assert np.array_equal(P.u32(R.point_list[:E]), ref["point_list"])
    assert np.array_equal(R.keys_sorted[:E].cpu().numpy().view(np.uint64), ref["keys"])
    assert np.array_equal(P.u32(R.tile_ranges), ref["ranges"])
    assert np.array_equal(R.image.cpu().numpy(), ref["image"])
    # overflow: nothing written, ranges empty, background image, count reported
    small = pipeline.Renderer(cam, g.n, capacity=E // 2)
    small.point_list.fill_(-7)
    small.forward_async(dg, res, bg=(0.25, 0.5, 0.75))
    torch.cuda.synchronize()
    assert int(res[0]) == E
    assert not small.tile_ranges.any()
    assert (small.point_list == -7).all()
    img = small.image.cpu().numpy()
    assert np.allclose(img[0], 0.25) and np.allclose(img[1], 0.5) and np.allclose(img[2], 0.75)
    with pytest.raises(rs.RsError) as e:
        small.check_async(res)
    assert e.value.code == rs.RS_ERR_CAPACITY and small.capacity >= E
    small.forward_async(dg, res)
    torch.cuda.synchronize()
    assert small.check_async(res) == E
    assert np.array_equal(P.u32(small.point_list[:E]), ref["point_list"])


def test_forward_is_deterministic():
    g = scenes.procedural_scene(seed=3, n_sphere=20_000, n_helix=5_000, n_plane=5_000)
    cam = scenes.procedural_camera(320, 240)
    a = P.run_gpu(g, cam)
    b = P.run_gpu(g, cam)
    for k in ("means2d", "conic", "color", "keys", "point_list", "ranges", "image", "final_T", "n_contrib"):
        assert np.array_equal(a[k], b[k]), k


def pair_codes(idx, tile):
    return (np.asarray(idx, np.uint64) << np.uint64(32)) | np.asarray(tile, np.uint64)


def check_ellipse_binning(cam, g, sq, el):
    """The GPU's ellipse binning against the oracle's, which states the test from its definition
    in double precision: keys, point lists and counts equal on every (Gaussian, tile) decision
    that is not a knife edge (at knife edges either outcome is correct, and those pairs are left
    out of the comparison on both sides).  The oracle reads the square test's projection (the
    radius square and the values of every Gaussian, including those the GPU's ellipse test culled)
    and the GPU's k where the GPU kept the Gaussian (else k from its definition, in float32)."""
    o = g.opacity.astype(np.float64)
    k_def = np.where(255 * o > 1, 2.002 * np.log(np.maximum(255 * o, 1.0)), 0.0).astype(np.float32)
    k = np.where(el["radius"] > 0, el["alpha_k"], k_def).astype(np.float32)
    Be = oracle.bin_ellipse(cam, sq["means2d"], sq["depth"], sq["radius"], sq["conic"], k)
    amb = pair_codes(Be["ambiguous"][:, 0], Be["ambiguous"][:, 1])
    gpu_pairs = pair_codes(el["point_list"], el["keys"] >> np.uint64(32))
    orc_pairs = pair_codes(Be["point_list"], Be["keys_sorted"] >> np.uint64(32))
    keep_g, keep_o = ~np.isin(gpu_pairs, amb), ~np.isin(orc_pairs, amb)
    assert np.array_equal(el["keys"][keep_g], Be["keys_sorted"][keep_o])
    assert np.array_equal(el["point_list"][keep_g], Be["point_list"][keep_o])
    clear = ~Be["ambiguous_gaussian"]
    assert np.array_equal(el["tiles_touched"][clear], Be["tiles_touched"][clear])
    assert np.array_equal(el["radius"][clear] > 0, Be["tiles_touched"][clear] > 0)
    # the GPU's ranges are those of its own sorted keys
    assert np.array_equal(el["ranges"].reshape(-1, 2), oracle.tile_ranges(el["keys"], cam.n_tiles))
    if amb.size == 0:
        assert np.array_equal(el["ranges"].reshape(-1, 2), Be["ranges"])
    assert amb.size <= 0.01 * max(1, Be["n_entries"])
    return Be


@pytest.mark.parametrize("which", ["tiny", "160k_1080p"])
def test_ellipse_tile_test(which):
    """RS_TILE_TEST_ELLIPSE: binning equal to the oracle's ellipse binning on the same projected
    data, decision by decision off knife edges; the image and final_T bit-identical to the square
    test's (the dropped tiles hold only alpha < 1/255); gradients equal to the square test's up to
    summation order; fewer entries; n_contrib never larger."""
    if which == "tiny":
        g, cam = scenes.tiny_scene(seed=0)
    else:
        g = scenes.procedural_scene(seed=0)
        cam = scenes.orbit_cameras(1920, 1080)[10]
    dg = rs.DeviceGaussians.from_numpy(g)
    dL = torch.from_numpy(scenes.image_grad(cam)).cuda()
    out = {}
    for mode in (rs.RS_TILE_TEST_SQUARE, rs.RS_TILE_TEST_ELLIPSE):
        R = pipeline.Renderer(cam, g.n, tile_test=mode)
        F = R.forward(dg)
        B = R.backward(dg, dL)
        torch.cuda.synchronize()
        st = P.gpu_state(R, dg, F)
        st.update({k: getattr(B, k).cpu().numpy() for k in ("dmeans2d", "dconic", "dopacity", "dcolor",
                                                            "dmeans", "dscales", "dquats")})
        if mode == rs.RS_TILE_TEST_ELLIPSE:
            st["alpha_k"] = R.proj.alpha_k.cpu().numpy()
        out[mode] = st
    sq, el = out[rs.RS_TILE_TEST_SQUARE], out[rs.RS_TILE_TEST_ELLIPSE]
    check_ellipse_binning(cam, g, sq, el)
    assert el["n_entries"] < sq["n_entries"]
    # projection: the ellipse test only culls; k = 2.002 ln(255 o)
    vis = el["radius"] > 0
    assert not (vis & (sq["radius"] == 0)).any()
    for k in ("means2d", "depth", "conic", "color"):
        assert np.array_equal(el[k][..., vis], sq[k][..., vis])
    o = g.opacity.astype(np.float64)[vis]
    P.allclose_report("alpha_k", el["alpha_k"][vis], 2.002 * np.log(255 * o), 1e-6, 1e-6)
    # the same transmittance, the same colour up to the rounding of its sums (a tile whose list
    # crosses 256-entry chunk boundaries sums its colour per stretch between them, and the
    # stretches fall at other entries when the lists differ), and gradients up to summation order
    assert np.array_equal(el["final_T"], sq["final_T"])
    P.allclose_report("image", el["image"], sq["image"], 1e-6, 1e-6)
    assert (el["n_contrib"] <= sq["n_contrib"]).all()
    # both are float32 sums over tiles in no fixed order; where those sums cancel, their rounding
    # scales with the terms, not the result, so the absolute part is 1e-5 of the largest gradient
    for k in ("dmeans2d", "dconic", "dopacity", "dcolor", "dmeans", "dscales", "dquats"):
        P.allclose_report(k, el[k], sq[k], P.GRAD_RTOL, P.GRAD_ATOL, atol_of_max=1e-5)


@pytest.mark.parametrize("degree", [-1, 3])
def test_staged_and_vectorised_projections_equal_the_scalar_one(degree):
    """rs_project has three paths with the same per-Gaussian arithmetic: input rows staged in
    shared memory by bulk copies (n a multiple of 4, rows 16-byte aligned), two Gaussians per
    thread with 8-byte loads (n even), one per thread otherwise.  The first 4000 Gaussians of an
    n = 4001 scene (scalar) and of an n = 4002 scene (vectorised) project bit for bit as the
    n = 4000 scene (staged, with a ragged last tile of 32 Gaussians)."""
    g = scenes.procedural_scene(seed=8, n_sphere=2500, n_helix=750, n_plane=751)
    if degree == -1:
        g.colors = np.ascontiguousarray(np.random.default_rng(1).uniform(0, 1, (3, g.n)), np.float32)
        g.sh, g.sh_degree = None, -1
    assert g.n == 4001

    def first(m, extra=0):
        idx = np.r_[np.arange(m), np.full(extra, m - 1)]
        pick = lambda a: None if a is None else np.ascontiguousarray(a[..., idx])
        return scenes.Gaussians(pick(g.means), pick(g.scales), pick(g.quats), pick(g.opacity), pick(g.sh),
                                g.sh_degree, pick(g.colors))

    cam = scenes.procedural_camera(320, 240, azimuth=0.9)
    runs = {"scalar": P.run_gpu(g, cam), "vectorised": P.run_gpu(first(4001, 1), cam),
            "staged": P.run_gpu(first(4000), cam)}
    b = runs["staged"]
    rb = b["renderer"].proj.records.cpu().numpy().view(np.float32).reshape(-1, 12)
    vis = b["radius"] > 0
    for name in ("scalar", "vectorised"):
        a = runs[name]
        for k in ("means2d", "depth", "conic", "color"):
            assert np.array_equal(a[k][..., :4000], b[k]), (name, k)
        assert np.array_equal(a["radius"][:4000], b["radius"]), name
        assert np.array_equal(a["tiles_touched"][:4000], b["tiles_touched"]), name
        ra = a["renderer"].proj.records.cpu().numpy().view(np.float32).reshape(-1, 12)[:4000]
        assert np.array_equal(ra[vis], rb[vis]), name
