"""The C-ABI library loads and exports every entry point include/rs.h declares; host-only calls
and argument validation behave as documented.  No GPU work is issued (CPU only)."""
import ctypes

import pytest

from gaussian_splatting_tile_gb300 import build_lib, rs, scenes


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return rs.lib()


def test_exports_every_declared_symbol(L):
    names = rs.declared_symbols()
    assert {"rs_project", "rs_bin", "rs_rasterize_fwd", "rs_rasterize_bwd", "rs_project_bwd",
            "rs_bin_workspace_size", "rs_error_string"} <= set(names)
    for name in names:
        assert hasattr(L, name), name


def test_header_constants_match_the_binding():
    """Every #define of include/rs.h that the binding mirrors has the same value there."""
    import pathlib
    import re
    text = (pathlib.Path(__file__).resolve().parents[1] / "include" / "rs.h").read_text()
    defs = {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define (RS_\w+) \(?(-?\d+)\)?", text, re.M)}
    mirrored = [k for k in defs if hasattr(rs, k)]
    assert {"RS_OK", "RS_ERR_CAPACITY", "RS_TILE_TEST_SQUARE", "RS_TILE_TEST_ELLIPSE", "RS_ELLIPSE_WORDS",
            "RS_ACT_EXP", "RS_ADAM_MAX_SEGMENTS"} <= set(mirrored)
    for k in mirrored:
        assert getattr(rs, k) == defs[k], k


def test_error_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, 7):
        assert rs.error_string(code)
    assert "capacity" in rs.error_string(rs.RS_ERR_CAPACITY)
    assert "out of range" in rs.error_string(rs.RS_ERR_DEVICE_CHECK)
    assert rs.error_string(rs.RS_ERR_DEVICE_CHECK) != rs.error_string(7)


def test_workspace_size_grows_with_capacity(L):
    cam = scenes.procedural_camera(1920, 1080)
    a = rs.rs_bin_workspace_size(160_000, cam, 1_000_000)
    b = rs.rs_bin_workspace_size(160_000, cam, 4_000_000)
    assert 0 < a < b
    # two 4-byte tile-key buffers and one 4-byte value buffer per entry at least
    assert b - a >= 3_000_000 * 12
    assert rs.rs_bin_workspace_size(0, cam, 0) > 0


def test_invalid_arguments_rejected_before_any_launch(L):
    cam = rs.camera_struct(scenes.procedural_camera(64, 48))
    nbytes = ctypes.c_size_t(0)
    assert L.rs_bin_workspace_size(-1, ctypes.byref(cam), 10, ctypes.byref(nbytes)) == rs.RS_ERR_INVALID_ARG
    assert L.rs_bin_workspace_size(10, None, 10, ctypes.byref(nbytes)) == rs.RS_ERR_INVALID_ARG
    assert L.rs_bin_workspace_size(10, ctypes.byref(cam), 10, None) == rs.RS_ERR_INVALID_ARG
    bad = rs.camera_struct(scenes.procedural_camera(64, 48))
    bad.fx = 0.0
    assert L.rs_bin_workspace_size(10, ctypes.byref(bad), 10, ctypes.byref(nbytes)) == rs.RS_ERR_INVALID_ARG
    bad = rs.camera_struct(scenes.procedural_camera(64, 48))
    bad.width = 0
    assert L.rs_bin_workspace_size(10, ctypes.byref(bad), 10, ctypes.byref(nbytes)) == rs.RS_ERR_INVALID_ARG
    # null pointers / bad degree are caught by validation, which runs before any CUDA call
    g = rs.rs_gaussians()
    g.n = 10
    g.sh_degree = 0
    assert L.rs_project(ctypes.byref(cam), ctypes.byref(g), None, None) == rs.RS_ERR_INVALID_ARG
    g.sh_degree = 4
    assert L.rs_project(ctypes.byref(cam), ctypes.byref(g), None, None) == rs.RS_ERR_INVALID_ARG
    g.n = -3
    g.sh_degree = 0
    assert L.rs_project(ctypes.byref(cam), ctypes.byref(g), None, None) == rs.RS_ERR_INVALID_ARG
    bgv = (ctypes.c_float * 3)(0, 0, 0)
    assert L.rs_rasterize_fwd(ctypes.byref(cam), None, 5, None, None, 0, bgv, None, None, None, None, 0,
                              None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_rasterize_bwd(ctypes.byref(cam), None, 5, None, None, 0, bgv, None, None, None, 0, None,
                              None, None, None, None, None) == rs.RS_ERR_INVALID_ARG
    E = ctypes.c_size_t(0)
    assert L.rs_bin(ctypes.byref(cam), None, 5, None, 0, 0, None, None, None, ctypes.byref(E), None) == rs.RS_ERR_INVALID_ARG
    # misaligned workspace
    assert L.rs_bin(ctypes.byref(cam), None, 0, ctypes.c_void_p(0x1001), 1 << 20, 0, None, None,
                    ctypes.c_void_p(0x2000), ctypes.byref(E), None) == rs.RS_ERR_INVALID_ARG
    # workspace too small (validated on the host, before launches)
    assert L.rs_bin(ctypes.byref(cam), None, 0, ctypes.c_void_p(0x1000), 16, 0, None, None,
                    ctypes.c_void_p(0x2000), ctypes.byref(E), None) == rs.RS_ERR_WORKSPACE


def test_raster_workspace_validation(L):
    """The compositing workspace: one 256-pixel float4 state and one tile index per 256 entries
    of capacity (plus one); too small or misaligned is refused before any launch."""
    camera = scenes.procedural_camera(64, 48)
    cam = rs.camera_struct(camera)
    chunk = rs.RS_RASTER_CHUNK
    for cap in (0, 1, 255, 256, 4_000_000):
        slots = cap // chunk + 1
        assert rs.rs_raster_workspace_size(camera, cap) >= slots * (chunk * 16 + 4) + 4 * 12
    assert rs.rs_raster_workspace_size(camera, 1_000_000) < rs.rs_raster_workspace_size(camera, 4_000_000)
    # sizes past 2^31 bytes come back whole (the binding takes the header's size_t return type)
    assert L.rs_raster_workspace_size.restype is ctypes.c_size_t
    assert rs.rs_raster_workspace_size(camera, rs.RS_MAX_ENTRIES) >= (rs.RS_MAX_ENTRIES // chunk) * chunk * 16 > 2**31
    big = scenes.procedural_camera(1920, 1080)
    assert rs.rs_raster_workspace_size(big, 1000) >= rs.rs_raster_workspace_size(camera, 1000) + 4 * (8160 - 12) - 256
    assert L.rs_raster_workspace_size(ctypes.byref(cam), rs.RS_MAX_ENTRIES + 1) == 0
    assert L.rs_raster_workspace_size(None, 10) == 0
    p = rs.rs_projected()
    p.d_records = 0x1000
    bgv = (ctypes.c_float * 3)(0, 0, 0)
    fake = lambda a: ctypes.c_void_p(a)
    cap = 10_000
    need = rs.rs_raster_workspace_size(camera, cap)
    fwd = lambda ws, nb, c=cap: L.rs_rasterize_fwd(ctypes.byref(cam), ctypes.byref(p), 5, fake(0x2000), fake(0x3000),
                                                    c, bgv, fake(0x4000), fake(0x5000), fake(0x6000), ws, nb, None)
    bwd = lambda ws, nb, c=cap: L.rs_rasterize_bwd(ctypes.byref(cam), ctypes.byref(p), 5, fake(0x2000),
                                                    fake(0x3000), c, bgv, fake(0x5000), fake(0x6000),
                                                    ws, nb, fake(0x7000), fake(0x8000), fake(0x9000),
                                                    fake(0xa000), fake(0xb000), None)
    for call in (fwd, bwd):
        assert call(fake(0xc000), need - 1) == rs.RS_ERR_WORKSPACE
        assert call(fake(0xc008), need) == rs.RS_ERR_INVALID_ARG
        assert call(None, need) == rs.RS_ERR_INVALID_ARG
        assert call(fake(0xc000), need, rs.RS_MAX_ENTRIES + 1) == rs.RS_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(L):
    import torch
    cam = scenes.procedural_camera(64, 48)
    g = rs.DeviceGaussians(torch.zeros(3, 4), torch.zeros(3, 4), torch.zeros(4, 4), torch.zeros(4),
                           torch.zeros(3, 4), 0)
    with pytest.raises(TypeError):
        g.struct()


def test_appearance_and_loss_validation(L):
    cam = rs.camera_struct(scenes.procedural_camera(64, 48))
    m = rs.rs_mlp()
    m.latent_dim, m.hidden = 8, 64
    m.d_W1 = m.d_b1 = m.d_W2 = m.d_b2 = ctypes.c_void_p(0x1000)
    ok = ctypes.c_void_p(0x2000)
    # unsupported widths and null weights are refused before any launch
    for latent, hidden in ((8, 48), (0, 64), (30, 64), (8, 128)):
        m.latent_dim, m.hidden = latent, hidden
        assert L.rs_appearance_fwd(ctypes.byref(cam), 10, ok, ok, ctypes.byref(m), ok, None) == rs.RS_ERR_INVALID_ARG
    m.latent_dim, m.hidden = 8, 64
    m.d_W2 = None
    assert L.rs_appearance_fwd(ctypes.byref(cam), 10, ok, ok, ctypes.byref(m), ok, None) == rs.RS_ERR_INVALID_ARG
    m.d_W2 = ctypes.c_void_p(0x1000)
    assert L.rs_appearance_fwd(ctypes.byref(cam), 10, None, ok, ctypes.byref(m), ok, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_appearance_fwd(ctypes.byref(cam), -1, ok, ok, ctypes.byref(m), ok, None) == rs.RS_ERR_INVALID_ARG
    # n = 0 needs no buffers and launches nothing
    assert L.rs_appearance_fwd(ctypes.byref(cam), 0, None, None, ctypes.byref(m), None, None) == rs.RS_OK
    assert L.rs_appearance_bwd(ctypes.byref(cam), 10, ok, ok, ctypes.byref(m), ok, ok, None, None) == rs.RS_ERR_INVALID_ARG
    gr = rs.rs_mlp_grads()
    gr.d_dW1 = gr.d_db1 = gr.d_dW2 = ok
    assert L.rs_appearance_bwd(ctypes.byref(cam), 10, ok, ok, ctypes.byref(m), ok, ok, ctypes.byref(gr),
                               None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_l1_loss_grad(10, ok, ok, ctypes.c_float(float("nan")), ok, None, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_l1_loss_grad(10, None, ok, ctypes.c_float(1.0), ok, None, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_l1_loss_grad(10, ok, ok, ctypes.c_float(1.0), ok, ctypes.c_void_p(0x2001), None) == rs.RS_ERR_INVALID_ARG


def test_bin_async_validation(L):
    cam = rs.camera_struct(scenes.procedural_camera(64, 48))
    ok = ctypes.c_void_p(0x2000)
    ws = ctypes.c_void_p(0x1000)
    # the pinned result pointer is required and must be 8-byte aligned; checked before any launch
    assert L.rs_bin_async(ctypes.byref(cam), None, 0, ws, 1 << 20, 0, None, None, ok, None, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_bin_async(ctypes.byref(cam), None, 0, ws, 1 << 20, 0, None, None, ok,
                          ctypes.c_void_p(0x3004), None) == rs.RS_ERR_INVALID_ARG
    # the workspace size is validated on the host as for rs_bin
    assert L.rs_bin_async(ctypes.byref(cam), None, 0, ws, 16, 0, None, None, ok, ctypes.c_void_p(0x3008),
                          None) == rs.RS_ERR_WORKSPACE


def test_adam_and_densify_validation(L):
    ok = ctypes.c_void_p(0x2000)
    seg = (rs.rs_adam_segment * 2)()
    for s in seg:
        s.d_param = s.d_grad = s.d_m = s.d_v = ok
        s.count, s.lr, s.activation = 10, 0.01, 0
    f = ctypes.c_double
    assert L.rs_adam_step(seg, 2, f(0.9), f(0.999), f(1e-15), 0, None) == rs.RS_ERR_INVALID_ARG  # step < 1
    assert L.rs_adam_step(seg, 2, f(1.0), f(0.999), f(1e-15), 1, None) == rs.RS_ERR_INVALID_ARG  # beta1 = 1
    assert L.rs_adam_step(seg, 2, f(0.9), f(0.999), f(0.0), 1, None) == rs.RS_ERR_INVALID_ARG    # eps = 0
    assert L.rs_adam_step(seg, 17, f(0.9), f(0.999), f(1e-15), 1, None) == rs.RS_ERR_INVALID_ARG
    seg[1].activation = 3
    assert L.rs_adam_step(seg, 2, f(0.9), f(0.999), f(1e-15), 1, None) == rs.RS_ERR_INVALID_ARG
    seg[1].activation = 1
    seg[1].d_v = None
    assert L.rs_adam_step(seg, 2, f(0.9), f(0.999), f(1e-15), 1, None) == rs.RS_ERR_INVALID_ARG
    seg[1].count = 0  # empty groups need no buffers
    seg[0].count = 0
    assert L.rs_adam_step(seg, 2, f(0.9), f(0.999), f(1e-15), 1, None) == rs.RS_OK
    assert L.rs_densify_stats(-1, ok, ok, ok, ok, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_densify_stats(5, None, ok, ok, ok, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_densify_stats(0, None, None, None, None, None) == rs.RS_OK


def test_l1_dssim_validation(L):
    ok = ctypes.c_void_p(0x2000)
    b = ctypes.c_size_t(0)
    assert L.rs_l1_dssim_workspace_size(0, 4, 4, ctypes.byref(b)) == rs.RS_ERR_INVALID_ARG
    assert L.rs_l1_dssim_workspace_size(3, 4, 4, ctypes.byref(b)) == rs.RS_OK and b.value >= 3 * 3 * 16 * 4
    f = ctypes.c_float
    assert L.rs_l1_dssim_loss_grad(3, 4, 4, ok, ok, f(1.5), f(1.0), ok, None, ok, b.value, None) == rs.RS_ERR_INVALID_ARG
    assert L.rs_l1_dssim_loss_grad(3, 4, 4, ok, ok, f(0.2), f(1.0), ok, None, ok, 8, None) == rs.RS_ERR_WORKSPACE
    assert L.rs_l1_dssim_loss_grad(3, 4, 4, ok, None, f(0.2), f(1.0), ok, None, ok, b.value, None) == rs.RS_ERR_INVALID_ARG
