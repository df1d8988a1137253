"""rs_bin_noalloc -- binning for callers that cannot give the library device memory (a plug-in
whose host application owns every device allocation, or a frame loop that may not call cudaMalloc
because it synchronises the device).  The call uses the library's fixed scratch array instead of a
workspace; its outputs must equal rs_bin's bit for bit (binning is integer work), on two calls in a
row, since the array keeps the previous call's contents.

This file is collected last so that a run stopping at the first failure has run every other test;
it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

from gaussian_splatting_tile_gb300 import build_lib, pipeline, rs, scenes

pytestmark = pytest.mark.gpu


def _bin_both(g, cam, capacity):
    dg = rs.DeviceGaussians.from_numpy(g)
    R = pipeline.Renderer(cam, g.n, capacity=capacity)
    R.project(dg)
    E_ref = R.bin()
    ref = (R.keys_sorted[:E_ref].clone(), R.point_list[:E_ref].clone(), R.tile_ranges.clone())
    keys = torch.full((capacity,), -1, dtype=torch.int64, device="cuda")
    plist = torch.full((capacity,), -1, dtype=torch.int32, device="cuda")
    ranges = torch.full_like(R.tile_ranges, -1)
    E = rs.rs_bin_noalloc(cam, R.proj, g.n, capacity, keys, plist, ranges)
    torch.cuda.synchronize()
    return E_ref, ref, E, (keys[:E], plist[:E], ranges)


def test_noalloc_matches_rs_bin_on_two_calls_in_a_row():
    build_lib.build()
    assert torch.cuda.is_available()
    tiny = scenes.tiny_scene(seed=0)
    cases = [tiny,
             (scenes.procedural_scene(seed=1, n_sphere=40_000, n_helix=10_000, n_plane=10_000),
              scenes.procedural_camera(640, 480, azimuth=0.7)),
             tiny]
    # calls in a row on one shared array: small, larger, then small again over the larger call's
    # leftovers
    for g, cam in cases:
        E_ref, ref, E, got = _bin_both(g, cam, capacity=1_000_000)
        assert E == E_ref > 0
        for a, b in zip(ref, got):
            assert torch.equal(a, b)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # the size check comes first: nothing is read or written when it fails
    build_lib.build()
    g, cam = scenes.tiny_scene(seed=0)
    R = pipeline.Renderer(cam, g.n, capacity=4096)
    R.project(rs.DeviceGaussians.from_numpy(g))
    R.keys_sorted.fill_(-3)
    R.point_list.fill_(-5)
    R.tile_ranges.fill_(-7)
    torch.cuda.synchronize()
    too_many = 8_000_000  # about 160 MB of sort buffers, beyond the 48 MiB array
    import ctypes
    c = rs.camera_struct(cam)
    p = R.proj.struct()
    E = ctypes.c_size_t(12345)
    rc = rs.lib().rs_bin_noalloc(ctypes.byref(c), ctypes.byref(p), g.n, too_many,
                                 ctypes.c_void_p(R.keys_sorted.data_ptr()),
                                 ctypes.c_void_p(R.point_list.data_ptr()),
                                 ctypes.c_void_p(R.tile_ranges.data_ptr()), ctypes.byref(E), None)
    torch.cuda.synchronize()
    assert rc == rs.RS_ERR_WORKSPACE
    assert E.value == 12345
    assert (R.keys_sorted == -3).all() and (R.point_list == -5).all() and (R.tile_ranges == -7).all()
