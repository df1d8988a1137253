"""Pins for the oracle's binning (c2): the worked examples printed on the viewer page
(4.1 Prefix Scan, 4.4 Tile Range), the three CPU claims of the learn-gs notebook "11 - Tiles",
and a brute-force stable sort written with Python's own (stable) sort.  CPU only."""
import os
import struct

import numpy as np
import pytest

from gaussian_splatting_tile_gb300 import scenes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "viewer_worked_examples.txt")


def golden_rows(kind):
    rows = []
    for line in open(GOLDEN, encoding="utf-8"):
        if not line.strip() or line.startswith("#"):
            continue
        name, section, inp, out = [s.strip() for s in line.split("|")]
        if name == kind:
            rows.append((section, inp, out))
    assert rows
    return rows


def test_viewer_scan_examples(orc):
    for section, inp, out in golden_rows("exclusive_scan"):
        vals = [int(x) for x in inp.split()]
        got, total = orc.exclusive_scan(vals)
        assert list(got) == [int(x) for x in out.split()], section
        assert total == sum(vals)


def test_viewer_tile_range_examples(orc):
    for section, inp, out in golden_rows("tile_ranges"):
        tiles = [int(x) for x in inp.split()]
        keys = np.array([(t << 32) | 0x3F800000 for t in tiles], np.uint64)
        exp = [tuple(int(v) for v in p.split(":")) for p in out.split()]
        got = orc.tile_ranges(keys, len(exp))
        assert [tuple(r) for r in got] == exp, section


def test_claim1_float_bits_sort_like_floats():
    # learn-gs "11 - Tiles", claim 1: positive float32 bit patterns are monotone in the value.
    rng = np.random.default_rng(11)
    d = (rng.random(20000) * 50 + 0.05).astype(np.float32)
    order = np.argsort(d.view(np.uint32), kind="stable")
    assert np.all(np.diff(d[order]) >= 0)


def brute_force_bin(cam, means2d, depth, radius):
    TX, TY = cam.tiles_x, cam.tiles_y
    entries = []
    for i in range(radius.shape[0]):
        if radius[i] <= 0:
            continue
        u, v, r = np.float32(means2d[0, i]), np.float32(means2d[1, i]), np.float32(radius[i])
        for ty in range(TY):
            for tx in range(TX):
                # the tile's square overlaps the splat's bounding square (claim 2's test)
                if (np.float32(tx * 16) <= u + r and np.float32((tx + 1) * 16) > u - r and
                        np.float32(ty * 16) <= v + r and np.float32((ty + 1) * 16) > v - r):
                    bits = struct.unpack("<I", struct.pack("<f", float(depth[i])))[0]
                    entries.append((((ty * TX + tx) << 32) | bits, i))
    entries = sorted(entries, key=lambda e: e[0])  # Python's sort is stable
    return [e[0] for e in entries], [e[1] for e in entries]


def test_matches_brute_force_stable_sort(orc):
    rng = np.random.default_rng(7)
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 60.0, 60.0, 70, 50)  # ragged tiles on both axes
    n = 300
    means2d = np.stack([rng.uniform(-20, 90, n), rng.uniform(-20, 70, n)]).astype(np.float32)
    # quantised depths force many exact key ties, which only a stable sort orders by index
    depth = rng.choice(np.array([0.5, 1.0, 1.5, 2.0], np.float32), n)
    radius = rng.integers(0, 25, n).astype(np.int32)
    B = orc.bin(cam, means2d, depth, radius)
    keys, vals = brute_force_bin(cam, means2d, depth, radius)
    assert B["n_entries"] == len(keys)
    assert list(B["keys_sorted"]) == keys
    assert list(B["point_list"]) == vals
    # ranges against a direct scan of the brute-force keys
    for t in range(cam.n_tiles):
        idx = [e for e, k in enumerate(keys) if (k >> 32) == t]
        exp = (idx[0], idx[-1] + 1) if idx else (0, 0)
        assert tuple(B["ranges"][t]) == exp


def test_claim3_ranges_partition_and_depth_order(orc):
    # learn-gs "11 - Tiles", claim 3 on a rendered scene.
    g = scenes.procedural_scene(seed=0, n_sphere=3000, n_helix=800, n_plane=800)
    cam = scenes.procedural_camera(256, 256)
    P = orc.project(cam, g, prec=32)
    B = orc.bin(cam, P["means2d"].astype(np.float32), P["depth"].astype(np.float32), P["radius"])
    r = B["ranges"].astype(np.int64)
    lens = r[:, 1] - r[:, 0]
    assert lens.sum() == B["n_entries"] == int(P["tiles_touched"].sum())
    nz = r[lens > 0]
    assert np.all(nz[1:, 0] == nz[:-1, 1]) and nz[0, 0] == 0 and nz[-1, 1] == B["n_entries"]
    tiles = (B["keys_sorted"] >> np.uint64(32)).astype(np.int64)
    depth = P["depth"].astype(np.float32)
    for t in np.nonzero(lens)[0]:
        s, e = r[t]
        assert np.all(tiles[s:e] == t)
        d = depth[B["point_list"][s:e]]
        assert np.all(np.diff(d) >= 0)
    assert np.array_equal(B["tiles_touched"], P["tiles_touched"])


def test_empty_and_all_culled(orc):
    cam = scenes.look_at([0, 0, 3], [0, 0, 0], 60.0, 60.0, 40, 40)
    B = orc.bin(cam, np.zeros((2, 0), np.float32), np.zeros(0, np.float32), np.zeros(0, np.int32))
    assert B["n_entries"] == 0 and not B["ranges"].any()
    B = orc.bin(cam, np.ones((2, 5), np.float32), np.ones(5, np.float32), np.zeros(5, np.int32))
    assert B["n_entries"] == 0 and not B["ranges"].any()
