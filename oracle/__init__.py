"""CPU oracle for tile-based Gaussian splatting -- TEST INFRASTRUCTURE ONLY.

Thin ctypes loader over `liboracle.so`, the plain single-threaded C++ statement of the
method in `oracle.cpp`.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the CUDA library never does, and this package
never touches the CUDA library.  All arrays are numpy; inputs are passed as float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_HDR = os.path.join(_HERE, "oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

AMB_NEAR, AMB_DET, AMB_RADIUS, AMB_SPAN, AMB_CLAMP = 1, 2, 4, 8, 16
AMB_ALPHA_MIN, AMB_T_STOP, AMB_ALPHA_MAX = 1, 2, 4


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (no fast-math, no FMA contraction) if it is missing or stale."""
    stale = (not os.path.exists(_SO) or
             os.path.getmtime(_SO) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               "-Wall", "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


class CCamera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_double * 9), ("t", ctypes.c_double * 3),
                ("fx", ctypes.c_double), ("fy", ctypes.c_double),
                ("cx", ctypes.c_double), ("cy", ctypes.c_double),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32)]


def _cam(cam) -> CCamera:
    c = CCamera()
    R = np.asarray(cam.R, np.float64).reshape(9)
    t = np.asarray(cam.t, np.float64).reshape(3)
    for i in range(9):
        c.R[i] = float(R[i])
    for i in range(3):
        c.t[i] = float(t[i])
    c.fx, c.fy, c.cx, c.cy = float(cam.fx), float(cam.fy), float(cam.cx), float(cam.cy)
    c.width, c.height = int(cam.width), int(cam.height)
    return c


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_SO)
        _lib.orc_exclusive_scan_u32.restype = ctypes.c_uint64
        _lib.orc_bin_count.restype = ctypes.c_int64
        _lib.orc_bin.restype = ctypes.c_int64
        _lib.orc_bin_ellipse.restype = ctypes.c_int64
        _lib.orc_ellipse_tiles.restype = ctypes.c_int32
        _lib.orc_densify_group.restype = ctypes.c_int32
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _d(a):
    return None if a is None else np.ascontiguousarray(a, np.float64)


def project(cam, g, prec: int = 64, margin: float = 0.0):
    """c1 + c6.  Returns dict of means2d [2,N], depth, conic [3,N], color [3,N], radius (int32),
    rect [4,N] (x_lo, x_hi, y_lo, y_hi), tiles_touched (uint32), ambig (uint8)."""
    n = g.n
    out = dict(means2d=np.zeros((2, n)), depth=np.zeros(n), conic=np.zeros((3, n)),
               color=np.zeros((3, n)), radius=np.zeros(n, np.int32), rect=np.zeros((4, n), np.int32),
               tiles_touched=np.zeros(n, np.uint32), ambig=np.zeros(n, np.uint8))
    c = _cam(cam)
    ins = [_d(g.means), _d(g.scales), _d(g.quats), _d(g.opacity), _d(g.sh), _d(g.colors)]
    rc = lib().orc_project(ctypes.c_int(prec), ctypes.byref(c), ctypes.c_int32(n),
                           _p(ins[0]), _p(ins[1]), _p(ins[2]), _p(ins[3]), _p(ins[4]),
                           ctypes.c_int32(g.sh_degree), _p(ins[5]),
                           _p(out["means2d"]), _p(out["depth"]), _p(out["conic"]), _p(out["color"]),
                           _p(out["radius"]), _p(out["rect"]), _p(out["tiles_touched"]),
                           ctypes.c_double(margin), _p(out["ambig"]))
    if rc != 0:
        raise ValueError(f"orc_project returned {rc}")
    return out


def project_intermediates(cam, g):
    n = g.n
    cov3d, cov2d = np.zeros((6, n)), np.zeros((3, n))
    jac, pcam = np.zeros((6, n)), np.zeros((3, n))
    c = _cam(cam)
    m, s, q = _d(g.means), _d(g.scales), _d(g.quats)
    lib().orc_project_intermediates(ctypes.byref(c), ctypes.c_int32(n), _p(m), _p(s), _p(q),
                                    _p(cov3d), _p(cov2d), _p(jac), _p(pcam))
    return dict(cov3d=cov3d, cov2d=cov2d, jac=jac, pcam=pcam)


def sh_basis(dirs):
    dirs = _d(dirs)
    m = dirs.shape[1]
    Y = np.zeros((16, m))
    lib().orc_sh_basis(_p(dirs), ctypes.c_int32(m), _p(Y))
    return Y


def exclusive_scan(values):
    v = np.ascontiguousarray(values, np.uint32)
    out = np.zeros(v.shape[0], np.uint64)
    total = lib().orc_exclusive_scan_u32(_p(v), ctypes.c_int64(v.shape[0]), _p(out))
    return out, int(total)


def tile_ranges(keys_sorted, n_tiles):
    k = np.ascontiguousarray(keys_sorted, np.uint64)
    r = np.zeros((n_tiles, 2), np.uint32)
    lib().orc_tile_ranges(_p(k), ctypes.c_int64(k.shape[0]), ctypes.c_int32(n_tiles), _p(r))
    return r


def bin(cam, means2d, depth, radius):
    """c2 from float32 projected data.  Returns keys_sorted (uint64), point_list (uint32),
    ranges [n_tiles,2] (uint32), tiles_touched (uint32)."""
    m2 = np.ascontiguousarray(means2d, np.float32)
    dp = np.ascontiguousarray(depth, np.float32)
    rd = np.ascontiguousarray(radius, np.int32)
    n = rd.shape[0]
    c = _cam(cam)
    E = lib().orc_bin_count(ctypes.byref(c), ctypes.c_int32(n), _p(m2), _p(rd))
    keys = np.zeros(max(E, 1), np.uint64)
    pl = np.zeros(max(E, 1), np.uint32)
    n_tiles = ((cam.width + 15) // 16) * ((cam.height + 15) // 16)
    ranges = np.zeros((n_tiles, 2), np.uint32)
    tt = np.zeros(n, np.uint32)
    E2 = lib().orc_bin(ctypes.byref(c), ctypes.c_int32(n), _p(m2), _p(dp), _p(rd),
                       ctypes.c_int64(E), _p(keys), _p(pl), _p(ranges), _p(tt))
    assert E2 == E
    return dict(keys_sorted=keys[:E], point_list=pl[:E], ranges=ranges, tiles_touched=tt,
                n_entries=int(E))


ELLIPSE_WIDEN = 0.02     # px: the square widened on every side for the "dropped for certain" test
ELLIPSE_MARGIN = 1e-5    # relative margin on k


def bin_ellipse(cam, means2d, depth, radius, conic, alpha_k, widen=ELLIPSE_WIDEN, margin=ELLIPSE_MARGIN):
    """c2' (ellipse-tile test, from its definition in double precision) from float32 projected data.
    Same outputs as bin(), plus the knife-edge decisions: `ambiguous` [M, 2] uint32 rows of
    (Gaussian index, tile id) where either outcome is correct, and `ambiguous_gaussian` [n] bool."""
    m2 = np.ascontiguousarray(means2d, np.float32)
    dp = np.ascontiguousarray(depth, np.float32)
    rd = np.ascontiguousarray(radius, np.int32)
    cn = np.ascontiguousarray(conic, np.float32)
    ak = np.ascontiguousarray(alpha_k, np.float32)
    n = rd.shape[0]
    c = _cam(cam)
    n_tiles = ((cam.width + 15) // 16) * ((cam.height + 15) // 16)
    ranges = np.zeros((n_tiles, 2), np.uint32)
    tt = np.zeros(n, np.uint32)
    ag = np.zeros(n, np.uint8)
    cap, acap = 1 << 16, 1 << 12
    na = ctypes.c_int64(0)
    while True:
        keys = np.zeros(cap, np.uint64)
        pl = np.zeros(cap, np.uint32)
        pairs = np.zeros((acap, 2), np.uint32)
        E = lib().orc_bin_ellipse(ctypes.byref(c), ctypes.c_int32(n), _p(m2), _p(dp), _p(rd), _p(cn), _p(ak),
                                  ctypes.c_double(widen), ctypes.c_double(margin), ctypes.c_int64(cap),
                                  _p(keys), _p(pl), _p(ranges), _p(tt), _p(ag), ctypes.c_int64(acap),
                                  _p(pairs), ctypes.byref(na))
        if E >= 0:
            break
        cap = max(cap, int(tt.astype(np.int64).sum()) + 1)
        acap = max(acap, na.value + 1)
    return dict(keys_sorted=keys[:E], point_list=pl[:E], ranges=ranges, tiles_touched=tt, n_entries=int(E),
                ambiguous=pairs[:na.value].copy(), ambiguous_gaussian=ag.astype(bool))


def ellipse_tiles(cam, u, v, A, B, C, k, radius, widen=ELLIPSE_WIDEN, margin=ELLIPSE_MARGIN):
    """Decisions of the ellipse-tile test over one Gaussian's radius square: (rect, codes) with
    rect = (xl, xh, yl, yh) half-open and codes [yh - yl, xh - xl] uint8, bit 0 kept, bit 1 knife edge."""
    c = _cam(cam)
    rect = np.zeros(4, np.int32)
    TX, TY = (cam.width + 15) // 16, (cam.height + 15) // 16
    codes = np.zeros(TX * TY, np.uint8)
    f = ctypes.c_float
    cnt = lib().orc_ellipse_tiles(ctypes.byref(c), f(u), f(v), f(A), f(B), f(C), f(k), ctypes.c_int32(radius),
                                  ctypes.c_double(widen), ctypes.c_double(margin), _p(rect), _p(codes),
                                  ctypes.c_int64(codes.size))
    assert cnt >= 0
    xl, xh, yl, yh = (int(x) for x in rect)
    return (xl, xh, yl, yh), codes[:cnt].reshape(yh - yl, xh - xl)


def quad_min_rect(A, B, C, x0, x1, y0, y1):
    lib().orc_quad_min_rect.restype = ctypes.c_double
    d = ctypes.c_double
    return lib().orc_quad_min_rect(d(A), d(B), d(C), d(x0), d(x1), d(y0), d(y1))


def raster_fwd(cam, means2d, conic, opacity, color, ranges, point_list, bg=(0.0, 0.0, 0.0),
               prec: int = 64, margin: float = 0.0, tile_mask=None):
    """c3.  Returns image [3,H,W], final_T [H,W], n_contrib [H,W] (uint32), ambig [H,W] (uint8),
    n_blend [H,W] (uint32, composited entries per pixel)."""
    n = int(np.asarray(opacity).shape[0])
    H, W = cam.height, cam.width
    image, final_T = np.zeros((3, H, W)), np.zeros((H, W))
    n_contrib, ambig = np.zeros((H, W), np.uint32), np.zeros((H, W), np.uint8)
    n_blend = np.zeros((H, W), np.uint32)
    c = _cam(cam)
    a = [_d(means2d), _d(conic), _d(opacity), _d(color)]
    rg = np.ascontiguousarray(ranges, np.uint32)
    pl = np.ascontiguousarray(point_list, np.uint32)
    if pl.size == 0:
        pl = np.zeros(1, np.uint32)
    b = np.asarray(bg, np.float64)
    tm = None if tile_mask is None else np.ascontiguousarray(tile_mask, np.uint8)
    rc = lib().orc_raster_fwd(ctypes.c_int(prec), ctypes.byref(c), ctypes.c_int32(n), _p(a[0]),
                              _p(a[1]), _p(a[2]), _p(a[3]), _p(rg), _p(pl), _p(b), _p(tm),
                              _p(image), _p(final_T), _p(n_contrib), ctypes.c_double(margin),
                              _p(ambig), _p(n_blend))
    if rc != 0:
        raise ValueError(f"orc_raster_fwd returned {rc}")
    return dict(image=image, final_T=final_T, n_contrib=n_contrib, ambig=ambig, n_blend=n_blend)


def raster_bwd(cam, means2d, conic, opacity, color, ranges, point_list, n_contrib, dL_dimage,
               bg=(0.0, 0.0, 0.0), tile_mask=None):
    """c4 in double.  Returns dmeans2d [2,N], dconic [3,N], dopacity [N], dcolor [3,N], and
    `abs_<name>` of the same shapes: per output, the sum of the magnitudes of the terms it adds up
    (the scale of a float computation's rounding error in that sum)."""
    n = int(np.asarray(opacity).shape[0])
    out = dict(dmeans2d=np.zeros((2, n)), dconic=np.zeros((3, n)), dopacity=np.zeros(n),
               dcolor=np.zeros((3, n)))
    absum = np.zeros((9, n))
    c = _cam(cam)
    a = [_d(means2d), _d(conic), _d(opacity), _d(color)]
    rg = np.ascontiguousarray(ranges, np.uint32)
    pl = np.ascontiguousarray(point_list, np.uint32)
    if pl.size == 0:
        pl = np.zeros(1, np.uint32)
    nc = np.ascontiguousarray(n_contrib, np.uint32)
    gi = _d(dL_dimage)
    b = np.asarray(bg, np.float64)
    tm = None if tile_mask is None else np.ascontiguousarray(tile_mask, np.uint8)
    rc = lib().orc_raster_bwd(ctypes.byref(c), ctypes.c_int32(n), _p(a[0]), _p(a[1]), _p(a[2]),
                              _p(a[3]), _p(rg), _p(pl), _p(b), _p(nc), _p(gi), _p(tm),
                              _p(out["dmeans2d"]), _p(out["dconic"]), _p(out["dopacity"]),
                              _p(out["dcolor"]), _p(absum))
    if rc != 0:
        raise ValueError(f"orc_raster_bwd returned {rc}")
    out.update(abs_dmeans2d=absum[0:2], abs_dconic=absum[2:5], abs_dopacity=absum[5], abs_dcolor=absum[6:9])
    return out


def project_bwd(cam, g, radius, dmeans2d, dconic, dcolor):
    """c5 in double.  Returns dmeans [3,N], dscales [3,N], dquats [4,N], dsh [3K,N] or None."""
    n = g.n
    K = (g.sh_degree + 1) ** 2 if g.sh_degree >= 0 else 0
    out = dict(dmeans=np.zeros((3, n)), dscales=np.zeros((3, n)), dquats=np.zeros((4, n)),
               dsh=np.zeros((3 * K, n)) if K else None)
    c = _cam(cam)
    m, s, q, sh = _d(g.means), _d(g.scales), _d(g.quats), _d(g.sh)
    rd = None if radius is None else np.ascontiguousarray(radius, np.int32)
    d2, dc, dcol = _d(dmeans2d), _d(dconic), _d(dcolor)
    rc = lib().orc_project_bwd(ctypes.byref(c), ctypes.c_int32(n), _p(m), _p(s), _p(q), _p(sh),
                               ctypes.c_int32(g.sh_degree), _p(rd), _p(d2), _p(dc), _p(dcol),
                               _p(out["dmeans"]), _p(out["dscales"]), _p(out["dquats"]),
                               _p(out["dsh"]))
    if rc != 0:
        raise ValueError(f"orc_project_bwd returned {rc}")
    return out


def appearance_fwd(cam, means, latents, W1, b1, W2, b2):
    lat = _d(latents)
    L, n = lat.shape
    H = int(np.asarray(W1).shape[0])
    colors = np.zeros((3, n))
    c = _cam(cam)
    args = [_d(means), lat, _d(W1), _d(b1), _d(W2), _d(b2)]
    rc = lib().orc_appearance_fwd(ctypes.byref(c), ctypes.c_int32(n), ctypes.c_int32(L),
                                  ctypes.c_int32(H), *[_p(a) for a in args], _p(colors))
    if rc != 0:
        raise ValueError(f"orc_appearance_fwd returned {rc}")
    return colors


def appearance_bwd(cam, means, latents, W1, b1, W2, b2, dcolors):
    lat = _d(latents)
    L, n = lat.shape
    H = int(np.asarray(W1).shape[0])
    out = dict(dlatents=np.zeros((L, n)), dW1=np.zeros((H, L + 3)), db1=np.zeros(H),
               dW2=np.zeros((3, H)), db2=np.zeros(3))
    c = _cam(cam)
    args = [_d(means), lat, _d(W1), _d(b1), _d(W2), _d(b2), _d(dcolors)]
    rc = lib().orc_appearance_bwd(ctypes.byref(c), ctypes.c_int32(n), ctypes.c_int32(L),
                                  ctypes.c_int32(H), *[_p(a) for a in args],
                                  _p(out["dlatents"]), _p(out["dW1"]), _p(out["db1"]),
                                  _p(out["dW2"]), _p(out["db2"]))
    if rc != 0:
        raise ValueError(f"orc_appearance_bwd returned {rc}")
    return out


def l1_loss_grad(image, target, scale):
    """L1 term of the training loss: (grad, loss) with grad = scale * sign(image - target) and
    loss = scale * sum |image - target|."""
    img = _d(image).reshape(-1)
    tgt = _d(target).reshape(-1)
    if img.size != tgt.size:
        raise ValueError("image and target differ in size")
    grad = np.zeros(img.size)
    loss = ctypes.c_double(0.0)
    rc = lib().orc_l1_loss_grad(ctypes.c_int64(img.size), _p(img), _p(tgt), ctypes.c_double(scale),
                                _p(grad), ctypes.byref(loss))
    if rc != 0:
        raise ValueError(f"orc_l1_loss_grad returned {rc}")
    return grad.reshape(np.shape(image)), float(loss.value)


def adam_step(param, grad, m, v, lr, activation=0, beta1=0.9, beta2=0.999, eps=1e-15, step=1):
    """One Adam step on float64 copies; returns (param, m, v, activated)."""
    p, g, mm, vv = (np.array(_d(a), copy=True).reshape(-1) for a in (param, grad, m, v))
    act = np.zeros_like(p)
    rc = lib().orc_adam_step(ctypes.c_int64(p.size), _p(p), _p(g), _p(mm), _p(vv), _p(act),
                             ctypes.c_double(lr), ctypes.c_int32(activation), ctypes.c_double(beta1),
                             ctypes.c_double(beta2), ctypes.c_double(eps), ctypes.c_int32(step))
    if rc != 0:
        raise ValueError(f"orc_adam_step returned {rc}")
    return p, mm, vv, act


def densify_stats(dmeans2d, radius, accum, count):
    d2 = _d(dmeans2d)
    n = d2.shape[1]
    a, c = np.array(_d(accum), copy=True), np.array(_d(count), copy=True)
    r = np.ascontiguousarray(radius, np.int32)
    rc = lib().orc_densify_stats(ctypes.c_int32(n), _p(d2), _p(r), _p(a), _p(c))
    if rc != 0:
        raise ValueError(f"orc_densify_stats returned {rc}")
    return a, c


def l1_dssim(image, target, lam=0.2, scale=1.0):
    """L1 + D-SSIM over [C,H,W] images: (grad [C,H,W], loss, ssim map [C,H,W])."""
    img = _d(image)
    tgt = _d(target)
    if img.ndim == 2:
        img, tgt = img[None], tgt[None]
    C, H, W = img.shape
    grad = np.zeros_like(img)
    smap = np.zeros_like(img)
    loss = ctypes.c_double(0.0)
    rc = lib().orc_l1_dssim(ctypes.c_int32(C), ctypes.c_int32(H), ctypes.c_int32(W), _p(img), _p(tgt),
                            ctypes.c_double(lam), ctypes.c_double(scale), _p(grad), ctypes.byref(loss), _p(smap))
    if rc != 0:
        raise ValueError(f"orc_l1_dssim returned {rc}")
    return grad, float(loss.value), smap


def densify_classify(accum, count, log_scales, logits, grad_threshold, dense_scale, min_opacity, max_scale=0.0):
    """c12 decisions: (action [n] int32: 0 removed, 1 kept, 2 kept and cloned, 3 split;
    ambiguous [n] bool; counts dict n_out, kept, cloned, split, removed)."""
    a = _d(accum)
    n = a.shape[0]
    action = np.zeros(n, np.int32)
    amb = np.zeros(n, np.uint8)
    counts = np.zeros(5, np.int32)
    rc = lib().orc_densify_classify(ctypes.c_int32(n), _p(a), _p(_d(count)), _p(_d(log_scales)), _p(_d(logits)),
                                    ctypes.c_double(grad_threshold), ctypes.c_double(dense_scale),
                                    ctypes.c_double(min_opacity), ctypes.c_double(max_scale), _p(action), _p(amb),
                                    _p(counts))
    if rc != 0:
        raise ValueError(f"orc_densify_classify returned {rc}")
    return action, amb.astype(bool), dict(zip(("n_out", "kept", "cloned", "split", "removed"), (int(x) for x in counts)))


def densify_group(action, param, m=None, v=None, kind=0, quats=None, log_scales=None, noise=None):
    """c12 for one parameter group [rows][n]: (param_out, m_out, v_out) of [rows][n_out]."""
    act = np.ascontiguousarray(action, np.int32)
    n = act.shape[0]
    P = _d(param).reshape(-1, n)
    rows = P.shape[0]
    n_out = int(((act == 1) | (act == 2)).sum() + (act == 2).sum() + 2 * (act == 3).sum())
    po = np.zeros((rows, max(n_out, 1)))
    mo = np.zeros((rows, max(n_out, 1))) if m is not None else None
    vo = np.zeros((rows, max(n_out, 1))) if v is not None else None
    M = None if m is None else _d(m).reshape(rows, n)
    V = None if v is None else _d(v).reshape(rows, n)
    q = None if quats is None else _d(quats)
    ls = None if log_scales is None else _d(log_scales)
    z = None if noise is None else _d(noise)
    if kind == 1 and (q is None or ls is None or z is None):
        raise ValueError("means need quats, log_scales and noise")
    wrote = lib().orc_densify_group(ctypes.c_int32(n), _p(act), ctypes.c_int32(rows), ctypes.c_int32(kind), _p(P),
                                    _p(M), _p(V), _p(q), _p(ls), _p(z), ctypes.c_int32(n_out), _p(po), _p(mo), _p(vo))
    assert wrote == n_out
    cut = lambda x: None if x is None else x[:, :n_out]
    return cut(po), cut(mo), cut(vo)


def render(cam, g, bg=(0.0, 0.0, 0.0), prec: int = 64):
    """Convenience: oracle project (decisions in `prec`) -> bin -> forward compositing."""
    P = project(cam, g, prec=prec)
    B = bin(cam, P["means2d"].astype(np.float32), P["depth"].astype(np.float32), P["radius"])
    F = raster_fwd(cam, P["means2d"], P["conic"], g.opacity, P["color"], B["ranges"],
                   B["point_list"], bg=bg, prec=prec)
    return P, B, F
