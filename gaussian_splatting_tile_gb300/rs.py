"""Thin Python binding of the C ABI in include/rs.h (librs.so), with the same names.

Argument marshalling only: torch tensors are checked (device, dtype, contiguity, shape) and
their device pointers and the current CUDA stream are handed to the library; every step of the
rasteriser runs in the library's kernels.  There is no fallback: if librs.so is missing or the
GPU is unavailable, the calls raise.
"""
from __future__ import annotations

import ctypes
import glob
import dataclasses
import os
import re

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librs.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "rs.h")

RS_OK, RS_ERR_INVALID_ARG, RS_ERR_CAPACITY, RS_ERR_WORKSPACE, RS_ERR_CUDA = 0, -1, -2, -3, -4
RS_ERR_DEVICE_TIMEOUT, RS_ERR_DEVICE_CHECK = -5, -6
RS_TILE, RS_RECORD_BYTES, RS_MAX_GAUSSIANS, RS_MAX_ENTRIES = 16, 48, 1 << 26, (1 << 30) - 1
RECORD_BYTES = 48
TILE = 16


class RsError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with {code}: {msg}")
        self.code = code


class rs_camera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3),
                ("fx", ctypes.c_float), ("fy", ctypes.c_float),
                ("cx", ctypes.c_float), ("cy", ctypes.c_float),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32)]


class rs_gaussians(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("d_means", ctypes.c_void_p), ("d_scales", ctypes.c_void_p),
                ("d_quats", ctypes.c_void_p), ("d_opacity", ctypes.c_void_p),
                ("d_sh", ctypes.c_void_p), ("sh_degree", ctypes.c_int32),
                ("d_colors", ctypes.c_void_p)]


class rs_projected(ctypes.Structure):
    _fields_ = [("d_means2d", ctypes.c_void_p), ("d_depth", ctypes.c_void_p),
                ("d_conic", ctypes.c_void_p), ("d_color", ctypes.c_void_p),
                ("d_radius", ctypes.c_void_p), ("d_tiles_touched", ctypes.c_void_p),
                ("d_records", ctypes.c_void_p), ("d_ellipse", ctypes.c_void_p),
                ("tile_test", ctypes.c_int32)]


RS_TILE_TEST_SQUARE, RS_TILE_TEST_ELLIPSE = 0, 1
RS_ELLIPSE_WORDS = 12  # rows of the ellipse tile test's per-Gaussian words
RS_RASTER_CHUNK = 256  # entries per backward task; spacing of the forward's recorded states


class rs_mlp(ctypes.Structure):
    _fields_ = [("latent_dim", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("d_W1", ctypes.c_void_p), ("d_b1", ctypes.c_void_p),
                ("d_W2", ctypes.c_void_p), ("d_b2", ctypes.c_void_p)]


class rs_mlp_grads(ctypes.Structure):
    _fields_ = [("d_dW1", ctypes.c_void_p), ("d_db1", ctypes.c_void_p),
                ("d_dW2", ctypes.c_void_p), ("d_db2", ctypes.c_void_p)]


class rs_adam_segment(ctypes.Structure):
    _fields_ = [("d_param", ctypes.c_void_p), ("d_grad", ctypes.c_void_p), ("d_m", ctypes.c_void_p),
                ("d_v", ctypes.c_void_p), ("d_activated", ctypes.c_void_p), ("count", ctypes.c_size_t),
                ("lr", ctypes.c_float), ("activation", ctypes.c_int32)]


RS_ACT_IDENTITY, RS_ACT_EXP, RS_ACT_SIGMOID = 0, 1, 2
RS_ADAM_MAX_SEGMENTS = 16

_lib = None
_VP = ctypes.c_void_p


def declared_signatures(header: str | None = None):
    """(return type, name) of the entry points the headers under include/ declare (or `header`)."""
    headers = [header] if header else sorted(glob.glob(os.path.join(os.path.dirname(HEADER), "*.h")))
    text = "".join(open(h).read() for h in headers)
    return sorted(set(re.findall(r"^\s*(int|const char\*|size_t)\s+(rs_\w+)\s*\(", text, re.M)))


def declared_symbols(header: str | None = None):
    """Names of the entry points the headers under include/ declare (or `header`)."""
    return sorted({name for _, name in declared_signatures(header)})


_RESTYPES = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char*": ctypes.c_char_p}


def lib():
    """Load librs.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m gaussian_splatting_tile_gb300.build_lib`")
        L = ctypes.CDLL(LIB_PATH)
        L.rs_error_string.restype = ctypes.c_char_p
        L.rs_error_string.argtypes = [ctypes.c_int]
        L.rs_project.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_gaussians),
                                 ctypes.POINTER(rs_projected), _VP]
        L.rs_bin_workspace_size.argtypes = [ctypes.c_int32, ctypes.POINTER(rs_camera), ctypes.c_size_t,
                                            ctypes.POINTER(ctypes.c_size_t)]
        L.rs_bin.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_projected), ctypes.c_int32,
                             _VP, ctypes.c_size_t, ctypes.c_size_t, _VP, _VP, _VP,
                             ctypes.POINTER(ctypes.c_size_t), _VP]
        L.rs_bin_async.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_projected), ctypes.c_int32,
                                   _VP, ctypes.c_size_t, ctypes.c_size_t, _VP, _VP, _VP, _VP, _VP]
        L.rs_bin_noalloc.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_projected), ctypes.c_int32,
                                     ctypes.c_size_t, _VP, _VP, _VP, ctypes.POINTER(ctypes.c_size_t), _VP]
        L.rs_raster_workspace_size.argtypes = [ctypes.POINTER(rs_camera), ctypes.c_size_t]
        L.rs_raster_workspace_size.restype = ctypes.c_size_t
        L.rs_rasterize_fwd.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_projected),
                                       ctypes.c_int32, _VP, _VP, ctypes.c_size_t, ctypes.POINTER(ctypes.c_float),
                                       _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]
        L.rs_rasterize_bwd.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_projected),
                                       ctypes.c_int32, _VP, _VP, ctypes.c_size_t, ctypes.POINTER(ctypes.c_float),
                                       _VP, _VP, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, _VP, _VP]
        L.rs_project_bwd.argtypes = [ctypes.POINTER(rs_camera), ctypes.POINTER(rs_gaussians),
                                     ctypes.POINTER(rs_projected), _VP, _VP, _VP, _VP, _VP, _VP,
                                     _VP, _VP]
        L.rs_appearance_fwd.argtypes = [ctypes.POINTER(rs_camera), ctypes.c_int32, _VP, _VP,
                                        ctypes.POINTER(rs_mlp), _VP, _VP]
        L.rs_appearance_bwd.argtypes = [ctypes.POINTER(rs_camera), ctypes.c_int32, _VP, _VP,
                                        ctypes.POINTER(rs_mlp), _VP, _VP, ctypes.POINTER(rs_mlp_grads), _VP]
        L.rs_l1_loss_grad.argtypes = [ctypes.c_size_t, _VP, _VP, ctypes.c_float, _VP, _VP, _VP]
        L.rs_adam_step.argtypes = [ctypes.POINTER(rs_adam_segment), ctypes.c_int32, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_double, ctypes.c_int32, _VP]
        L.rs_densify_stats.argtypes = [ctypes.c_int32, _VP, _VP, _VP, _VP, _VP]
        L.rs_densify_workspace_size.argtypes = [ctypes.c_int32]
        L.rs_densify_plan.argtypes = [ctypes.c_int32, _VP, _VP, _VP, _VP, ctypes.POINTER(rs_densify_rule), _VP,
                                      ctypes.c_size_t, _VP, ctypes.POINTER(ctypes.c_int32), _VP]
        L.rs_densify_apply.argtypes = [ctypes.c_int32, _VP, ctypes.c_size_t, _VP, _VP, _VP,
                                       ctypes.POINTER(rs_densify_group), ctypes.c_int32, ctypes.c_int32, _VP]
        L.rs_l1_dssim_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.POINTER(ctypes.c_size_t)]
        L.rs_l1_dssim_loss_grad.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _VP, _VP, ctypes.c_float,
                                            ctypes.c_float, _VP, _VP, _VP, ctypes.c_size_t, _VP]
        L.rs_device_error.argtypes = []
        for ret, name in declared_signatures():
            getattr(L, name).restype = _RESTYPES[ret]
        _lib = L
    return _lib


def error_string(code: int) -> str:
    return lib().rs_error_string(code).decode()


def _check(fn: str, code: int):
    if code != RS_OK:
        raise RsError(fn, code, error_string(code))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t, dtype=None, numel=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return ctypes.c_void_p(t.data_ptr())


def camera_struct(cam) -> rs_camera:
    c = rs_camera()
    R = np.asarray(cam.R, np.float32).reshape(9)
    t = np.asarray(cam.t, np.float32).reshape(3)
    for i in range(9):
        c.R[i] = float(R[i])
    for i in range(3):
        c.t[i] = float(t[i])
    c.fx, c.fy, c.cx, c.cy = float(cam.fx), float(cam.fy), float(cam.cx), float(cam.cy)
    c.width, c.height = int(cam.width), int(cam.height)
    return c


@dataclasses.dataclass
class DeviceGaussians:
    """Planar float32 CUDA tensors: means [3,N], scales [3,N], quats [4,N], opacity [N],
    sh [3K,N] (sh_degree 0..3) or colors [3,N] (sh_degree -1)."""
    means: torch.Tensor
    scales: torch.Tensor
    quats: torch.Tensor
    opacity: torch.Tensor
    sh: torch.Tensor | None
    sh_degree: int
    colors: torch.Tensor | None = None

    @property
    def n(self) -> int:
        return int(self.opacity.shape[0])

    @staticmethod
    def from_numpy(g, device="cuda"):
        f = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
        return DeviceGaussians(f(g.means), f(g.scales), f(g.quats), f(g.opacity), f(g.sh),
                               int(g.sh_degree), f(g.colors))

    def struct(self) -> rs_gaussians:
        n = self.n
        s = rs_gaussians()
        s.n = n
        s.d_means = _ptr(self.means, torch.float32, 3 * n, "means")
        s.d_scales = _ptr(self.scales, torch.float32, 3 * n, "scales")
        s.d_quats = _ptr(self.quats, torch.float32, 4 * n, "quats")
        s.d_opacity = _ptr(self.opacity, torch.float32, n, "opacity")
        s.sh_degree = int(self.sh_degree)
        if self.sh_degree >= 0:
            s.d_sh = _ptr(self.sh, torch.float32, 3 * (self.sh_degree + 1) ** 2 * n, "sh")
        else:
            s.d_colors = _ptr(self.colors, torch.float32, 3 * n, "colors")
        return s


@dataclasses.dataclass
class DeviceProjected:
    means2d: torch.Tensor
    depth: torch.Tensor
    conic: torch.Tensor
    color: torch.Tensor
    radius: torch.Tensor
    tiles_touched: torch.Tensor
    records: torch.Tensor  # uint8 [N*48]
    ellipse: torch.Tensor | None = None  # [RS_ELLIPSE_WORDS, N], the ellipse tile test's words:
                                         # row 0 its k, the rest its setup for the binning
    tile_test: int = 0                   # RS_TILE_TEST_SQUARE or RS_TILE_TEST_ELLIPSE

    @staticmethod
    def empty(n: int, device="cuda", tile_test: int = 0):
        f = lambda *s: torch.empty(*s, dtype=torch.float32, device=device)
        return DeviceProjected(f(2, n), f(n), f(3, n), f(3, n),
                               torch.empty(n, dtype=torch.int32, device=device),
                               torch.empty(n, dtype=torch.int32, device=device),
                               torch.empty(max(n, 1) * RECORD_BYTES, dtype=torch.uint8, device=device),
                               f(RS_ELLIPSE_WORDS, max(n, 1)) if tile_test == RS_TILE_TEST_ELLIPSE else None,
                               int(tile_test))

    @property
    def alpha_k(self) -> torch.Tensor | None:
        """k of the alpha >= 1/255 ellipse, per Gaussian (0 when culled); ellipse test only."""
        return None if self.ellipse is None else self.ellipse[0, : self.depth.shape[0]]

    def struct(self) -> rs_projected:
        n = int(self.depth.shape[0])
        s = rs_projected()
        s.d_means2d = _ptr(self.means2d, torch.float32, 2 * n, "means2d")
        s.d_depth = _ptr(self.depth, torch.float32, n, "depth")
        s.d_conic = _ptr(self.conic, torch.float32, 3 * n, "conic")
        s.d_color = _ptr(self.color, torch.float32, 3 * n, "color")
        s.d_radius = _ptr(self.radius, torch.int32, n, "radius")
        s.d_tiles_touched = _ptr(self.tiles_touched, None, n, "tiles_touched")
        s.d_records = _ptr(self.records, torch.uint8, n * RECORD_BYTES, "records")
        s.tile_test = int(self.tile_test)
        if self.tile_test == RS_TILE_TEST_ELLIPSE:
            if self.ellipse is None or self.ellipse.dtype != torch.float32 or not self.ellipse.is_contiguous() \
                    or tuple(self.ellipse.shape) != (RS_ELLIPSE_WORDS, max(n, 1)):
                raise ValueError(f"ellipse: want a contiguous float32 [{RS_ELLIPSE_WORDS}, {max(n, 1)}] tensor")
            s.d_ellipse = ctypes.c_void_p(self.ellipse.data_ptr())
        return s


# ------------------------------------------------------------------ prepared calls
class PreparedCall:
    """One C-ABI call with its arguments marshalled once: the pointer arguments of a fixed set of
    buffers are built a single time and the camera struct is shared (and updated in place when the
    view changes), so a frame loop pays only the foreign call.  `run(stream_handle)` returns the
    library's return code after raising on errors."""

    def __init__(self, name: str, args):
        self.name = name
        self.fn = getattr(lib(), name)
        self.args = tuple(args)

    def run(self, stream_handle) -> int:
        rc = self.fn(*self.args, stream_handle)
        if rc != RS_OK:
            raise RsError(self.name, rc, error_string(rc))
        return rc


def set_camera_struct(c: rs_camera, cam) -> rs_camera:
    """Overwrite an existing rs_camera with `cam` (prepared calls keep pointing at it)."""
    R = np.asarray(cam.R, np.float32).reshape(9)
    t = np.asarray(cam.t, np.float32).reshape(3)
    c.R[:] = [float(x) for x in R]
    c.t[:] = [float(x) for x in t]
    c.fx, c.fy, c.cx, c.cy = float(cam.fx), float(cam.fy), float(cam.cx), float(cam.cy)
    c.width, c.height = int(cam.width), int(cam.height)
    return c


def stream_handle(stream=None):
    return _stream(stream)


# ------------------------------------------------------------------ the five calls

def rs_project(camera, gaussians: DeviceGaussians, out: DeviceProjected, stream=None):
    c, g, o = camera_struct(camera), gaussians.struct(), out.struct()
    _check("rs_project", lib().rs_project(ctypes.byref(c), ctypes.byref(g), ctypes.byref(o), _stream(stream)))


def rs_bin_workspace_size(n: int, camera, capacity: int) -> int:
    c = camera_struct(camera)
    b = ctypes.c_size_t(0)
    _check("rs_bin_workspace_size", lib().rs_bin_workspace_size(int(n), ctypes.byref(c), int(capacity), ctypes.byref(b)))
    return int(b.value)


def rs_bin(camera, proj: DeviceProjected, n: int, workspace: torch.Tensor, capacity: int,
           keys_sorted, point_list: torch.Tensor, tile_ranges: torch.Tensor, stream=None) -> int:
    """Returns the entry count E; raises RsError (code RS_ERR_CAPACITY, .n_entries set) when
    E exceeds `capacity`."""
    c = camera_struct(camera)
    p = proj.struct()
    E = ctypes.c_size_t(0)
    rc = lib().rs_bin(ctypes.byref(c), ctypes.byref(p), int(n), _ptr(workspace, torch.uint8, None, "workspace"),
                      int(workspace.numel()), int(capacity), _ptr(keys_sorted, torch.int64, capacity, "keys_sorted"),
                      _ptr(point_list, torch.int32, capacity, "point_list"),
                      _ptr(tile_ranges, torch.int32, 2 * ((camera.width + 15) // 16) * ((camera.height + 15) // 16),
                           "tile_ranges"),
                      ctypes.byref(E), _stream(stream))
    if rc == RS_ERR_CAPACITY:
        err = RsError("rs_bin", rc, error_string(rc))
        err.n_entries = int(E.value)
        raise err
    _check("rs_bin", rc)
    return int(E.value)


def rs_bin_async(camera, proj: DeviceProjected, n: int, workspace: torch.Tensor, capacity: int,
                 keys_sorted, point_list: torch.Tensor, tile_ranges: torch.Tensor, result: torch.Tensor,
                 stream=None):
    """rs_bin without the host wait: enqueues the binning and a copy of (E, error flag) into
    `result` (int64 [2], pinned host memory); read it after synchronising the stream."""
    if result.is_cuda or result.dtype != torch.int64 or result.numel() < 2 or not result.is_contiguous():
        raise TypeError("result must be a contiguous int64 host tensor with 2 elements (pinned)")
    c = camera_struct(camera)
    p = proj.struct()
    _check("rs_bin_async", lib().rs_bin_async(
        ctypes.byref(c), ctypes.byref(p), int(n), _ptr(workspace, torch.uint8, None, "workspace"),
        int(workspace.numel()), int(capacity), _ptr(keys_sorted, torch.int64, capacity, "keys_sorted"),
        _ptr(point_list, torch.int32, capacity, "point_list"),
        _ptr(tile_ranges, torch.int32, 2 * ((camera.width + 15) // 16) * ((camera.height + 15) // 16), "tile_ranges"),
        ctypes.c_void_p(result.data_ptr()), _stream(stream)))


def rs_bin_noalloc(camera, proj: DeviceProjected, n: int, capacity: int, keys_sorted,
                   point_list: torch.Tensor, tile_ranges: torch.Tensor, stream=None) -> int:
    """rs_bin without a workspace (the library's fixed scratch array is used).  Returns E; raises
    RsError (RS_ERR_CAPACITY with .n_entries, or RS_ERR_WORKSPACE when the sizes exceed the
    fixed scratch)."""
    c = camera_struct(camera)
    p = proj.struct()
    E = ctypes.c_size_t(0)
    rc = lib().rs_bin_noalloc(ctypes.byref(c), ctypes.byref(p), int(n), int(capacity),
                              _ptr(keys_sorted, torch.int64, capacity, "keys_sorted"),
                              _ptr(point_list, torch.int32, capacity, "point_list"),
                              _ptr(tile_ranges, torch.int32,
                                   2 * ((camera.width + 15) // 16) * ((camera.height + 15) // 16), "tile_ranges"),
                              ctypes.byref(E), _stream(stream))
    if rc == RS_ERR_CAPACITY:
        err = RsError("rs_bin_noalloc", rc, error_string(rc))
        err.n_entries = int(E.value)
        raise err
    _check("rs_bin_noalloc", rc)
    return int(E.value)


def _bg(bg):
    arr = (ctypes.c_float * 3)(*[float(x) for x in bg])
    return arr


def rs_raster_workspace_size(camera, capacity: int) -> int:
    """Bytes of the compositing workspace for a point list of `capacity` entries."""
    c = camera_struct(camera)
    n = int(lib().rs_raster_workspace_size(ctypes.byref(c), int(capacity)))
    if n == 0:
        raise ValueError("invalid camera or capacity")
    return n


def rs_rasterize_fwd(camera, proj: DeviceProjected, n: int, tile_ranges, point_list, bg, image,
                     final_T, n_contrib, workspace, stream=None):
    c = camera_struct(camera)
    p = proj.struct()
    HW = camera.width * camera.height
    _check("rs_rasterize_fwd", lib().rs_rasterize_fwd(
        ctypes.byref(c), ctypes.byref(p), int(n), _ptr(tile_ranges, torch.int32, None, "tile_ranges"),
        _ptr(point_list, torch.int32, None, "point_list"), int(point_list.numel()), _bg(bg),
        _ptr(image, torch.float32, 3 * HW, "image"), _ptr(final_T, torch.float32, HW, "final_T"),
        _ptr(n_contrib, torch.int32, HW, "n_contrib"), _ptr(workspace, torch.uint8, None, "workspace"),
        int(workspace.numel()), _stream(stream)))


def rs_rasterize_bwd(camera, proj: DeviceProjected, n: int, tile_ranges, point_list, bg, final_T,
                     n_contrib, workspace, dL_dimage, dL_dmeans2d, dL_dconic, dL_dopacity, dL_dcolor,
                     stream=None):
    c = camera_struct(camera)
    p = proj.struct()
    HW = camera.width * camera.height
    _check("rs_rasterize_bwd", lib().rs_rasterize_bwd(
        ctypes.byref(c), ctypes.byref(p), int(n), _ptr(tile_ranges, torch.int32, None, "tile_ranges"),
        _ptr(point_list, torch.int32, None, "point_list"), int(point_list.numel()), _bg(bg),
        _ptr(final_T, torch.float32, HW, "final_T"),
        _ptr(n_contrib, torch.int32, HW, "n_contrib"), _ptr(workspace, torch.uint8, None, "workspace"),
        int(workspace.numel()), _ptr(dL_dimage, torch.float32, 3 * HW, "dL_dimage"),
        _ptr(dL_dmeans2d, torch.float32, 2 * n, "dL_dmeans2d"), _ptr(dL_dconic, torch.float32, 3 * n, "dL_dconic"),
        _ptr(dL_dopacity, torch.float32, n, "dL_dopacity"), _ptr(dL_dcolor, torch.float32, 3 * n, "dL_dcolor"),
        _stream(stream)))


def rs_project_bwd(camera, gaussians: DeviceGaussians, proj: DeviceProjected, dL_dmeans2d, dL_dconic,
                   dL_dcolor, dL_dmeans, dL_dscales, dL_dquats, dL_dsh, stream=None):
    c = camera_struct(camera)
    g = gaussians.struct()
    p = proj.struct()
    n = gaussians.n
    K = (gaussians.sh_degree + 1) ** 2 if gaussians.sh_degree >= 0 else 0
    _check("rs_project_bwd", lib().rs_project_bwd(
        ctypes.byref(c), ctypes.byref(g), ctypes.byref(p), _ptr(dL_dmeans2d, torch.float32, 2 * n, "dL_dmeans2d"),
        _ptr(dL_dconic, torch.float32, 3 * n, "dL_dconic"), _ptr(dL_dcolor, torch.float32, 3 * n, "dL_dcolor"),
        _ptr(dL_dmeans, torch.float32, 3 * n, "dL_dmeans"), _ptr(dL_dscales, torch.float32, 3 * n, "dL_dscales"),
        _ptr(dL_dquats, torch.float32, 4 * n, "dL_dquats"),
        _ptr(dL_dsh, torch.float32, 3 * K * n, "dL_dsh") if K else None, _stream(stream)))


# ------------------------------------------------------------------ appearance MLP and L1 loss

@dataclasses.dataclass
class DeviceMLP:
    """Appearance MLP weights as float32 CUDA tensors: W1 [hidden, latent_dim + 3], b1 [hidden],
    W2 [3, hidden], b2 [3]."""
    W1: torch.Tensor
    b1: torch.Tensor
    W2: torch.Tensor
    b2: torch.Tensor

    @property
    def hidden(self) -> int:
        return int(self.W1.shape[0])

    @property
    def latent_dim(self) -> int:
        return int(self.W1.shape[1]) - 3

    @staticmethod
    def from_numpy(p, device="cuda"):
        f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
        return DeviceMLP(f(p["W1"]), f(p["b1"]), f(p["W2"]), f(p["b2"]))

    def struct(self) -> rs_mlp:
        m = rs_mlp()
        H, L = self.hidden, self.latent_dim
        m.latent_dim, m.hidden = L, H
        m.d_W1 = _ptr(self.W1, torch.float32, H * (L + 3), "W1")
        m.d_b1 = _ptr(self.b1, torch.float32, H, "b1")
        m.d_W2 = _ptr(self.W2, torch.float32, 3 * H, "W2")
        m.d_b2 = _ptr(self.b2, torch.float32, 3, "b2")
        return m


@dataclasses.dataclass
class DeviceMLPGrads:
    dW1: torch.Tensor
    db1: torch.Tensor
    dW2: torch.Tensor
    db2: torch.Tensor

    @staticmethod
    def like(m: DeviceMLP):
        return DeviceMLPGrads(torch.empty_like(m.W1), torch.empty_like(m.b1), torch.empty_like(m.W2),
                              torch.empty_like(m.b2))

    def struct(self) -> rs_mlp_grads:
        g = rs_mlp_grads()
        g.d_dW1 = _ptr(self.dW1, torch.float32, None, "dW1")
        g.d_db1 = _ptr(self.db1, torch.float32, None, "db1")
        g.d_dW2 = _ptr(self.dW2, torch.float32, None, "dW2")
        g.d_db2 = _ptr(self.db2, torch.float32, None, "db2")
        return g


def rs_appearance_fwd(camera, means: torch.Tensor, latents: torch.Tensor, mlp: DeviceMLP,
                      colors: torch.Tensor, stream=None):
    n = int(latents.shape[1])
    c, m = camera_struct(camera), mlp.struct()
    _check("rs_appearance_fwd", lib().rs_appearance_fwd(
        ctypes.byref(c), n, _ptr(means, torch.float32, 3 * n, "means"),
        _ptr(latents, torch.float32, mlp.latent_dim * n, "latents"), ctypes.byref(m),
        _ptr(colors, torch.float32, 3 * n, "colors"), _stream(stream)))


def rs_device_error() -> int:
    """RS_ERR_DEVICE_CHECK if a compositing kernel skipped caller data out of range (a point-list
    entry >= n, a tile range past the capacity), RS_ERR_DEVICE_TIMEOUT if a bounded wait gave up,
    since the last call (the flags are cleared), else RS_OK; synchronises the device."""
    return int(lib().rs_device_error())


def rs_appearance_bwd(camera, means: torch.Tensor, latents: torch.Tensor, mlp: DeviceMLP,
                      dL_dcolors: torch.Tensor, dL_dlatents: torch.Tensor, grads: DeviceMLPGrads,
                      stream=None):
    n = int(latents.shape[1])
    c, m, g = camera_struct(camera), mlp.struct(), grads.struct()
    _check("rs_appearance_bwd", lib().rs_appearance_bwd(
        ctypes.byref(c), n, _ptr(means, torch.float32, 3 * n, "means"),
        _ptr(latents, torch.float32, mlp.latent_dim * n, "latents"), ctypes.byref(m),
        _ptr(dL_dcolors, torch.float32, 3 * n, "dL_dcolors"),
        _ptr(dL_dlatents, torch.float32, mlp.latent_dim * n, "dL_dlatents"), ctypes.byref(g), _stream(stream)))


def rs_l1_loss_grad(image: torch.Tensor, target: torch.Tensor, scale: float, dL_dimage: torch.Tensor,
                    loss: torch.Tensor | None = None, stream=None):
    count = int(image.numel())
    if int(target.numel()) != count:
        raise ValueError("image and target differ in size")
    _check("rs_l1_loss_grad", lib().rs_l1_loss_grad(
        count, _ptr(image, torch.float32, count, "image"), _ptr(target, torch.float32, count, "target"),
        ctypes.c_float(scale), _ptr(dL_dimage, torch.float32, count, "dL_dimage"),
        _ptr(loss, torch.float32, 1, "loss"), _stream(stream)))


# ------------------------------------------------------------------ optimiser

@dataclasses.dataclass
class AdamGroup:
    """One parameter group of rs_adam_step: float32 CUDA tensors of equal size."""
    param: torch.Tensor
    grad: torch.Tensor
    m: torch.Tensor
    v: torch.Tensor
    lr: float
    activation: int = RS_ACT_IDENTITY
    activated: torch.Tensor | None = None


def rs_adam_step(groups, step: int, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-15,
                 stream=None):
    if len(groups) > RS_ADAM_MAX_SEGMENTS:
        raise ValueError(f"at most {RS_ADAM_MAX_SEGMENTS} groups per call")
    arr = (rs_adam_segment * max(1, len(groups)))()
    for i, gr in enumerate(groups):
        k = int(gr.param.numel())
        arr[i].d_param = _ptr(gr.param, torch.float32, k, "param")
        arr[i].d_grad = _ptr(gr.grad, torch.float32, k, "grad")
        arr[i].d_m = _ptr(gr.m, torch.float32, k, "m")
        arr[i].d_v = _ptr(gr.v, torch.float32, k, "v")
        arr[i].d_activated = _ptr(gr.activated, torch.float32, k, "activated")
        arr[i].count = k
        arr[i].lr = float(gr.lr)
        arr[i].activation = int(gr.activation)
    _check("rs_adam_step", lib().rs_adam_step(arr, len(groups), float(beta1), float(beta2), float(eps), int(step),
                                              _stream(stream)))


def rs_densify_stats(dL_dmeans2d: torch.Tensor, radius: torch.Tensor, accum: torch.Tensor, count: torch.Tensor,
                     stream=None):
    n = int(radius.numel())
    _check("rs_densify_stats", lib().rs_densify_stats(
        n, _ptr(dL_dmeans2d, torch.float32, 2 * n, "dL_dmeans2d"), _ptr(radius, torch.int32, n, "radius"),
        _ptr(accum, torch.float32, n, "accum"), _ptr(count, torch.float32, n, "count"), _stream(stream)))


RS_DENSIFY_COPY, RS_DENSIFY_MEANS, RS_DENSIFY_LOG_SCALES, RS_DENSIFY_MAX_GROUPS = 0, 1, 2, 8


class rs_densify_rule(ctypes.Structure):
    _fields_ = [("grad_threshold", ctypes.c_float), ("dense_scale", ctypes.c_float),
                ("min_opacity", ctypes.c_float), ("max_scale", ctypes.c_float)]


class rs_densify_group(ctypes.Structure):
    _fields_ = [("d_param", _VP), ("d_m", _VP), ("d_v", _VP), ("d_param_out", _VP), ("d_m_out", _VP),
                ("d_v_out", _VP), ("rows", ctypes.c_int32), ("kind", ctypes.c_int32)]


@dataclasses.dataclass
class DensifyGroup:
    """One parameter array [rows, n] of rs_densify_apply with its Adam moments (m, v may be None);
    the outputs [rows, n_out] (m_out, v_out may be None)."""
    param: torch.Tensor
    param_out: torch.Tensor
    m: torch.Tensor | None = None
    v: torch.Tensor | None = None
    m_out: torch.Tensor | None = None
    v_out: torch.Tensor | None = None
    kind: int = RS_DENSIFY_COPY


def rs_densify_workspace_size(n: int) -> int:
    return int(lib().rs_densify_workspace_size(int(n)))


def rs_densify_plan(accum, count, log_scales, opacity_logits, grad_threshold: float, dense_scale: float,
                    min_opacity: float, max_scale: float, workspace: torch.Tensor, action: torch.Tensor | None = None,
                    stream=None) -> dict:
    """Classification and counts of rs_densify_plan (float32 CUDA tensors; workspace uint8 CUDA of at
    least rs_densify_workspace_size(n) bytes; action: optional uint8 CUDA [n])."""
    n = int(accum.numel())
    rule = rs_densify_rule(float(grad_threshold), float(dense_scale), float(min_opacity), float(max_scale))
    counts = (ctypes.c_int32 * 5)()
    _check("rs_densify_plan", lib().rs_densify_plan(
        n, _ptr(accum, torch.float32, n, "accum"), _ptr(count, torch.float32, n, "count"),
        _ptr(log_scales, torch.float32, 3 * n, "log_scales"), _ptr(opacity_logits, torch.float32, n, "opacity_logits"),
        ctypes.byref(rule), _ptr(workspace, torch.uint8, rs_densify_workspace_size(n), "workspace"),
        ctypes.c_size_t(workspace.numel()), _ptr(action, torch.uint8, n, "action"), counts, _stream(stream)))
    return dict(zip(("n_out", "kept", "cloned", "split", "removed"), (int(x) for x in counts)))


def rs_densify_apply(n: int, workspace: torch.Tensor, quats, log_scales, noise, groups, n_out: int, stream=None):
    """Moves every group (list of DensifyGroup) to its densified outputs; noise: float32 CUDA [2, 3, n]."""
    if len(groups) > RS_DENSIFY_MAX_GROUPS:
        raise ValueError(f"at most {RS_DENSIFY_MAX_GROUPS} groups per call")
    arr = (rs_densify_group * max(1, len(groups)))()
    for k, gr in enumerate(groups):
        rows = int(gr.param.numel()) // max(n, 1)
        arr[k].d_param = _ptr(gr.param, torch.float32, rows * n, "param")
        arr[k].d_m = _ptr(gr.m, torch.float32, rows * n, "m")
        arr[k].d_v = _ptr(gr.v, torch.float32, rows * n, "v")
        arr[k].d_param_out = _ptr(gr.param_out, torch.float32, rows * n_out, "param_out")
        arr[k].d_m_out = _ptr(gr.m_out, torch.float32, rows * n_out, "m_out")
        arr[k].d_v_out = _ptr(gr.v_out, torch.float32, rows * n_out, "v_out")
        arr[k].rows = rows
        arr[k].kind = int(gr.kind)
    _check("rs_densify_apply", lib().rs_densify_apply(
        int(n), _ptr(workspace, torch.uint8, rs_densify_workspace_size(n), "workspace"),
        ctypes.c_size_t(workspace.numel()), _ptr(quats, torch.float32, 4 * n, "quats"),
        _ptr(log_scales, torch.float32, 3 * n, "log_scales"), _ptr(noise, torch.float32, 6 * n, "noise"),
        arr, len(groups), int(n_out), _stream(stream)))


def rs_l1_dssim_workspace_size(channels: int, height: int, width: int) -> int:
    b = ctypes.c_size_t(0)
    _check("rs_l1_dssim_workspace_size", lib().rs_l1_dssim_workspace_size(int(channels), int(height), int(width),
                                                                          ctypes.byref(b)))
    return int(b.value)


def rs_l1_dssim_loss_grad(image: torch.Tensor, target: torch.Tensor, lam: float, scale: float,
                          dL_dimage: torch.Tensor, loss: torch.Tensor | None, workspace: torch.Tensor, stream=None):
    """image, target, dL_dimage: float32 CUDA [C, H, W]; workspace: uint8 CUDA tensor of at least
    rs_l1_dssim_workspace_size bytes."""
    C, H, W = (int(x) for x in image.shape)
    n = C * H * W
    _check("rs_l1_dssim_loss_grad", lib().rs_l1_dssim_loss_grad(
        C, H, W, _ptr(image, torch.float32, n, "image"), _ptr(target, torch.float32, n, "target"),
        ctypes.c_float(lam), ctypes.c_float(scale), _ptr(dL_dimage, torch.float32, n, "dL_dimage"),
        _ptr(loss, torch.float32, 1, "loss"), _ptr(workspace, torch.uint8, None, "workspace"),
        int(workspace.numel()), _stream(stream)))
