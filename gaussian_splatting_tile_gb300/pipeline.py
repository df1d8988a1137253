"""Forward and backward of one view through the five C-ABI calls, with torch-owned buffers.

This layer only allocates (through torch's caching allocator) and sequences the calls of
`rs`; all arithmetic happens in librs.so.  Buffers are kept between frames and grown when
rs_bin reports that the entry count exceeded the capacity.
"""
from __future__ import annotations

import dataclasses

import torch

from . import rs


@dataclasses.dataclass
class Forward:
    proj: rs.DeviceProjected
    n_entries: int
    point_list: torch.Tensor   # int32 [capacity] (uint32 bits)
    keys_sorted: torch.Tensor  # int64 [capacity] (uint64 bits)
    tile_ranges: torch.Tensor  # int32 [n_tiles, 2] (uint32 bits)
    image: torch.Tensor        # [3, H, W]
    final_T: torch.Tensor      # [H, W]
    n_contrib: torch.Tensor    # int32 [H, W] (uint32 bits)
    bg: tuple


@dataclasses.dataclass
class Backward:
    dmeans2d: torch.Tensor
    dconic: torch.Tensor
    dopacity: torch.Tensor
    dcolor: torch.Tensor
    dmeans: torch.Tensor
    dscales: torch.Tensor
    dquats: torch.Tensor
    dsh: torch.Tensor | None


class Renderer:
    """Holds the buffers for one camera size and Gaussian count."""

    def __init__(self, camera, n: int, device="cuda", capacity: int | None = None,
                 keep_keys: bool = True):
        self.camera = camera
        self.n = int(n)
        self.device = torch.device(device)
        self.n_tiles = ((camera.width + 15) // 16) * ((camera.height + 15) // 16)
        self.keep_keys = keep_keys
        self.proj = rs.DeviceProjected.empty(self.n, self.device)
        H, W = camera.height, camera.width
        self.image = torch.empty(3, H, W, dtype=torch.float32, device=self.device)
        self.final_T = torch.empty(H, W, dtype=torch.float32, device=self.device)
        self.n_contrib = torch.empty(H, W, dtype=torch.int32, device=self.device)
        self.tile_ranges = torch.empty(self.n_tiles, 2, dtype=torch.int32, device=self.device)
        self._alloc(capacity if capacity is not None else max(4096, 16 * self.n))
        self.grads = None

    def _alloc(self, capacity: int):
        self.capacity = int(capacity)
        ws = rs.rs_bin_workspace_size(self.n, self.camera, self.capacity)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.point_list = torch.empty(max(self.capacity, 1), dtype=torch.int32, device=self.device)
        self.keys_sorted = (torch.empty(max(self.capacity, 1), dtype=torch.int64, device=self.device)
                            if self.keep_keys else None)

    def set_camera(self, camera):
        assert camera.width == self.camera.width and camera.height == self.camera.height
        self.camera = camera

    def project(self, g: rs.DeviceGaussians, stream=None):
        rs.rs_project(self.camera, g, self.proj, stream)

    def bin(self, stream=None) -> int:
        while True:
            try:
                return rs.rs_bin(self.camera, self.proj, self.n, self.workspace, self.capacity,
                                 self.keys_sorted, self.point_list, self.tile_ranges, stream)
            except rs.RsError as e:
                if e.code != rs.RS_ERR_CAPACITY:
                    raise
                self._alloc(int(e.n_entries * 1.25) + 1024)

    def rasterize(self, bg=(0.0, 0.0, 0.0), stream=None):
        rs.rs_rasterize_fwd(self.camera, self.proj, self.n, self.tile_ranges, self.point_list, bg,
                            self.image, self.final_T, self.n_contrib, stream)

    def forward(self, g: rs.DeviceGaussians, bg=(0.0, 0.0, 0.0), stream=None) -> Forward:
        self.project(g, stream)
        E = self.bin(stream)
        self.rasterize(bg, stream)
        self.bg = tuple(bg)
        self.n_entries = E
        return Forward(self.proj, E, self.point_list, self.keys_sorted, self.tile_ranges,
                       self.image, self.final_T, self.n_contrib, self.bg)

    def _grads(self, sh_degree: int):
        n, d = self.n, self.device
        K = (sh_degree + 1) ** 2 if sh_degree >= 0 else 0
        if self.grads is None or (self.grads.dsh is None) != (K == 0) or (K and self.grads.dsh.shape[0] != 3 * K):
            f = lambda *s: torch.empty(*s, dtype=torch.float32, device=d)
            self.grads = Backward(f(2, n), f(3, n), f(n), f(3, n), f(3, n), f(3, n), f(4, n),
                                  f(3 * K, n) if K else None)
        return self.grads

    def rasterize_backward(self, dL_dimage, stream=None) -> Backward:
        g = self.grads
        rs.rs_rasterize_bwd(self.camera, self.proj, self.n, self.tile_ranges, self.point_list,
                            self.bg, self.final_T, self.n_contrib, dL_dimage, g.dmeans2d, g.dconic,
                            g.dopacity, g.dcolor, stream)
        return g

    def project_backward(self, gs: rs.DeviceGaussians, stream=None) -> Backward:
        g = self.grads
        rs.rs_project_bwd(self.camera, gs, self.proj, g.dmeans2d, g.dconic, g.dcolor, g.dmeans,
                          g.dscales, g.dquats, g.dsh, stream)
        return g

    def backward(self, gs: rs.DeviceGaussians, dL_dimage, stream=None) -> Backward:
        self._grads(gs.sh_degree)
        self.rasterize_backward(dL_dimage, stream)
        return self.project_backward(gs, stream)
