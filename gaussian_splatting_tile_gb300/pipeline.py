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
                 keep_keys: bool = True, tile_test: int = rs.RS_TILE_TEST_SQUARE):
        self.camera = camera
        self.n = int(n)
        self.device = torch.device(device)
        self.n_tiles = ((camera.width + 15) // 16) * ((camera.height + 15) // 16)
        self.keep_keys = keep_keys
        self.cam_struct = rs.camera_struct(camera)
        self._bound = None
        self.proj = rs.DeviceProjected.empty(self.n, self.device, tile_test)
        H, W = camera.height, camera.width
        self.image = torch.empty(3, H, W, dtype=torch.float32, device=self.device)
        self.final_T = torch.empty(H, W, dtype=torch.float32, device=self.device)
        self.n_contrib = torch.empty(H, W, dtype=torch.int32, device=self.device)
        self.tile_ranges = torch.empty(self.n_tiles, 2, dtype=torch.int32, device=self.device)
        self._alloc(capacity if capacity is not None else max(4096, 16 * self.n))
        self.grads = None

    def _alloc(self, capacity: int):
        self._fwd_valid = False  # new entry buffers: a forward must run before any backward
        self.capacity = int(capacity)
        ws = rs.rs_bin_workspace_size(self.n, self.camera, self.capacity)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.point_list = torch.empty(max(self.capacity, 1), dtype=torch.int32, device=self.device)
        self.raster_ws = torch.empty(rs.rs_raster_workspace_size(self.camera, self.capacity), dtype=torch.uint8,
                                     device=self.device)
        self.keys_sorted = (torch.empty(max(self.capacity, 1), dtype=torch.int64, device=self.device)
                            if self.keep_keys else None)

    def set_camera(self, camera):
        assert camera.width == self.camera.width and camera.height == self.camera.height
        self.camera = camera
        rs.set_camera_struct(self.cam_struct, camera)

    # ---- prepared calls: the ctypes arguments of this renderer's buffers, built once
    def _prepare(self, g: rs.DeviceGaussians, bg):
        ptrs = tuple(0 if t is None else t.data_ptr() for t in (g.means, g.scales, g.quats, g.opacity, g.sh, g.colors))
        key = (ptrs, g.n, g.sh_degree, tuple(float(x) for x in bg), self.capacity, self.grads is not None)
        if self._bound is not None and self._bound[0] == key:
            return self._bound[1]
        import ctypes
        cam = ctypes.byref(self.cam_struct)
        gs = g.struct()
        ps = self.proj.struct()
        self._keep = (gs, ps)
        self._E = ctypes.c_size_t(0)
        bgv = (ctypes.c_float * 3)(*[float(x) for x in bg])
        self._bgv = bgv
        vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        self._hres = ctypes.c_void_p(0)  # pinned (E, error) slot of the next rs_bin_async call
        calls = dict(
            project=rs.PreparedCall("rs_project", (cam, ctypes.byref(gs), ctypes.byref(ps))),
            bin_async=rs.PreparedCall("rs_bin_async", (cam, ctypes.byref(ps), self.n, vp(self.workspace),
                                                       self.workspace.numel(), self.capacity, vp(self.keys_sorted),
                                                       vp(self.point_list), vp(self.tile_ranges), self._hres)),
            bin=rs.PreparedCall("rs_bin", (cam, ctypes.byref(ps), self.n, vp(self.workspace),
                                           self.workspace.numel(), self.capacity, vp(self.keys_sorted),
                                           vp(self.point_list), vp(self.tile_ranges), ctypes.byref(self._E))),
            fwd=rs.PreparedCall("rs_rasterize_fwd", (cam, ctypes.byref(ps), self.n, vp(self.tile_ranges),
                                                     vp(self.point_list), self.capacity, bgv, vp(self.image),
                                                     vp(self.final_T), vp(self.n_contrib), vp(self.raster_ws),
                                                     self.raster_ws.numel())))
        if self.grads is not None:
            gr = self.grads
            calls["rbwd_args"] = (cam, ctypes.byref(ps), self.n, vp(self.tile_ranges), vp(self.point_list),
                                  self.capacity, bgv, vp(self.final_T), vp(self.n_contrib),
                                  vp(self.raster_ws), self.raster_ws.numel())
            calls["rbwd_out"] = (vp(gr.dmeans2d), vp(gr.dconic), vp(gr.dopacity), vp(gr.dcolor))
            calls["pbwd"] = rs.PreparedCall("rs_project_bwd", (
                cam, ctypes.byref(gs), ctypes.byref(ps), vp(gr.dmeans2d), vp(gr.dconic), vp(gr.dcolor),
                vp(gr.dmeans), vp(gr.dscales), vp(gr.dquats), vp(gr.dsh)))
        self._bound = (key, calls)
        return calls

    def project(self, g: rs.DeviceGaussians, stream=None):
        self._g = g
        self._prepare(g, getattr(self, "bg", (0.0, 0.0, 0.0)))["project"].run(rs.stream_handle(stream))

    def bin(self, stream=None) -> int:
        h = rs.stream_handle(stream)
        while True:
            try:
                self._prepare(self._g, getattr(self, "bg", (0.0, 0.0, 0.0)))["bin"].run(h)
                return int(self._E.value)
            except rs.RsError as e:
                if e.code != rs.RS_ERR_CAPACITY:
                    raise
                self._alloc(int(self._E.value * 1.25) + 1024)
                self._bound = None

    def bin_async(self, result: torch.Tensor, stream=None):
        """Enqueue the binning without waiting: (E, error flag) land in `result` (pinned int64
        [2]) once the stream gets there.  If E turns out above the capacity, the frame rendered
        the background: grow with `reserve(E)` and redo it."""
        if result.is_cuda or result.dtype != torch.int64 or result.numel() < 2:
            raise TypeError("result must be a pinned int64 host tensor with 2 elements")
        calls = self._prepare(self._g, getattr(self, "bg", (0.0, 0.0, 0.0)))
        self._hres.value = result.data_ptr()
        calls["bin_async"].run(rs.stream_handle(stream))

    def reserve(self, entries: int):
        """Grow the entry buffers to hold at least `entries` entries."""
        if entries > self.capacity:
            self._alloc(int(entries * 1.25) + 1024)
            self._bound = None

    def rasterize(self, bg=(0.0, 0.0, 0.0), stream=None):
        self.bg = tuple(bg)
        self._prepare(self._g, self.bg)["fwd"].run(rs.stream_handle(stream))
        self._fwd_valid = True

    def forward(self, g: rs.DeviceGaussians, bg=(0.0, 0.0, 0.0), stream=None) -> Forward:
        self.bg = tuple(bg)
        self.project(g, stream)
        E = self.bin(stream)
        self.rasterize(bg, stream)
        self.n_entries = E
        return Forward(self.proj, E, self.point_list, self.keys_sorted, self.tile_ranges,
                       self.image, self.final_T, self.n_contrib, self.bg)

    def forward_async(self, g: rs.DeviceGaussians, result: torch.Tensor, bg=(0.0, 0.0, 0.0), stream=None):
        """forward() with the sync-free binning: nothing waits for the entry count, which lands
        in `result` (pinned int64 [2]: E, error flag).  After synchronising, check it with
        `check_async(result)`; a frame whose E exceeded the capacity rendered the background."""
        self.bg = tuple(bg)
        self.project(g, stream)
        self.bin_async(result, stream)
        self.rasterize(bg, stream)

    def check_async(self, result: torch.Tensor) -> int:
        """E of a finished rs_bin_async; raises (after growing the buffers) on overflow or timeout."""
        E, err = int(result[0]), int(result[1])
        if err:
            raise rs.RsError("rs_bin_async", rs.RS_ERR_DEVICE_TIMEOUT, rs.error_string(rs.RS_ERR_DEVICE_TIMEOUT))
        if E > self.capacity:
            self.reserve(E)
            err = rs.RsError("rs_bin_async", rs.RS_ERR_CAPACITY, rs.error_string(rs.RS_ERR_CAPACITY))
            err.n_entries = E
            raise err
        self.n_entries = E
        return E

    def _grads(self, sh_degree: int):
        n, d = self.n, self.device
        K = (sh_degree + 1) ** 2 if sh_degree >= 0 else 0
        if self.grads is None or (self.grads.dsh is None) != (K == 0) or (K and self.grads.dsh.shape[0] != 3 * K):
            f = lambda *s: torch.empty(*s, dtype=torch.float32, device=d)
            self.grads = Backward(f(2, n), f(3, n), f(n), f(3, n), f(3, n), f(3, n), f(4, n),
                                  f(3 * K, n) if K else None)
            self._bound = None  # prepared calls must point at the new gradient buffers
            return True
        return False

    def rasterize_backward(self, dL_dimage, stream=None) -> Backward:
        import ctypes
        if not (dL_dimage.is_cuda and dL_dimage.dtype == torch.float32 and dL_dimage.is_contiguous()
                and dL_dimage.numel() >= 3 * self.camera.width * self.camera.height):
            raise ValueError("dL_dimage must be a contiguous float32 CUDA tensor [3, H, W]")
        if not self._fwd_valid:
            raise RuntimeError("the entry buffers changed since the last forward: run the forward again")
        calls = self._prepare(self._g, self.bg)
        fn = rs.PreparedCall("rs_rasterize_bwd", calls["rbwd_args"] + (ctypes.c_void_p(dL_dimage.data_ptr()),)
                             + calls["rbwd_out"])
        fn.run(rs.stream_handle(stream))
        return self.grads

    def project_backward(self, gs: rs.DeviceGaussians, stream=None) -> Backward:
        self._prepare(gs, self.bg)["pbwd"].run(rs.stream_handle(stream))
        return self.grads

    def backward(self, gs: rs.DeviceGaussians, dL_dimage, stream=None) -> Backward:
        self._grads(gs.sh_degree)
        self.rasterize_backward(dL_dimage, stream)
        return self.project_backward(gs, stream)


class AppearanceStep:
    """The training-shaped step of rigel's appearance-MLP model ("Appearance MLP" and its training
    loop): per view, the MLP gives every Gaussian its colour, the rasteriser renders it, the L1
    loss against the view's target gives dL/dimage, and the backward runs through compositing,
    projection and the MLP.  Every stage is a call of the C ABI; this class only owns buffers.

    `forward` and `backward` are separate so that a caller can inspect or change dL/dimage in
    between; `view` runs both."""

    def __init__(self, camera, g: rs.DeviceGaussians, mlp: rs.DeviceMLP, latents: torch.Tensor,
                 device="cuda", capacity: int | None = None):
        self.device = torch.device(device)
        self.g, self.mlp, self.latents = g, mlp, latents
        n = g.n
        self.R = Renderer(camera, n, self.device, capacity)
        self.colors = torch.empty(3, n, dtype=torch.float32, device=self.device)
        # geometry of g with the MLP's colours as the colour source
        self.gc = rs.DeviceGaussians(g.means, g.scales, g.quats, g.opacity, None, -1, self.colors)
        H, W = camera.height, camera.width
        self.dL_dimage = torch.empty(3, H, W, dtype=torch.float32, device=self.device)
        self.loss = torch.zeros(1, dtype=torch.float32, device=self.device)
        self.dL_dlatents = torch.empty_like(latents)
        self.mlp_grads = rs.DeviceMLPGrads.like(mlp)

    def forward(self, camera, target: torch.Tensor, scale: float, bg=(0.0, 0.0, 0.0), stream=None) -> Forward:
        """MLP colours, render, L1 loss and its gradient (into self.dL_dimage, self.loss)."""
        self.R.set_camera(camera)
        rs.rs_appearance_fwd(camera, self.g.means, self.latents, self.mlp, self.colors, stream)
        F = self.R.forward(self.gc, bg=bg, stream=stream)
        rs.rs_l1_loss_grad(F.image, target, scale, self.dL_dimage, self.loss, stream)
        return F

    def forward_async(self, camera, target: torch.Tensor, scale: float, result: torch.Tensor, bg=(0.0, 0.0, 0.0),
                      stream=None):
        """forward() with the sync-free binning (Renderer.forward_async): nothing waits on the
        host; check the entry count in `result` with self.R.check_async after the stream."""
        self.R.set_camera(camera)
        rs.rs_appearance_fwd(camera, self.g.means, self.latents, self.mlp, self.colors, stream)
        self.R.forward_async(self.gc, result, bg=bg, stream=stream)
        rs.rs_l1_loss_grad(self.R.image, target, scale, self.dL_dimage, self.loss, stream)

    def backward(self, dL_dimage: torch.Tensor | None = None, stream=None) -> Backward:
        """Compositing and projection backward from dL/dimage (default: the L1 gradient), then
        the MLP backward (into self.dL_dlatents and self.mlp_grads)."""
        B = self.R.backward(self.gc, self.dL_dimage if dL_dimage is None else dL_dimage, stream)
        self.mlp_backward(B.dcolor, stream)
        return B

    def mlp_backward(self, dL_dcolor: torch.Tensor, stream=None):
        rs.rs_appearance_bwd(self.R.camera, self.g.means, self.latents, self.mlp, dL_dcolor,
                             self.dL_dlatents, self.mlp_grads, stream)

    def view(self, camera, target, scale, bg=(0.0, 0.0, 0.0), stream=None):
        F = self.forward(camera, target, scale, bg, stream)
        return F, self.backward(stream=stream)


class AppearanceGraph:
    """One view of the training-shaped step (MLP colours, render, L1 loss, render backward, MLP
    backward) captured as a single CUDA graph, like FrameGraph: the camera is fixed, the
    latents, weights, Gaussians and target are read from their buffers at every replay, and
    `check()` (after the stream has passed the replay) returns the entry count."""

    def __init__(self, step: AppearanceStep, camera, target: torch.Tensor, scale: float, bg=(0.0, 0.0, 0.0)):
        self.step, self.camera = step, camera
        self.result = torch.zeros(2, dtype=torch.int64).pin_memory()
        R = step.R
        R._grads(-1)
        step.forward_async(camera, target, scale, self.result, bg)
        step.backward()
        torch.cuda.current_stream(R.device).synchronize()
        R.check_async(self.result)
        self.capacity = R.capacity
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            step.forward_async(camera, target, scale, self.result, bg)
            step.backward()

    def replay(self):
        if self.step.R.capacity != self.capacity:
            raise RuntimeError("the renderer's buffers changed since the capture")
        self.graph.replay()

    def check(self) -> int:
        return self.step.R.check_async(self.result)


class FrameGraph:
    """One view's forward and backward captured as a single CUDA graph and replayed.

    Every call of the frame is stream-ordered with no host wait (the binning's entry count is
    copied to pinned host memory in stream order, `rs_bin_async`), so projection, binning,
    compositing and both backward passes fit in one graph launch -- the sync-free, graph-captured
    pipeline that "3D Gaussian Splatting ビューワを作る" (4.2-4.3, indirect dispatch) and the rigel
    README ("Binning", the one device-to-host sync) point to.  The kernels take the camera by
    value, so a graph belongs to one view (`FrameGraphs` keeps one per view).  A replay reads the
    Gaussians and dL/dimage from the buffers given at capture and writes the renderer's buffers.
    `check()` (after the stream has passed the replay) returns the entry count and raises when
    it exceeded the capacity: that frame rendered the background, the renderer has grown and the
    graph must be captured again."""

    def __init__(self, R: Renderer, gs: rs.DeviceGaussians, dL_dimage: torch.Tensor, camera,
                 bg=(0.0, 0.0, 0.0)):
        self.R, self.camera, self.bg = R, camera, tuple(bg)
        self.result = torch.zeros(2, dtype=torch.int64).pin_memory()
        R.set_camera(camera)
        R._grads(gs.sh_degree)
        # one eager frame: builds the prepared calls and checks that the buffers are big enough
        R.forward_async(gs, self.result, bg)
        R.backward(gs, dL_dimage)
        torch.cuda.current_stream(R.device).synchronize()
        R.check_async(self.result)
        self.capacity = R.capacity
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            R.forward_async(gs, self.result, bg)
            R.backward(gs, dL_dimage)

    def replay(self):
        if self.R.capacity != self.capacity:
            raise RuntimeError("the renderer's buffers changed since the capture")
        self.graph.replay()

    def check(self) -> int:
        return self.R.check_async(self.result)


class FrameGraphs:
    """One `FrameGraph` per view of a fixed camera list, captured on first use."""

    def __init__(self, R: Renderer, gs: rs.DeviceGaussians, dL_dimage: torch.Tensor, cameras,
                 bg=(0.0, 0.0, 0.0)):
        self.R, self.gs, self.dL, self.cameras, self.bg = R, gs, dL_dimage, list(cameras), tuple(bg)
        self.graphs: dict[int, FrameGraph] = {}

    def get(self, view: int) -> FrameGraph:
        fg = self.graphs.get(view)
        if fg is None or fg.capacity != self.R.capacity:
            fg = FrameGraph(self.R, self.gs, self.dL, self.cameras[view], self.bg)
            self.graphs[view] = fg
        return fg


class StreamedFrames:
    """Forward + backward of a sequence of views whose Gaussian parameters and dL/dimage come
    from pinned host memory and whose per-Gaussian gradients go back to pinned host memory, with
    the copies of one frame overlapping the compute of its neighbours.

    `slots` slots (at least two), each a renderer with its own device inputs, gradients,
    per-view frame graphs and compute stream, take the frames in turn.  Frame k's host-to-device
    copies run on an input copy stream once frame k - slots (same slot) has finished reading its
    inputs; its graph replays on its slot's compute stream once those copies and frame
    k - slots' device-to-host copies are done; its gradients go back on an output copy stream
    once it has finished.  So the two copy directions and the compute of neighbouring frames
    proceed at once (one frame's latency-bound binning overlaps another's compositing), and a
    step costs about the longest of them.

    `host_in`: pinned float32 tensors means [3,N], scales [3,N], quats [4,N], opacity [N] and
    sh [3K,N] (or colors [3,N] with sh_degree -1); `host_dL`: pinned [3,H,W].  `host_out[slot]`
    receives dmeans, dscales, dquats, dopacity, dsh (or dcolor) of that slot's frames."""

    OUT = ("dmeans", "dscales", "dquats", "dopacity")

    def __init__(self, cameras, host_in: dict, sh_degree: int, host_dL: torch.Tensor, device="cuda",
                 capacity: int | None = None, bg=(0.0, 0.0, 0.0), slots: int = 2):
        self.device = torch.device(device)
        self.cameras = list(cameras)
        self.host_in, self.host_dL, self.sh_degree = host_in, host_dL, sh_degree
        n = int(host_in["opacity"].shape[0])
        self.out_names = self.OUT + (("dsh",) if sh_degree >= 0 else ("dcolor",))
        self.slots = []
        self.n_slots = max(2, int(slots))
        for _ in range(self.n_slots):
            R = Renderer(self.cameras[0], n, self.device, capacity=capacity, keep_keys=False)
            dev = {k: torch.empty_like(v, device=self.device) for k, v in host_in.items()}
            if sh_degree >= 0:
                dg = rs.DeviceGaussians(dev["means"], dev["scales"], dev["quats"], dev["opacity"], dev["sh"],
                                        sh_degree)
            else:
                dg = rs.DeviceGaussians(dev["means"], dev["scales"], dev["quats"], dev["opacity"], None, -1,
                                        dev["colors"])
            ddL = torch.empty_like(host_dL, device=self.device)
            R._grads(sh_degree)
            host_out = {k: torch.empty(tuple(getattr(R.grads, k).shape), dtype=torch.float32).pin_memory()
                        for k in self.out_names}
            ev = lambda: torch.cuda.Event()
            self.slots.append(dict(R=R, dev=dev, dg=dg, ddL=ddL, host_out=host_out,
                                   graphs=FrameGraphs(R, dg, ddL, self.cameras, bg), in_ready=ev(),
                                   comp_done=ev(), out_done=ev(), frames=[]))
        self.compute = [torch.cuda.Stream(self.device) for _ in self.slots]
        self.h2d = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self.k = 0

    @property
    def host_out(self):
        return [s["host_out"] for s in self.slots]

    def prepare(self, views):
        """Captures the frame graphs of `views` in both slots (each capture runs one frame)."""
        cur = torch.cuda.current_stream(self.device)
        for s in self.slots:
            for v in sorted(set(views)):
                self._copy_in(s)
                cur.wait_event(s["in_ready"])
                s["graphs"].get(v)
        torch.cuda.synchronize(self.device)

    def _copy_in(self, s):
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(s["comp_done"])  # the slot's previous frame has read its inputs
            for k, v in self.host_in.items():
                s["dev"][k].copy_(v, non_blocking=True)
            s["ddL"].copy_(self.host_dL, non_blocking=True)
            s["in_ready"].record(self.h2d)

    def frame(self, view: int):
        """Enqueues one frame of `view`; nothing waits on the host."""
        slot = self.k % self.n_slots
        s, cs = self.slots[slot], self.compute[slot]
        self.k += 1
        fg = s["graphs"].get(view)  # captured already after prepare(); else captured here
        self._copy_in(s)
        cs.wait_event(s["in_ready"])
        cs.wait_event(s["out_done"])  # the slot's previous gradients are on the host
        with torch.cuda.stream(cs):
            fg.replay()
        s["comp_done"].record(cs)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(s["comp_done"])
            for k in self.out_names:
                s["host_out"][k].copy_(getattr(s["R"].grads, k), non_blocking=True)
            s["out_done"].record(self.d2h)
        s["frames"].append(fg)

    def finish(self) -> list[int]:
        """Waits for every enqueued frame; returns their entry counts (raises on an overflow)."""
        torch.cuda.synchronize(self.device)
        counts = []
        for s in self.slots:
            counts += [fg.check() for fg in s["frames"]]
            s["frames"].clear()
        return counts
