"""Seeded synthetic inputs for tile-based Gaussian splatting.

This module only draws inputs: Gaussian parameters, cameras and upstream gradients, as
float32 numpy arrays.  It holds none of the rendering arithmetic; both the CUDA path and
the CPU oracle receive exactly the same arrays from it.

Scene shapes follow the workloads of the rigel README ("Gallery": a sphere shell coloured
by its normals, a three-turn helix and a checkered plane, 160,000 Gaussians; "Numbers":
720x720, 1280x720 and 1920x1080 timings) and the learn-gs notebook "11 - Tiles" (sphere
shells).  Parameters arrive already activated: scales are exp(log-scale), opacities are
sigmoid(logit), as the model layer of rigel applies them before the kernels.

Layout: planar float32, one row per component: means [3,N], scales [3,N],
quats [4,N] (w,x,y,z, unnormalised is allowed), opacity [N], sh [3K,N] with row k*3+ch.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

TILE = 16


@dataclasses.dataclass
class Camera:
    """Pinhole camera; a world point m maps to p = R m + t (row-major R), pixels u = fx x/z + cx."""

    R: np.ndarray  # [3,3] float32
    t: np.ndarray  # [3] float32
    fx: float
    fy: float
    cx: float
    cy: float
    width: int
    height: int

    @property
    def tiles_x(self) -> int:
        return (self.width + TILE - 1) // TILE

    @property
    def tiles_y(self) -> int:
        return (self.height + TILE - 1) // TILE

    @property
    def n_tiles(self) -> int:
        return self.tiles_x * self.tiles_y


def _f32(x) -> float:
    return float(np.float32(x))


def look_at(eye, target, fx, fy, width, height, cx=None, cy=None) -> Camera:
    """Camera at `eye` looking at `target` in a y-up world; image x right, y down, z forward."""
    eye = np.asarray(eye, np.float64)
    target = np.asarray(target, np.float64)
    f = target - eye
    f /= np.linalg.norm(f)
    up = np.array([0.0, 1.0, 0.0])
    if abs(float(f @ up)) > 0.999:
        up = np.array([0.0, 0.0, 1.0])
    right = np.cross(f, up)
    right /= np.linalg.norm(right)
    down = np.cross(f, right)
    R = np.stack([right, down, f]).astype(np.float32)
    t = (-(R.astype(np.float64) @ eye)).astype(np.float32)
    cx = width / 2.0 if cx is None else cx
    cy = height / 2.0 if cy is None else cy
    return Camera(R, t, _f32(fx), _f32(fy), _f32(cx), _f32(cy), int(width), int(height))


def focal_for_vfov(height: int, vfov_deg: float) -> float:
    return (height / 2.0) / math.tan(math.radians(vfov_deg) / 2.0)


def orbit_eye(radius: float, elevation: float, azimuth: float) -> np.ndarray:
    return np.array([radius * math.cos(elevation) * math.sin(azimuth),
                     radius * math.sin(elevation),
                     radius * math.cos(elevation) * math.cos(azimuth)])


@dataclasses.dataclass
class Gaussians:
    means: np.ndarray    # [3,N]
    scales: np.ndarray   # [3,N]
    quats: np.ndarray    # [4,N]
    opacity: np.ndarray  # [N]
    sh: np.ndarray | None  # [3K,N]
    sh_degree: int         # -1 when `colors` is given instead
    colors: np.ndarray | None = None  # [3,N]

    @property
    def n(self) -> int:
        return int(self.opacity.shape[0])


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _random_quats(rng, n):
    q = rng.standard_normal((4, n))
    q /= np.linalg.norm(q, axis=0, keepdims=True)
    return q


def _sphere_dirs(rng, n):
    d = rng.standard_normal((3, n))
    return d / np.linalg.norm(d, axis=0, keepdims=True)


def _pack(means, log_scales, quats, logits, sh, degree):
    return Gaussians(means=np.ascontiguousarray(means, np.float32),
                     scales=np.ascontiguousarray(np.exp(log_scales), np.float32),
                     quats=np.ascontiguousarray(quats, np.float32),
                     opacity=np.ascontiguousarray(_sigmoid(logits), np.float32),
                     sh=None if sh is None else np.ascontiguousarray(sh, np.float32),
                     sh_degree=degree)


def tiny_scene(seed: int = 0, n: int = 2000, opacity_cap: float | None = None):
    """2,000 Gaussians on a unit sphere shell (radial N(0,0.02) noise), log-scales U[-4.5,-3],
    random unit quaternions, opacity sigmoid(N(0,1)), SH degree 0 (DC U[0,1]); 128x128 image,
    fx=fy=150, cx=cy=64, camera at distance 4 looking at the origin."""
    rng = np.random.default_rng(seed)
    means = _sphere_dirs(rng, n) * (1.0 + rng.normal(0.0, 0.02, n))
    log_scales = rng.uniform(-4.5, -3.0, (3, n))
    quats = _random_quats(rng, n)
    logits = rng.standard_normal(n)
    sh = rng.uniform(0.0, 1.0, (3, n))
    g = _pack(means, log_scales, quats, logits, sh, 0)
    if opacity_cap is not None:
        g.opacity = np.minimum(g.opacity, np.float32(opacity_cap))
    cam = look_at([0.0, 0.0, 4.0], [0.0, 0.0, 0.0], 150.0, 150.0, 128, 128)
    return g, cam


def procedural_scene(seed: int = 0, n_sphere: int = 100_000, n_helix: int = 30_000,
                     n_plane: int = 30_000, sh_degree: int = 3,
                     log_scale_range=(-5.0, -3.5)):
    """The 160,000-Gaussian gallery-like scene: a unit sphere shell coloured by its normals, a
    three-turn helix of radius 1.5 and height 2, and a 4x4 checkered plane at y = -1.2.
    Log-scales U[-5,-3.5], random quaternions, opacity sigmoid(N(1,1)); SH degree 3 with DC
    colours as described and higher coefficients N(0, 0.05)."""
    rng = np.random.default_rng(seed)
    n = n_sphere + n_helix + n_plane
    dirs = _sphere_dirs(rng, n_sphere)
    th = rng.uniform(0.0, 1.0, n_helix)
    ang = 6.0 * math.pi * th
    helix = np.stack([1.5 * np.cos(ang), -1.0 + 2.0 * th, 1.5 * np.sin(ang)])
    px = rng.uniform(-2.0, 2.0, n_plane)
    pz = rng.uniform(-2.0, 2.0, n_plane)
    plane = np.stack([px, np.full(n_plane, -1.2), pz])
    means = np.concatenate([dirs, helix, plane], axis=1)
    log_scales = rng.uniform(log_scale_range[0], log_scale_range[1], (3, n))
    quats = _random_quats(rng, n)
    logits = rng.normal(1.0, 1.0, n)
    K = (sh_degree + 1) ** 2
    sh = rng.normal(0.0, 0.05, (3 * K, n))
    dc = np.empty((3, n))
    dc[:, :n_sphere] = (dirs + 1.0) / 2.0
    dc[:, n_sphere:n_sphere + n_helix] = rng.uniform(0.0, 1.0, (3, n_helix))
    checker = (np.floor(px) + np.floor(pz)) % 2
    dc[:, n_sphere + n_helix:] = np.where(checker > 0, 0.85, 0.15)[None, :]
    sh[0:3] = dc
    return _pack(means, log_scales, quats, logits, sh, sh_degree)


def procedural_camera(width: int, height: int, azimuth: float = 0.0, elevation: float = 0.5,
                      radius: float = 4.3, focal: float | None = None) -> Camera:
    """Orbit camera around the origin; focal defaults to a 50-degree vertical field of view."""
    f = focal_for_vfov(height, 50.0) if focal is None else focal
    return look_at(orbit_eye(radius, elevation, azimuth), [0.0, 0.0, 0.0], f, f, width, height)


def orbit_cameras(width: int, height: int, views: int = 60):
    return [procedural_camera(width, height, azimuth=2.0 * math.pi * k / views) for k in range(views)]


def stress_scene(seed: int = 0, n: int = 1_000_000):
    """1,000,000 Gaussians uniform in a 6x6x6 cube, log-scales U[-6,-2], random quaternions,
    opacity sigmoid(N(0,1.5)), SH degree 3 (DC U[0,1], rest N(0,0.05)); 1920x1080 from distance 5."""
    rng = np.random.default_rng(seed)
    means = rng.uniform(-3.0, 3.0, (3, n))
    log_scales = rng.uniform(-6.0, -2.0, (3, n))
    quats = _random_quats(rng, n)
    logits = rng.normal(0.0, 1.5, n)
    sh = rng.normal(0.0, 0.05, (48, n))
    sh[0:3] = rng.uniform(0.0, 1.0, (3, n))
    g = _pack(means, log_scales, quats, logits, sh, 3)
    f = focal_for_vfov(1080, 50.0)
    cam = look_at([0.0, 0.0, 5.0], [0.0, 0.0, 0.0], f, f, 1920, 1080)
    return g, cam


def training_scene(seed: int = 0, n: int = 250_000, views: int = 8, size: int = 400,
                   latent_dim: int = 8, hidden: int = 64):
    """Training-shaped workload: the sphere/helix/plane mix at 250,000 Gaussians, 8 random views of
    400x400 at radius 4.3 (50-degree field of view), an 8-d latent N(0,1) per Gaussian and a
    Xavier-uniform initialised MLP (latent+3 -> hidden ReLU -> 3 sigmoid), biases zero."""
    n_sphere = n * 100 // 160
    n_helix = (n - n_sphere) // 2
    g = procedural_scene(seed, n_sphere, n_helix, n - n_sphere - n_helix, sh_degree=0)
    rng = np.random.default_rng(seed + 1)
    cams = []
    for _ in range(views):
        d = rng.standard_normal(3)
        d /= np.linalg.norm(d)
        cams.append(look_at(4.3 * d, [0.0, 0.0, 0.0], focal_for_vfov(size, 50.0),
                            focal_for_vfov(size, 50.0), size, size))
    latents = rng.standard_normal((latent_dim, g.n)).astype(np.float32)
    d_in = latent_dim + 3
    a1 = math.sqrt(6.0 / (d_in + hidden))
    a2 = math.sqrt(6.0 / (hidden + 3))
    W1 = rng.uniform(-a1, a1, (hidden, d_in)).astype(np.float32)
    W2 = rng.uniform(-a2, a2, (3, hidden)).astype(np.float32)
    b1 = np.zeros(hidden, np.float32)
    b2 = np.zeros(3, np.float32)
    return g, cams, dict(latents=latents, W1=W1, b1=b1, W2=W2, b2=b2)


def image_grad(cam: Camera, seed: int = 0) -> np.ndarray:
    """dL/dimage ~ N(0,1), [3,H,W] float32."""
    rng = np.random.default_rng(seed + 12345)
    return rng.standard_normal((3, cam.height, cam.width)).astype(np.float32)


def random_grads(n: int, rows: int, seed: int = 0, scale: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed + 777)
    return (scale * rng.standard_normal((rows, n))).astype(np.float32)
