"""Seeded synthetic inputs shared by the CUDA path's tests and bench and by the oracle.

This module holds none of the method's arithmetic (no projection, compositing,
gradient or optimiser step): it only draws parameters, builds cameras and packs
them into the parameter-plane layout.  The scenes stand in for the pages'
Kingsnake (~4M points) and Miranda (~18M points) isosurface point clouds and their
448-view structured orbit ("Toward Distributed 3D Gaussian Splatting for
High-Resolution Isosurface Visualization", sections III and IV), which are not
available here.

Parameter layout (59 fp32 planes of stride n_pad, the 59 learnable values per
Gaussian at SH degree 3 of "Scaling 3D Gaussian Splatting with Distributed
Compute", memory-wall section):
    0-2   mean mu
    3-5   log-scale
    6-9   quaternion (w, x, y, z)
    10    opacity logit
    11-58 SH coefficient k of channel ch at plane 11 + 3 k + ch (k < 16)
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

N_PLANES = 59
PLANE_MEAN, PLANE_LOGSCALE, PLANE_QUAT, PLANE_LOGIT, PLANE_SH = 0, 3, 6, 10, 11
PAD = 256

# Per-plane Adam learning rates.  The pages state none; these are the published
# defaults of the 3DGS method the pages build on (positions scaled by a scene
# extent of 3.3 for a camera orbit of radius 3).
LR_MEAN = 1.6e-4 * 3.3
LR_SH_DC = 2.5e-3
LR_SH_REST = 2.5e-3 / 20.0
LR_OPACITY = 0.05
LR_SCALE = 5e-3
LR_QUAT = 1e-3
BETA1, BETA2, EPS = 0.9, 0.999, 1e-15


def lr_planes() -> np.ndarray:
    lr = np.empty(N_PLANES, np.float64)
    lr[0:3] = LR_MEAN
    lr[3:6] = LR_SCALE
    lr[6:10] = LR_QUAT
    lr[10] = LR_OPACITY
    lr[11:14] = LR_SH_DC
    lr[14:59] = LR_SH_REST
    return lr


def n_pad_of(n: int) -> int:
    return max(PAD, -(-n // PAD) * PAD)


# ----------------------------------------------------------------------------- cameras

def look_at(eye, target=(0.0, 0.0, 0.0), up=(0.0, 0.0, 1.0)) -> tuple[np.ndarray, np.ndarray]:
    """World->camera rotation (rows: right, down, forward; OpenCV axes) and
    translation for a camera at ``eye`` looking at ``target``."""
    eye = np.asarray(eye, np.float64)
    f = np.asarray(target, np.float64) - eye
    f /= np.linalg.norm(f)
    up = np.asarray(up, np.float64)
    if np.linalg.norm(np.cross(f, up)) < 1e-6:
        up = np.array([0.0, 1.0, 0.0]) if abs(f[1]) < 0.9 else np.array([1.0, 0.0, 0.0])
    right = np.cross(f, up)
    right /= np.linalg.norm(right)
    down = np.cross(f, right)
    R = np.stack([right, down, f])
    t = -R @ eye
    return R, t


def camera(eye, width: int, height: int, fov_deg: float = 50.0, target=(0.0, 0.0, 0.0),
           near_z: float = 0.01) -> dict:
    """Pinhole camera dict (fp32 values): principal point at the image centre,
    square pixels, horizontal field of view ``fov_deg``."""
    R, t = look_at(eye, target)
    f = (width / 2.0) / math.tan(math.radians(fov_deg) / 2.0)
    return {
        "R": R.astype(np.float32), "t": t.astype(np.float32),
        "fx": np.float32(f), "fy": np.float32(f),
        "cx": np.float32(width / 2.0), "cy": np.float32(height / 2.0),
        "width": int(width), "height": int(height),
        "campos": np.asarray(eye, np.float32), "near_z": np.float32(near_z),
    }


def fibonacci_cameras(n_views: int, width: int, height: int, radius: float = 3.0,
                      fov_deg: float = 50.0) -> list[dict]:
    """``n_views`` cameras on a Fibonacci sphere of ``radius`` looking at the
    origin: z_i = 1 - (2i+1)/n, azimuth i * pi (3 - sqrt 5)."""
    cams = []
    ga = math.pi * (3.0 - math.sqrt(5.0))
    for i in range(n_views):
        z = 1.0 - (2.0 * i + 1.0) / n_views
        r = math.sqrt(max(0.0, 1.0 - z * z))
        phi = i * ga
        eye = radius * np.array([r * math.cos(phi), r * math.sin(phi), z])
        cams.append(camera(eye, width, height, fov_deg))
    return cams


# ----------------------------------------------------------------------------- scenes

def pack(means, log_scales, quats, logits, sh, n_pad: int | None = None) -> np.ndarray:
    """Pack per-Gaussian arrays into (59, n_pad) fp32 planes; padding is zero."""
    n = means.shape[0]
    n_pad = n_pad or n_pad_of(n)
    P = np.zeros((N_PLANES, n_pad), np.float32)
    P[0:3, :n] = means.T
    P[3:6, :n] = log_scales.T
    P[6:10, :n] = quats.T
    P[10, :n] = logits
    P[11:59, :n] = sh.reshape(n, 48).T   # sh is (n, 16, 3) -> plane 11 + 3k + ch
    return P


def _sh_init(rng: np.random.Generator, n: int) -> np.ndarray:
    sh = np.empty((n, 16, 3), np.float64)
    sh[:, 0, :] = rng.uniform(-1.0, 1.0, (n, 3))
    sh[:, 1:, :] = rng.normal(0.0, 0.05, (n, 15, 3))
    return sh


def random_cube_scene(seed: int, n: int, n_pad: int | None = None) -> np.ndarray:
    """Tiny correctness scene: means U[-1,1]^3, log-scales N(-3.5, 0.3^2), quaternions
    normalised N(0, I4), opacity logits N(0,1), SH DC U(-1,1), higher bands N(0, 0.05^2)."""
    rng = np.random.default_rng(seed)
    means = rng.uniform(-1.0, 1.0, (n, 3))
    log_scales = rng.normal(-3.5, 0.3, (n, 3))
    q = rng.normal(0.0, 1.0, (n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    logits = rng.normal(0.0, 1.0, n)
    sh = _sh_init(rng, n)
    return pack(means, log_scales, q, logits, sh, n_pad)


@dataclass
class BlobField:
    """f(x) = sum_j exp(-|x - c_j|^2 / (2 s_j^2)) - 0.5 over 32 random blobs."""
    centres: np.ndarray
    sigmas: np.ndarray

    @staticmethod
    def make(seed: int, n_blobs: int = 32) -> "BlobField":
        rng = np.random.default_rng(seed)
        return BlobField(rng.uniform(-0.6, 0.6, (n_blobs, 3)), rng.uniform(0.15, 0.35, n_blobs))

    def value_grad(self, x: np.ndarray):
        f = np.full(x.shape[0], -0.5)
        g = np.zeros_like(x)
        for c, s in zip(self.centres, self.sigmas):
            d = x - c
            e = np.exp(-np.einsum("ij,ij->i", d, d) / (2.0 * s * s))
            f += e
            g -= (e / (s * s))[:, None] * d
        return f, g

    def value_grad_torch(self, x):
        import torch
        c = torch.as_tensor(self.centres, dtype=x.dtype, device=x.device)     # (B, 3)
        s2 = torch.as_tensor(self.sigmas, dtype=x.dtype, device=x.device) ** 2  # (B,)
        d = x[:, None, :] - c[None]                                              # (n, B, 3)
        e = torch.exp(-(d * d).sum(-1) / (2.0 * s2))                              # (n, B)
        f = e.sum(1) - 0.5
        g = -((e / s2)[:, :, None] * d).sum(1)
        return f, g


@dataclass
class TurbulenceField:
    """f(x) = sum_j a_j sin(2 pi nu_j u_j . x + phi_j) over 256 random-phase
    sinusoids, nu_j in [1, 16], a_j = 1/nu_j, u_j uniform on the sphere."""
    u: np.ndarray
    nu: np.ndarray
    phase: np.ndarray

    @staticmethod
    def make(seed: int, n_terms: int = 256) -> "TurbulenceField":
        rng = np.random.default_rng(seed)
        u = rng.normal(0.0, 1.0, (n_terms, 3))
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        return TurbulenceField(u, rng.uniform(1.0, 16.0, n_terms), rng.uniform(0.0, 2 * math.pi, n_terms))

    def value_grad(self, x: np.ndarray):
        k = 2.0 * math.pi * self.nu[:, None] * self.u          # (T, 3)
        arg = x @ k.T + self.phase                              # (n, T)
        a = 1.0 / self.nu
        f = np.sin(arg) @ a
        g = (np.cos(arg) * a) @ k
        return f, g

    def value_grad_torch(self, x):
        import torch
        k = torch.as_tensor(2.0 * math.pi * self.nu[:, None] * self.u, dtype=x.dtype, device=x.device)
        ph = torch.as_tensor(self.phase, dtype=x.dtype, device=x.device)
        a = torch.as_tensor(1.0 / self.nu, dtype=x.dtype, device=x.device)
        arg = x @ k.T + ph
        return torch.sin(arg) @ a, (torch.cos(arg) * a) @ k


def sample_level_set(field, n: int, rng: np.random.Generator, jitter: float = 0.002,
                     newton_steps: int = 8, tol: float = 1e-5, chunk: int = 1 << 18, device=None) -> np.ndarray:
    """Points on the zero level set: uniform candidates in [-1,1]^3, Newton steps
    x <- x - f grad f / |grad f|^2, keep |f| < tol inside the cube, then jitter.
    The candidates and jitter come from ``rng``; with ``device`` (a torch device)
    the Newton iterations run in torch fp64 there instead of numpy."""
    out, have = [], 0
    while have < n:
        x = rng.uniform(-1.0, 1.0, (chunk, 3))
        if device is None:
            for _ in range(newton_steps):
                f, g = field.value_grad(x)
                gg = np.einsum("ij,ij->i", g, g)
                x = x - (f / np.maximum(gg, 1e-30))[:, None] * g
            f, _ = field.value_grad(x)
        else:
            import torch
            xt = torch.as_tensor(x, dtype=torch.float64, device=device)
            for _ in range(newton_steps):
                f, g = field.value_grad_torch(xt)
                gg = (g * g).sum(1)
                xt = xt - (f / torch.clamp(gg, min=1e-30))[:, None] * g
            f, _ = field.value_grad_torch(xt)
            x, f = xt.cpu().numpy(), f.cpu().numpy()
        ok = (np.abs(f) < tol) & np.all(np.abs(x) <= 1.0, axis=1)
        x = x[ok]
        out.append(x)
        have += x.shape[0]
    pts = np.concatenate(out)[:n]
    return pts + rng.normal(0.0, jitter, pts.shape)


def knn_log_scale(points: np.ndarray, k: int = 3) -> np.ndarray:
    """log of the mean Euclidean distance to the k nearest other points (floor 1e-7)."""
    from scipy.spatial import cKDTree
    tree = cKDTree(points)
    d, _ = tree.query(points, k=k + 1, workers=-1)
    mean = d[:, 1:].mean(axis=1)
    return np.log(np.maximum(mean, 1e-7))


def isosurface_scene(field_seed: int, sample_seed: int, n: int, kind: str = "blobs",
                     n_pad: int | None = None, device=None) -> np.ndarray:
    """Isosurface scene: means on the level set of the seeded field, kNN log-scales
    on all three axes, quaternions identity + N(0, 0.1^2) normalised, opacity
    logits 0.1 N(0,1), SH DC U(-1,1) and higher bands N(0, 0.05^2)."""
    field = BlobField.make(field_seed) if kind == "blobs" else TurbulenceField.make(field_seed)
    rng = np.random.default_rng(sample_seed)
    if device is None:
        chunk = 1 << 18 if kind == "blobs" else 1 << 15
    else:
        chunk = 1 << 21 if kind == "blobs" else 1 << 18
    means = sample_level_set(field, n, rng, chunk=chunk, device=device)
    ls = knn_log_scale(means)
    log_scales = np.repeat(ls[:, None], 3, axis=1)
    q = np.zeros((n, 4))
    q[:, 0] = 1.0
    q += rng.normal(0.0, 0.1, (n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    logits = 0.1 * rng.normal(0.0, 1.0, n)
    sh = _sh_init(rng, n)
    return pack(means, log_scales, q, logits, sh, n_pad)


# ----------------------------------------------------------------------------- configs

@dataclass
class Config:
    name: str
    n: int
    width: int
    height: int
    n_views: int
    kind: str          # "cube", "blobs" or "turbulence"
    description: str


CONFIGS = {
    "tiny": Config("tiny", 4096, 128, 128, 1, "cube",
                   "4,096 Gaussians in [-1,1]^3, one 128x128 camera at distance 3"),
    "iso1m_512": Config("iso1m_512", 1_000_000, 512, 512, 64, "blobs",
                        "1M-Gaussian blob isosurface, 512x512, 64 orbit views"),
    "iso4m_1024": Config("iso4m_1024", 4_000_000, 1024, 1024, 448, "blobs",
                         "4M-Gaussian blob isosurface, 1024x1024, 448 orbit views"),
    "iso4m_2048": Config("iso4m_2048", 4_000_000, 2048, 2048, 448, "blobs",
                         "4M-Gaussian blob isosurface, 2048x2048, 448 orbit views"),
    "turb18m_2048": Config("turb18m_2048", 18_000_000, 2048, 2048, 448, "turbulence",
                           "18M-Gaussian turbulence isosurface, 2048x2048, 448 orbit views"),
}


def cameras_for(cfg: Config) -> list[dict]:
    if cfg.kind == "cube":
        return [camera((0.0, 0.0, 3.0), cfg.width, cfg.height)]
    return fibonacci_cameras(cfg.n_views, cfg.width, cfg.height)


def scene_for(cfg: Config, seed: int = 0, n: int | None = None, device=None) -> np.ndarray:
    """Model parameters for a config (``n`` overrides the Gaussian count for
    reduced-size parity cases of the same generator; ``device`` runs the level-set
    Newton iterations in torch on that device)."""
    n = cfg.n if n is None else n
    if cfg.kind == "cube":
        return random_cube_scene(seed, n)
    return isosurface_scene(seed, 1000 + seed, n, cfg.kind, device=device)


def target_scene_for(cfg: Config, seed: int = 0, n: int | None = None, device=None) -> np.ndarray:
    """The second seeded Gaussian set whose renders are the targets: for the
    isosurface configs the same surface sampled with another seed."""
    n = cfg.n if n is None else n
    if cfg.kind == "cube":
        return random_cube_scene(seed + 1, n)
    return isosurface_scene(seed, 2000 + seed, n, cfg.kind, device=device)


def offset_target(image: np.ndarray, seed: int, lo: float = 0.05, hi: float = 0.15) -> np.ndarray:
    """A target that differs from ``image`` by a seeded offset of magnitude in
    [lo, hi] with random sign in every value, so that the sign of every L1
    residual is far from a tie."""
    rng = np.random.default_rng(seed)
    mag = rng.uniform(lo, hi, image.shape)
    sgn = np.where(rng.random(image.shape) < 0.5, -1.0, 1.0)
    return (image + sgn * mag).astype(image.dtype)


def uniform_target(seed: int, width: int, height: int) -> np.ndarray:
    """A seeded target image (3, height, width) fp32, U(0, 1) in every value: an L1
    target that depends on no render, for checks where both sides render the same
    image bit for bit (so they take every residual sign alike)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(0.0, 1.0, (3, height, width)).astype(np.float32)


def random_grad2d(seed: int, n: int, n_pad: int, scale: float = 1e-3) -> np.ndarray:
    """Seeded stand-in for the nine per-Gaussian 2D gradients (9, n_pad) fp32."""
    rng = np.random.default_rng(seed)
    g = np.zeros((9, n_pad), np.float32)
    g[:, :n] = rng.normal(0.0, scale, (9, n))
    return g
