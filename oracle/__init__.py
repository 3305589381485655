"""Plain CPU oracle for one 3D Gaussian Splatting optimisation step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``gaussian_splatting_differentiable_project_gb300``) never imports it and has no
CPU fallback; the two share no code, only the seeded inputs from ``gs_inputs``.

The arithmetic lives in ``gs_oracle.cpp`` (plain C++17, compiled with
``-O2 -ffp-contract=off``); this module compiles it on first use and wraps its
entry points for numpy arrays.  Each function names the step of the method it
follows ("3D Gaussian splatting for real-time radiance field rendering", the
method both pages name; the pages' own statement of the step is "Scaling 3D
Gaussian Splatting with Distributed Compute", sections on the representation, the
memory wall and the single-step walkthrough).

Parity status of every function is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants, library routines and finite differences.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gs_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

N_PLANES = 59
TILE = 16


def build(force: bool = False) -> str:
    """Compile ``gs_oracle.cpp`` into ``_build/liboracle.so`` (plain g++)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class OrCamera(ctypes.Structure):
    """Camera as the oracle reads it (declared independently of the product)."""
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3),
                ("fx", ctypes.c_float), ("fy", ctypes.c_float),
                ("cx", ctypes.c_float), ("cy", ctypes.c_float),
                ("width", ctypes.c_int32), ("height", ctypes.c_int32),
                ("campos", ctypes.c_float * 3), ("near_z", ctypes.c_float)]


def camera(cam: dict) -> OrCamera:
    c = OrCamera()
    c.R[:] = [float(v) for v in np.asarray(cam["R"], np.float32).reshape(9)]
    c.t[:] = [float(v) for v in np.asarray(cam["t"], np.float32).reshape(3)]
    c.fx, c.fy, c.cx, c.cy = (float(np.float32(cam[k])) for k in ("fx", "fy", "cx", "cy"))
    c.width, c.height = int(cam["width"]), int(cam["height"])
    c.campos[:] = [float(v) for v in np.asarray(cam["campos"], np.float32).reshape(3)]
    c.near_z = float(np.float32(cam.get("near_z", 0.01)))
    return c


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.or_set_threads.argtypes = [ctypes.c_int]
            lib.or_threads.restype = ctypes.c_int
            lib.or_expf.argtypes = [P, P, i64]
            lib.or_sh_basis.argtypes = [P, P, i64]
            for name in ("or_project_f32", "or_project_f64"):
                f = getattr(lib, name)
                f.argtypes = [P, i64, i64, ctypes.POINTER(OrCamera), P, P, P]
                f.restype = i64
            lib.or_tile_lists_f32.argtypes = [i64, P, P, ctypes.c_int, ctypes.c_int, P, P, P, i64]
            lib.or_tile_lists_f32.restype = i64
            for name in ("or_render_f32", "or_render_f64"):
                getattr(lib, name).argtypes = [i64, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P,
                                               ctypes.c_double, P, P]
            lib.or_project_bwd.argtypes = [P, i64, i64, ctypes.POINTER(OrCamera), ctypes.c_int, P, P]
            lib.or_ssim.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_double, P]
            lib.or_ssim.restype = ctypes.c_double
            lib.or_adam.argtypes = [P, P, P, P, ctypes.c_int, i64, P, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_double, i64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    _load().or_set_threads(int(n))


def threads() -> int:
    return int(_load().or_threads())


def expf(x) -> np.ndarray:
    """Single-precision exp used for every decision: Cody-Waite reduction plus a
    degree-7 Taylor polynomial, scaled by 2^k."""
    x = _c(x, np.float32)
    y = np.empty_like(x)
    _load().or_expf(_ptr(x), _ptr(y), x.size)
    return y


def sh_basis(dirs) -> np.ndarray:
    """Real SH basis (degree 3, Condon-Shortley phase) at unit directions, fp64."""
    d = _c(dirs, np.float64).reshape(-1, 3)
    Y = np.empty((d.shape[0], 16), np.float64)
    _load().or_sh_basis(_ptr(d), _ptr(Y), d.shape[0])
    return Y


def project(params: np.ndarray, n: int, cam: dict, prec: int = 32) -> dict:
    """Projection of every Gaussian: camera transform, Sigma = R S S^T R^T, EWA
    2D covariance (+0.3), conic, radius, tile rect and count, sigmoid opacity,
    degree-3 SH colour.  ``params`` is (59, n_pad) float32.  prec 32 takes the
    frozen fp32 sequence the kernels follow; prec 64 is the same algorithm in
    fp64 (for the pins)."""
    params = _c(params, np.float32)
    n_pad = params.shape[1]
    if params.shape[0] != N_PLANES or not 0 <= n <= n_pad:
        raise ValueError(f"project: params {params.shape} cannot hold {n} Gaussians")
    dt = np.float32 if prec == 32 else np.float64
    proj16 = np.zeros((n, 16), dt)
    iproj6 = np.zeros((n, 6), np.int32)
    flags = np.zeros(n, np.uint32)
    cam_c = camera(cam)
    f = _load().or_project_f32 if prec == 32 else _load().or_project_f64
    bad = f(_ptr(params), n, n_pad, ctypes.byref(cam_c), _ptr(proj16), _ptr(iproj6), _ptr(flags))
    return {
        "proj16": proj16, "iproj6": iproj6, "flags": flags, "nonfinite": int(bad),
        "mean2d": proj16[:, 0:2], "conic": proj16[:, 2:5], "opacity": proj16[:, 5],
        "rgb": proj16[:, 6:9], "depth": proj16[:, 9], "cov2d": proj16[:, 10:13],
        "radius": iproj6[:, 0], "rect": iproj6[:, 1:5], "count": iproj6[:, 5].astype(np.uint32),
        "visible": (flags & 1).astype(bool),
    }


def tile_lists(proj: dict, width: int, height: int, cap: int | None = None) -> dict:
    """Per tile, the ordered subsequence of the global (depth, index) order whose
    rect contains the tile, as (tile << 32 | depth bits) keys, ids and ranges."""
    n = proj["proj16"].shape[0]
    TX, TY = -(-width // TILE), -(-height // TILE)
    if cap is None:
        cap = int(proj["count"].astype(np.int64).sum())
    keys = np.zeros(max(cap, 1), np.uint64)
    ids = np.zeros(max(cap, 1), np.uint32)
    ranges = np.zeros((TX * TY, 2), np.uint32)
    K = _load().or_tile_lists_f32(n, _ptr(_c(proj["proj16"], np.float32)), _ptr(proj["iproj6"]),
                                  width, height, _ptr(keys), _ptr(ids), _ptr(ranges), cap)
    return {"K": int(K), "keys": keys[:min(K, cap)], "ids": ids[:min(K, cap)], "ranges": ranges}


def render(proj: dict, width: int, height: int, bg=(0.0, 0.0, 0.0), target=None, prec: int = 32,
           l1_weight: float = 1.0, dLdC_extra=None, count_used: bool = False) -> dict:
    """Front-to-back compositing of every pixel over its tile's list; with a
    target, also the loss l1_weight * mean |C - C*| (over 3 P values) and the
    per-Gaussian 2D gradients (9 x n fp64: d mx, d my, d A, d B, d C, d o, d r, d g,
    d b) from the suffix-sum backward, with dLdC_extra (3 x H x W fp64) added to the
    loss gradient if given.  With count_used, also each pixel's number of composited
    entries (alpha >= 1/255, before the transmittance stop) as "n_used"."""
    n = proj["proj16"].shape[0]
    dt = np.float32 if prec == 32 else np.float64
    image = np.zeros((3, height, width), dt)
    T_final = np.zeros((height, width), dt)
    n_contrib = np.zeros((height, width), np.uint32)
    bg_a = np.asarray(bg, dt)
    grad2d = loss = None
    tgt = None
    if target is not None:
        tgt = _c(target, dt).reshape(3, height, width)
        grad2d = np.zeros((9, n), np.float64)
        loss = np.zeros(1, np.float64)
    f = _load().or_render_f32 if prec == 32 else _load().or_render_f64
    extra = None if dLdC_extra is None else _c(dLdC_extra, np.float64).reshape(3, height, width)
    n_used = np.zeros((height, width), np.uint32) if count_used else None
    f(n, _ptr(_c(proj["proj16"], dt)), _ptr(proj["iproj6"]), width, height, _ptr(bg_a), _ptr(tgt),
      _ptr(image), _ptr(T_final), _ptr(n_contrib), _ptr(grad2d), _ptr(loss), float(l1_weight), _ptr(extra),
      _ptr(n_used))
    out = {"image": image, "T_final": T_final, "n_contrib": n_contrib}
    if count_used:
        out["n_used"] = n_used
    if target is not None:
        out["grad2d"] = grad2d
        out["loss"] = float(loss[0])
    return out


def project_bwd(params: np.ndarray, n: int, cam: dict, grad2d: np.ndarray, prec: int = 32) -> np.ndarray:
    """Chain rule from the nine 2D gradients to the 59 parameter gradients (fp64);
    decisions (culling, clamps) are taken in precision ``prec``."""
    params = _c(params, np.float32)
    if params.shape[0] != N_PLANES or not 0 <= n <= params.shape[1]:
        raise ValueError(f"project_bwd: params {params.shape} cannot hold {n} Gaussians")
    g2 = _c(grad2d, np.float64).reshape(9, n)
    grads = np.zeros((N_PLANES, n), np.float64)
    cam_c = camera(cam)
    _load().or_project_bwd(_ptr(params), n, params.shape[1], ctypes.byref(cam_c), int(prec),
                           _ptr(g2), _ptr(grads))
    return grads


def ssim(x, y, lam: float = 1.0):
    """Mean SSIM of x against y (3 x H x W; 11x11 Gaussian window, sigma 1.5, C1 =
    0.01^2, C2 = 0.03^2, zero padding) and the gradient of lam (1 - SSIM) with
    respect to x, in fp64."""
    x = _c(x, np.float64)
    y = _c(y, np.float64)
    C, H, W = x.shape
    assert C == 3 and y.shape == x.shape
    g = np.zeros_like(x)
    val = _load().or_ssim(W, H, _ptr(x), _ptr(y), float(lam), _ptr(g))
    return float(val), g


def adam(p, g, m, v, lr_plane, beta1: float, beta2: float, eps: float, t: int):
    """Textbook Adam in fp64 on (planes, stride) arrays; returns (p, m, v)."""
    p = np.array(p, np.float64, copy=True)
    m = np.array(m, np.float64, copy=True)
    v = np.array(v, np.float64, copy=True)
    g = _c(g, np.float64)
    planes, stride = p.shape
    lr = _c(lr_plane, np.float64)
    _load().or_adam(_ptr(p), _ptr(g), _ptr(m), _ptr(v), planes, stride, _ptr(lr), beta1, beta2, eps, int(t))
    return p, m, v


def batch_hyper(batch: int, lr_plane, beta1: float, beta2: float, eps: float):
    """Adam hyperparameters for a step over ``batch`` views ("Scaling 3D Gaussian
    Splatting with Distributed Compute", batch-size section): learning rates times
    sqrt(batch), epsilon divided by sqrt(batch), and each momentum coefficient by the
    linearisation 1 - batch (1 - beta) of beta^batch (the page's formula did not
    survive; this reading makes beta1 = 0.9 reach zero at batch 10, as the page
    states), clamped at zero beyond that."""
    s = math.sqrt(batch)
    lr = np.asarray(lr_plane, np.float64) * s
    return lr, max(0.0, 1.0 - batch * (1.0 - beta1)), max(0.0, 1.0 - batch * (1.0 - beta2)), eps / s


def step_batch(params, n: int, cams, targets, m, v, t: int, lr_plane, beta1=0.9, beta2=0.999, eps=1e-15,
               bg=(0.0, 0.0, 0.0), dssim: float = 0.0) -> dict:
    """One optimisation step over several views: the loss is the mean of the per-view
    losses, so each view's loss gradient carries 1 / batch; the per-view parameter
    gradients are summed and one Adam step with ``batch_hyper`` follows."""
    B = len(cams)
    assert B >= 1 and len(targets) == B
    n_pad = params.shape[1]
    grads = np.zeros((N_PLANES, n_pad), np.float64)
    loss = 0.0
    views = []
    for cam, target in zip(cams, targets):
        pr = project(params, n, cam, 32)
        W, H = int(cam["width"]), int(cam["height"])
        if dssim > 0.0:
            img = render(pr, W, H, bg, None, 32)["image"]
            s_val, extra = ssim(img.astype(np.float64), np.asarray(target, np.float64), dssim / B)
            rd = render(pr, W, H, bg, target, 32, l1_weight=(1.0 - dssim) / B, dLdC_extra=extra)
            rd["ssim"] = s_val
            rd["loss"] += dssim * (1.0 - s_val) / B
        else:
            rd = render(pr, W, H, bg, target, 32, l1_weight=1.0 / B)
        grads[:, :n] += project_bwd(params, n, cam, rd["grad2d"], 32)
        loss += rd["loss"]
        views.append({"proj": pr, "render": rd})
    lr_b, b1, b2, eps_b = batch_hyper(B, lr_plane, beta1, beta2, eps)
    p1, m1, v1 = adam(params.astype(np.float64), grads, m, v, lr_b, b1, b2, eps_b, t)
    return {"views": views, "grads": grads, "loss": loss, "params": p1, "m": m1, "v": v1,
            "hyper": (lr_b, b1, b2, eps_b)}


def step(params, n: int, cam: dict, target, m, v, t: int, lr_plane, beta1=0.9, beta2=0.999, eps=1e-15,
         bg=(0.0, 0.0, 0.0), dssim: float = 0.0) -> dict:
    """One whole optimisation step for one view, stage by stage; with dssim = lambda
    > 0 the loss is (1 - lambda) L1 + lambda (1 - SSIM)."""
    pr = project(params, n, cam, 32)
    W, H = int(cam["width"]), int(cam["height"])
    if dssim > 0.0:
        img = render(pr, W, H, bg, None, 32)["image"]
        s_val, extra = ssim(img.astype(np.float64), np.asarray(target, np.float64), dssim)
        rd = render(pr, W, H, bg, target, 32, l1_weight=1.0 - dssim, dLdC_extra=extra)
        rd["ssim"] = s_val
        rd["loss"] += dssim * (1.0 - s_val)
    else:
        rd = render(pr, W, H, bg, target, 32)
    grads = project_bwd(params, n, cam, rd["grad2d"], 32)
    n_pad = params.shape[1]
    gfull = np.zeros((N_PLANES, n_pad), np.float64)
    gfull[:, :n] = grads
    p1, m1, v1 = adam(params.astype(np.float64), gfull, m, v, lr_plane, beta1, beta2, eps, t)
    return {"proj": pr, "render": rd, "grads": gfull, "params": p1, "m": m1, "v": v1}


from . import densify  # noqa: E402,F401  (adaptive density control)
