"""Oracle: adaptive density control (test infrastructure; see the package header).

"Scaling 3D Gaussian Splatting with Distributed Compute": adaptive density control
clones, splits and prunes Gaussians every hundred steps (memory-wall section), from
2D position gradients accumulated over the steps (step walkthrough, "densify
locally"), starting at step 500 (trace section).  The thresholds and the split rule
are those of the 3DGS method the pages cite (Kerbl et al. 2023), with gsplat's
normalisation of the 2D gradient to NDC units:

  accumulate (every step, visible Gaussians):  acc += |(g_mx W / 2, g_my H / 2)|,  cnt += 1
  plan (every refinement):
    prune  if sigmoid(opacity) < prune_opa, or (optionally) max scale > prune_scale3d * extent
    else grow if acc / cnt > grow_grad2d:
      clone  if max scale <= grow_scale3d * extent   (the copy appended after the original)
      split  otherwise: two children at mu + R S xi_k (xi_k ~ N(0, I), inputs), scales / 1.6
    else keep
  opacity reset:  opacity <- min(opacity, 2 prune_opa), its Adam moments zeroed

Every decision is taken in fp32 against thresholds formed in fp64 and rounded once:
sigmoid(x) < p  <=>  x < ln(p / (1 - p));  max exp(s) <= t  <=>  max s <= ln t.
"""
from __future__ import annotations

import math

import numpy as np

PRUNE, KEEP, CLONE, SPLIT = 0, 1, 2, 3
N_PLANES = 59


def thresholds(grow_grad2d=2e-4, grow_scale3d=0.01, prune_opa=0.005, prune_scale3d=0.1, extent=1.0,
               split_shrink=1.6) -> dict:
    """The fp32 thresholds of the decisions (formed in fp64, rounded once)."""
    return {
        "grad": np.float32(grow_grad2d),
        "logit_prune": np.float32(math.log(prune_opa / (1.0 - prune_opa))),
        "log_grow_scale": np.float32(math.log(grow_scale3d * extent)),
        "log_prune_scale": np.float32(math.log(prune_scale3d * extent)),
        "log_shrink": np.float32(math.log(split_shrink)),
        "logit_reset": np.float32(math.log(2.0 * prune_opa / (1.0 - 2.0 * prune_opa))),
    }


def accumulate(grad2d_planes: np.ndarray, visible: np.ndarray, width: int, height: int, acc: np.ndarray,
               cnt: np.ndarray) -> None:
    """acc += the NDC-scaled norm of each visible Gaussian's 2D mean gradient (fp32);
    cnt += 1 for the visible.  grad2d_planes: (9, n) planes (0: d mx, 1: d my)."""
    gx = np.asarray(grad2d_planes[0], np.float32) * np.float32(0.5 * width)
    gy = np.asarray(grad2d_planes[1], np.float32) * np.float32(0.5 * height)
    norm = np.sqrt(gx * gx + gy * gy).astype(np.float32)
    vis = np.asarray(visible, bool)
    acc[vis] = (acc[vis] + norm[vis]).astype(np.float32)
    cnt[vis] += 1


def plan(params: np.ndarray, n: int, acc: np.ndarray, cnt: np.ndarray, th: dict, prune_big: bool = False):
    """Per Gaussian i < n: its action and the offset of its outputs (exclusive scan of
    0 / 1 / 2 outputs); and the new count."""
    P = np.asarray(params, np.float32)
    logit = P[10, :n]
    smax = P[3:6, :n].max(axis=0)
    avg = (np.asarray(acc[:n], np.float32) / np.maximum(np.asarray(cnt[:n]), 1).astype(np.float32)).astype(np.float32)
    prune = logit < th["logit_prune"]
    if prune_big:
        prune |= smax > th["log_prune_scale"]
    high = avg > th["grad"]
    small = smax <= th["log_grow_scale"]
    action = np.full(n, KEEP, np.uint8)
    action[high & small] = CLONE
    action[high & ~small] = SPLIT
    action[prune] = PRUNE
    outs = np.array([0, 1, 2, 2], np.int64)[action]
    offset = np.concatenate([[0], np.cumsum(outs)[:-1]]).astype(np.uint32) if n else np.zeros(0, np.uint32)
    return action, offset, int(outs.sum())


def _rotation(q: np.ndarray) -> np.ndarray:
    """Rotation matrices of normalised quaternions (w, x, y, z), shape (k, 3, 3), fp64."""
    q = q / np.linalg.norm(q, axis=1, keepdims=True)
    w, x, y, z = q.T
    return np.stack([
        np.stack([1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)], -1),
        np.stack([2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)], -1),
        np.stack([2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)], -1),
    ], 1)


def apply(params: np.ndarray, m: np.ndarray, v: np.ndarray, n: int, action: np.ndarray, offset: np.ndarray,
          n_out: int, randn: np.ndarray, th: dict, n_pad_out: int | None = None):
    """The new parameter and moment planes (59 x n_pad_out, padding zero).  A kept
    Gaussian and a clone's original keep their Adam moments; the copy of a clone and
    both children of a split start with zero moments.  randn: (n, 6) normals, the
    two children's xi.  Child means in fp64 from the fp32 inputs, rounded once."""
    if n_pad_out is None:
        n_pad_out = max(256, -(-n_out // 256) * 256)
    P = np.asarray(params, np.float32)
    out_p = np.zeros((N_PLANES, n_pad_out), np.float32)
    out_m = np.zeros_like(out_p)
    out_v = np.zeros_like(out_p)
    act = np.asarray(action[:n])
    off = np.asarray(offset[:n]).astype(np.int64)
    keep = (act == KEEP) | (act == CLONE)
    out_p[:, off[keep]] = P[:, :n][:, keep]
    out_m[:, off[keep]] = np.asarray(m, np.float32)[:, :n][:, keep]
    out_v[:, off[keep]] = np.asarray(v, np.float32)[:, :n][:, keep]
    cl = act == CLONE
    out_p[:, off[cl] + 1] = P[:, :n][:, cl]
    sp = np.nonzero(act == SPLIT)[0]
    if len(sp):
        mu = P[0:3, sp].T.astype(np.float64)
        scale = np.exp(P[3:6, sp].T.astype(np.float64))
        R = _rotation(P[6:10, sp].T.astype(np.float64))
        xi = np.asarray(randn, np.float32)[sp].astype(np.float64)
        for k in range(2):
            child = P[:, sp].copy()
            d = np.einsum("kij,kj->ki", R, scale * xi[:, 3 * k:3 * k + 3])
            child[0:3] = (mu + d).T.astype(np.float32)
            child[3:6] = (P[3:6, sp] - th["log_shrink"]).astype(np.float32)
            out_p[:, off[sp] + k] = child
    return out_p, out_m, out_v


def opacity_reset(params: np.ndarray, m: np.ndarray, v: np.ndarray, n: int, th: dict) -> None:
    """opacity <- min(opacity, 2 prune_opa) as a logit clamp; the opacity plane's Adam
    moments are zeroed (in place)."""
    params[10, :n] = np.minimum(params[10, :n], th["logit_reset"])
    m[10, :n] = 0.0
    v[10, :n] = 0.0
