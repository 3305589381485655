"""Pins of the CPU oracle against things other than itself: closed forms, invariants,
library routines, brute force and finite differences.  CPU only.

Each test names what fixes the expected value.  A plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest

import gs_inputs as gi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers

def _ulp_err(y32: np.ndarray, ref: np.ndarray) -> np.ndarray:
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return np.abs(y32.astype(np.float64) - ref) / ulp


def _cam(W=32, H=32, eye=(0.0, 0.0, 3.0)):
    return gi.camera(eye, W, H)


def _scene(means, log_scale, quats=None, logits=None, sh=None):
    means = np.asarray(means, np.float64).reshape(-1, 3)
    n = means.shape[0]
    ls = np.broadcast_to(np.asarray(log_scale, np.float64), (n, 3)) if np.ndim(log_scale) < 2 else log_scale
    if quats is None:
        quats = np.tile([1.0, 0.0, 0.0, 0.0], (n, 1))
    if logits is None:
        logits = np.zeros(n)
    if sh is None:
        sh = np.zeros((n, 16, 3))
    return gi.pack(means, np.array(ls), np.asarray(quats), np.asarray(logits), np.asarray(sh)), n


# ----------------------------------------------------------------------------- layout

def test_layout_matches_pages():
    """59 parameters per Gaussian at SH degree 3 (16 per channel, 192 B), 708 B with
    two Adam moments, 12-scalar / 48-B projected record: the pages' numbers."""
    g = json.load(open(os.path.join(GOLDEN, "pages_layout.json")))
    assert gi.N_PLANES == g["params_per_gaussian_sh3"]["value"] == oracle.N_PLANES
    sh_planes = gi.N_PLANES - gi.PLANE_SH
    assert sh_planes == 3 * g["sh_coeffs_per_channel_sh3"]["value"]
    assert sh_planes * 4 == g["sh_bytes_sh3"]["value"]
    # SH degree 2 would keep 9 coefficients per channel: 59 - 3 * (16 - 9) = 38
    assert gi.N_PLANES - 3 * (16 - g["sh_coeffs_per_channel_sh2"]["value"]) == g["params_per_gaussian_sh2"]["value"]
    assert gi.N_PLANES * 4 * 3 == g["bytes_per_gaussian_with_adam_sh3"]["value"]
    assert g["record_scalars"]["value"] * 4 == g["record_bytes"]["value"] == 48
    assert 3 * 4 == g["rgb_bytes"]["value"]


# ----------------------------------------------------------------------------- exp

def test_expf_within_two_ulp_of_fp64():
    """The decision exponential stays within 2 ulp of the correctly rounded fp64 exp
    across its whole domain, and within 1 ulp here (a wrong polynomial coefficient or
    reduction constant breaks this).  The samples include the reduction's corners:
    arguments within a few ulps of (j + 1/2) ln2, where the nearest integer k flips and
    |r| reaches ln2/2, for every j whose result is normal."""
    half = np.concatenate([(np.arange(-125, 127) + 0.5) * math.log(2.0)])
    half = half[(half > -87.0) & (half < 88.0)].astype(np.float32)
    corners = np.concatenate([np.nextafter(half, np.float32(np.inf) * np.sign(d)) if d else half
                              for d in (-1, 0, 1)] +
                             [(half.view(np.int32) + d).view(np.float32) for d in (-3, -2, 2, 3)])
    x = np.concatenate([np.linspace(-87.0, 88.0, 400_001, dtype=np.float32),
                        np.random.default_rng(0).uniform(-6.0, 0.0, 200_000).astype(np.float32),
                        corners.astype(np.float32)])
    x = x[(x >= -87.0) & (x <= 88.0)]
    y = oracle.expf(x)
    err = _ulp_err(y, np.exp(x.astype(np.float64)))
    assert err.max() <= 1.0, err.max()
    assert np.mean(err <= 0.5) > 0.9


def test_expf_special_values():
    x = np.array([0.0, -0.0, np.nan, 100.0, -100.0, 88.0, -87.0, 1.0], np.float32)
    y = oracle.expf(x)
    assert y[0] == 1.0 and y[1] == 1.0
    assert np.isnan(y[2])
    assert y[3] == np.inf and y[4] == 0.0
    assert np.isfinite(y[5]) and y[6] > np.finfo(np.float32).tiny
    assert abs(float(y[7]) - math.e) <= np.spacing(np.float32(math.e))


# ----------------------------------------------------------------------------- SH

def _random_dirs(n, seed=0):
    d = np.random.default_rng(seed).normal(size=(n, 3))
    return d / np.linalg.norm(d, axis=1, keepdims=True)


def test_sh_addition_theorem():
    """sum_m Y_lm(d)^2 = (2l+1)/(4 pi) for every unit d and each band l."""
    Y = oracle.sh_basis(_random_dirs(1000))
    for l in range(4):
        s = (Y[:, l * l:(l + 1) * (l + 1)] ** 2).sum(axis=1)
        np.testing.assert_allclose(s, (2 * l + 1) / (4 * math.pi), rtol=1e-12)


def test_sh_orthonormal_by_quadrature():
    """Gauss-Legendre in cos(theta) x uniform azimuth integrates products of degree
    <= 6 exactly: the Gram matrix of the 16 basis functions is the identity."""
    mu, w = np.polynomial.legendre.leggauss(8)
    n_phi = 16
    phi = 2 * math.pi * np.arange(n_phi) / n_phi
    M, P = np.meshgrid(mu, phi, indexing="ij")
    S = np.sqrt(1 - M ** 2)
    dirs = np.stack([S * np.cos(P), S * np.sin(P), M], axis=-1).reshape(-1, 3)
    wt = (w[:, None] * np.full(n_phi, 2 * math.pi / n_phi)[None, :]).reshape(-1)
    Y = oracle.sh_basis(dirs)
    G = (Y * wt[:, None]).T @ Y
    np.testing.assert_allclose(G, np.eye(16), atol=1e-12)


def test_sh_matches_scipy_complex_harmonics():
    """Real SH with the Condon-Shortley phase from scipy's complex harmonics:
    sqrt(2) Re Y_l^m (m > 0), sqrt(2) Im Y_l^|m| (m < 0), Y_l^0 (m = 0)."""
    special = pytest.importorskip("scipy.special")
    if not hasattr(special, "sph_harm_y"):
        pytest.skip("scipy without sph_harm_y")
    d = _random_dirs(500, seed=3)
    theta = np.arccos(np.clip(d[:, 2], -1, 1))
    phi = np.arctan2(d[:, 1], d[:, 0])
    Y = oracle.sh_basis(d)
    for l in range(4):
        for m in range(-l, l + 1):
            c = special.sph_harm_y(l, abs(m), theta, phi)
            ref = c.real if m == 0 else (math.sqrt(2) * (c.real if m > 0 else c.imag))
            np.testing.assert_allclose(Y[:, l * l + l + m], ref, atol=1e-12, err_msg=f"l={l} m={m}")
    # explicit l = 1 sign convention: (-y, z, -x) sqrt(3 / 4 pi)
    k1 = math.sqrt(3 / (4 * math.pi))
    np.testing.assert_allclose(Y[:, 1:4], np.stack([-k1 * d[:, 1], k1 * d[:, 2], -k1 * d[:, 0]], 1), atol=1e-14)


# ----------------------------------------------------------------------------- projection

@pytest.mark.parametrize("prec", [64, 32])
def test_projection_isotropic_on_axis_closed_form(prec):
    """An isotropic Gaussian of scale s on the optical axis at depth z projects to
    Sigma_2 = (f s / z)^2 I + 0.3 I, conic I / that, mean at the principal point,
    radius ceil(3 sqrt(lambda)) with lambda = diag + sqrt(0.1) (the discriminant is
    0 and takes the 0.1 floor), opacity sigmoid(logit)."""
    W = H = 64
    cam = _cam(W, H)
    sig = np.array([0.05, 0.1, 0.2])
    logits = np.array([0.3, -1.0, 2.0])
    P, n = _scene(np.zeros((3, 3)), np.log(sig)[:, None].repeat(3, 1), logits=logits)
    pr = oracle.project(P, n, cam, prec)
    f = float(cam["fx"])
    sig = np.exp(P[3, :n].astype(np.float64))      # the scale the fp32 planes hold
    logits = P[10, :n].astype(np.float64)
    s2 = (f * sig / 3.0) ** 2 + 0.3
    tol = dict(rtol=1e-12) if prec == 64 else dict(rtol=2e-6)
    np.testing.assert_allclose(pr["cov2d"][:, 0], s2, **tol)
    np.testing.assert_allclose(pr["cov2d"][:, 2], s2, **tol)
    np.testing.assert_allclose(pr["cov2d"][:, 1], 0.0, atol=1e-12 if prec == 64 else 1e-6)
    np.testing.assert_allclose(pr["conic"][:, 0], 1 / s2, **tol)
    np.testing.assert_allclose(pr["conic"][:, 2], 1 / s2, **tol)
    np.testing.assert_allclose(pr["mean2d"], np.full((3, 2), W / 2), rtol=1e-7)
    np.testing.assert_allclose(pr["depth"], 3.0, rtol=1e-7)
    np.testing.assert_allclose(pr["opacity"], 1 / (1 + np.exp(-logits)), rtol=1e-12 if prec == 64 else 1e-6)
    np.testing.assert_array_equal(pr["radius"], np.ceil(3 * np.sqrt(s2 + math.sqrt(0.1))).astype(int))


def test_projection_ewa_matches_finite_difference_of_perspective():
    """The 2D covariance minus the 0.3 low-pass equals sum_j d_j d_j^T where d_j is
    the central difference of the exact pinhole map along the j-th scaled principal
    axis (rotation from scipy): the EWA linearisation, fixed independently."""
    Rot = pytest.importorskip("scipy.spatial.transform").Rotation
    rng = np.random.default_rng(5)
    n = 12
    means = rng.uniform(-0.5, 0.5, (n, 3))
    ls = rng.normal(-3.0, 0.4, (n, 3))
    q = rng.normal(size=(n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    P, _ = _scene(means, ls, quats=q)
    # the values the fp32 planes hold
    means = P[0:3, :n].T.astype(np.float64)
    ls = P[3:6, :n].T.astype(np.float64)
    q = P[6:10, :n].T.astype(np.float64)
    cam = gi.camera((2.0, -1.5, 1.8), 256, 192)
    pr = oracle.project(P, n, cam, 64)
    R = cam["R"].astype(np.float64)
    t = cam["t"].astype(np.float64)
    fx, fy, cx, cy = (float(cam[k]) for k in ("fx", "fy", "cx", "cy"))

    def pinhole(x):
        c = R @ x + t
        return np.array([fx * c[0] / c[2] + cx, fy * c[1] / c[2] + cy])

    for i in range(n):
        # scipy quaternions are (x, y, z, w)
        rot = Rot.from_quat([q[i, 1], q[i, 2], q[i, 3], q[i, 0]]).as_matrix()
        L = rot @ np.diag(np.exp(ls[i]))
        h = 1e-4
        cov = np.zeros((2, 2))
        for j in range(3):
            d = (pinhole(means[i] + h * L[:, j]) - pinhole(means[i] - h * L[:, j])) / (2 * h)
            cov += np.outer(d, d)
        got = np.array([[pr["cov2d"][i, 0] - 0.3, pr["cov2d"][i, 1]], [pr["cov2d"][i, 1], pr["cov2d"][i, 2] - 0.3]])
        np.testing.assert_allclose(got, cov, rtol=1e-6, atol=1e-8 * np.abs(cov).max())
        np.testing.assert_allclose(pr["mean2d"][i], pinhole(means[i]), rtol=1e-12)
        # the conic (A, B, C) is the inverse of the full 2D covariance (low-pass included)
        S2 = got + 0.3 * np.eye(2)
        A, B, C = pr["conic"][i]
        np.testing.assert_allclose(np.array([[A, B], [B, C]]) @ S2, np.eye(2), atol=1e-9)


def test_projection_invariant_under_joint_rotation():
    """Rotating the scene and the camera together leaves mean2d, conic and depth
    unchanged (catches a transposed camera rotation or quaternion product)."""
    Rot = pytest.importorskip("scipy.spatial.transform").Rotation
    rng = np.random.default_rng(7)
    n = 64
    means = rng.uniform(-0.6, 0.6, (n, 3))
    ls = rng.normal(-3.0, 0.3, (n, 3))
    q = rng.normal(size=(n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    cam = gi.camera((0.5, -2.5, 1.2), 200, 160)
    Q = Rot.from_rotvec([0.3, -0.7, 0.4])
    Qm = Q.as_matrix()
    rq = (Q * Rot.from_quat(q[:, [1, 2, 3, 0]])).as_quat()[:, [3, 0, 1, 2]]
    cam2 = dict(cam)
    cam2["R"] = (cam["R"].astype(np.float64) @ Qm.T).astype(np.float32)
    cam2["campos"] = (Qm @ cam["campos"].astype(np.float64)).astype(np.float32)
    P1, _ = _scene(means, ls, quats=q)
    P2, _ = _scene(means @ Qm.T, ls, quats=rq)
    a = oracle.project(P1, n, cam, 64)
    b = oracle.project(P2, n, cam2, 64)
    for k, tol in (("mean2d", 1e-4), ("conic", 1e-5), ("depth", 1e-6)):
        np.testing.assert_allclose(b[k], a[k], rtol=tol, atol=tol * 1e-2)


def test_projection_fp32_tracks_fp64():
    """The frozen fp32 sequence agrees with the fp64 instantiation to fp32 rounding;
    integer outputs agree except where a value sits within rounding of a ceiling."""
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg)
    cam = gi.cameras_for(cfg)[0]
    a = oracle.project(P, cfg.n, cam, 32)
    b = oracle.project(P, cfg.n, cam, 64)
    v = a["visible"] & b["visible"]
    assert v.sum() > 0.95 * cfg.n
    # mean2d = fx u + cx: absolute error scales with the image coordinates (~100 px)
    np.testing.assert_allclose(a["mean2d"][v], b["mean2d"][v], rtol=2e-5, atol=128 * 4e-7)
    for k in ("conic", "opacity", "rgb", "depth"):
        np.testing.assert_allclose(a[k][v], b[k][v], rtol=2e-5, atol=1e-6)
    assert np.mean(a["radius"][v] == b["radius"][v]) > 0.999


# ----------------------------------------------------------------------------- binning

def test_tile_lists_brute_force():
    """Every tile's list equals, as a sequence, the Gaussians whose closed box
    [m - r, m + r]^2 overlaps the tile's half-open pixel square, sorted by
    (fp32 depth, index): interval overlap, not the floor arithmetic of the rect.
    Copies of a few Gaussians, placed before and after their originals, tie in depth
    exactly: the lower index comes first."""
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg, n=600).copy()
    for src, dst in ((10, 400), (500, 20), (123, 124), (300, 7)):
        P[:, dst] = P[:, src]
    cam = gi.camera((0.0, 0.0, 3.0), 72, 56)   # ragged tiles on both axes
    pr = oracle.project(P, 600, cam, 32)
    vis0 = pr["count"] > 0
    assert len(np.unique(pr["depth"][vis0])) <= vis0.sum() - 3
    tl = oracle.tile_lists(pr, 72, 56)
    m, r, z = pr["mean2d"].astype(np.float64), pr["radius"].astype(np.float64), pr["depth"]
    vis = pr["count"] > 0
    order = np.lexsort((np.arange(600), z))
    TX, TY = 5, 4
    keys, ids, ranges = tl["keys"], tl["ids"], tl["ranges"]
    for ty in range(TY):
        for tx in range(TX):
            hit = (vis & (m[:, 0] - r < 16 * (tx + 1)) & (m[:, 0] + r >= 16 * tx)
                   & (m[:, 1] - r < 16 * (ty + 1)) & (m[:, 1] + r >= 16 * ty))
            exp = [g for g in order if hit[g]]
            t = ty * TX + tx
            s, e = ranges[t]
            assert list(ids[s:e]) == exp
            assert np.all((keys[s:e] >> np.uint64(32)) == t)
            zb = z[ids[s:e]].view(np.uint32)
            assert np.all((keys[s:e] & np.uint64(0xFFFFFFFF)) == zb)
    assert tl["K"] == int(pr["count"].astype(np.int64).sum())


def test_colour_along_the_view_axis_closed_form():
    """A Gaussian at the origin seen from (0, 0, 3): the view direction runs from the
    camera to the mean, d = (0, 0, -1).  On the axis only the m = 0 harmonics are
    nonzero, Y_l0 = sqrt((2l + 1) / 4 pi) P_l(d_z) with P_l(-1) = (-1)^l, at indices
    l^2 + l = 0, 2, 6, 12; so rgb = max(0, 0.5 + sum of those Y_k sh_k) per channel
    (the degree-1 terms sqrt(3 / 4 pi) (-y, z, -x) give -k1 at index 2 and 0 at 1 and
    3), and a channel below zero is clamped and passes no gradient; the others take
    d rgb / d sh_k = Y_k."""
    cam = _cam(32, 32)
    k1 = math.sqrt(3 / (4 * math.pi))
    y0 = 0.5 / math.sqrt(math.pi)
    sh = np.zeros((1, 16, 3))
    sh[0, 0] = [0.2, -0.4, 0.1]
    sh[0, 2] = [0.3, -0.3, 2.0]                     # blue: 0.5 + 0.1 y0 - 2 k1 < 0
    sh[0, 1] = sh[0, 3] = [5.0, -5.0, 5.0]          # Y_1 = Y_3 = 0 along d
    sh[0, 6] = [0.1, 0.2, 0.1]
    sh[0, 12] = [-0.05, 0.1, -0.05]
    P, n = _scene(np.zeros((1, 3)), math.log(0.05), sh=sh)
    pr = oracle.project(P, n, cam, 64)
    Y = np.zeros(16)
    for l in range(4):
        Y[l * l + l] = math.sqrt((2 * l + 1) / (4 * math.pi)) * (-1) ** l
    assert Y[0] == pytest.approx(y0) and Y[2] == pytest.approx(-k1)
    coef = P[11:11 + 48, 0].astype(np.float64).reshape(16, 3)   # as the fp32 planes hold them
    want = np.maximum(0.0, 0.5 + Y @ coef)
    assert want[2] == 0.0 and want[:2].min() > 0
    np.testing.assert_allclose(pr["rgb"][0], want, rtol=1e-12, atol=1e-15)
    for ch in range(3):
        w = np.zeros((9, 1))
        w[6 + ch] = 1.0                             # d rgb[ch] / d params
        g = oracle.project_bwd(P, n, cam, w, prec=64)[:, 0]
        got = g[11 + ch::3][:16]
        if ch == 2:
            assert not got.any()
        else:
            np.testing.assert_allclose(got, Y, atol=1e-12)


def test_loss_is_the_mean_absolute_residual():
    """The loss is l1_weight x the mean of |C - C*| over the 3 H W values (the
    configs' L1 objective), whatever the weight."""
    P, n, cam = _fd_scene()
    pr = oracle.project(P, n, cam, 64)
    img = oracle.render(pr, 32, 32, prec=64)["image"]
    tgt = gi.offset_target(img, seed=3)
    for wgt in (1.0, 0.3):
        rd = oracle.render(pr, 32, 32, target=tgt, prec=64, l1_weight=wgt)
        want = wgt * np.abs(img - tgt.astype(np.float64)).sum() / (3 * 32 * 32)
        assert rd["loss"] == pytest.approx(want, rel=1e-12)


# ----------------------------------------------------------------------------- compositing

def _on_pixel_scene(k, opacity, rgb, W=32, H=32, sigma=0.05):
    """k coincident isotropic Gaussians centred on the centre of pixel (W/2, H/2)."""
    cam = _cam(W, H)
    f = float(cam["fx"])
    # mean2d = f x / z + cx -> world x for a pixel-centre offset of 0.5 px
    x = 0.5 * 3.0 / f
    means = np.tile([x, -x, 0.0], (k, 1))           # camera y axis points down
    logit = math.log(opacity / (1 - opacity))
    sh = np.zeros((k, 16, 3))
    sh[:, 0, :] = (np.asarray(rgb) - 0.5) / (0.5 / math.sqrt(math.pi))
    P, n = _scene(means, math.log(sigma), logits=np.full(k, logit), sh=sh)
    return P, n, cam


@pytest.mark.parametrize("prec", [64, 32])
def test_stacked_gaussians_transmittance_closed_form(prec):
    """k identical coincident Gaussians at a pixel centre (power = 0, alpha = o):
    T = (1 - o)^j after j entries; the pixel stops at the first j with
    (1 - o)^j < 1e-4, and C = rgb (1 - (1 - o)^(j - 1))."""
    o, k = 0.4, 40
    rgb = np.array([0.9, 0.3, 0.6])
    P, n, cam = _on_pixel_scene(k, o, rgb)
    pr = oracle.project(P, n, cam, prec)
    assert np.allclose(pr["mean2d"], 16.5, atol=1e-4)
    rd = oracle.render(pr, 32, 32, prec=prec, count_used=True)
    o = 1.0 / (1.0 + math.exp(-float(P[10, 0])))   # the opacity the fp32 logit holds
    rgb = np.array([0.5 + float(P[11 + c, 0]) * 0.5 / math.sqrt(math.pi) for c in range(3)])
    j_stop = next(j for j in range(1, k + 1) if (1 - o) ** j < 1e-4)
    comp = j_stop - 1
    tol = 1e-12 if prec == 64 else 2e-6
    assert rd["n_contrib"][16, 16] == comp
    assert rd["n_used"][16, 16] == comp             # every entry before the stop composites
    np.testing.assert_allclose(rd["T_final"][16, 16], (1 - o) ** comp, rtol=tol * 10)
    np.testing.assert_allclose(rd["image"][:, 16, 16], rgb * (1 - (1 - o) ** comp), rtol=tol * 10)


def test_single_gaussian_alpha_falloff_closed_form():
    """One isotropic on-axis Gaussian: each pixel's colour is rgb o exp(-|d|^2 / (2 s^2))
    with s^2 = (f sigma / z)^2 + 0.3, zero where that is below 1/255, 0.99 cap."""
    W = H = 48
    cam = _cam(W, H)
    sig, o = 0.08, 0.7
    P, n = _scene(np.zeros((1, 3)), math.log(sig), logits=[math.log(o / (1 - o))],
                  sh=np.tile(np.array([[[(1.0 - 0.5) * 2 * math.sqrt(math.pi)] * 3] + [[0.0] * 3] * 15]), (1, 1, 1)))
    pr = oracle.project(P, n, cam, 64)
    rd = oracle.render(pr, W, H, prec=64, count_used=True)
    sig = math.exp(float(P[3, 0]))                  # values the fp32 planes hold
    o = 1.0 / (1.0 + math.exp(-float(P[10, 0])))
    rgb0 = 0.5 + float(P[11, 0]) * 0.5 / math.sqrt(math.pi)
    s2 = (float(cam["fx"]) * sig / 3.0) ** 2 + 0.3
    ys, xs = np.mgrid[0:H, 0:W] + 0.5
    a = o * np.exp(-((xs - W / 2) ** 2 + (ys - H / 2) ** 2) / (2 * s2))
    a = np.minimum(a, 0.99)
    a[a < 1 / 255] = 0.0
    r = int(pr["radius"][0])
    inside = (np.floor((xs - 0.5) / 16) >= np.floor((W / 2 - r) / 16)) & (np.floor((xs - 0.5) / 16) <= np.floor((W / 2 + r) / 16))
    inside &= (np.floor((ys - 0.5) / 16) >= np.floor((H / 2 - r) / 16)) & (np.floor((ys - 0.5) / 16) <= np.floor((H / 2 + r) / 16))
    a[~inside] = 0.0
    np.testing.assert_allclose(rd["image"][0], rgb0 * a, atol=1e-12)
    np.testing.assert_allclose(rd["T_final"], 1 - a, atol=1e-12)
    # one composited entry exactly where alpha reaches 1/255 (none on the level itself)
    edge = np.abs(o * np.exp(-((xs - W / 2) ** 2 + (ys - H / 2) ** 2) / (2 * s2)) * 255 - 1) < 1e-9
    assert not edge.any()
    np.testing.assert_array_equal(rd["n_used"], (a > 0).astype(np.uint32))


def test_anisotropic_footprint_is_the_gaussian_of_the_2d_covariance():
    """One rotated, elongated Gaussian: each pixel's alpha is o exp(-d^T Sigma_2^-1 d / 2)
    with Sigma_2 the projected 2D covariance (fixed by the EWA pin) inverted here by
    numpy, capped at 0.99, zero below 1/255 and outside the tile rect; the image is
    rgb alpha on black."""
    W = H = 48
    cam = _cam(W, H)
    Rot = pytest.importorskip("scipy.spatial.transform").Rotation
    q = Rot.from_euler("xyz", [0.4, -0.3, 0.7]).as_quat()          # (x, y, z, w)
    sh = np.zeros((1, 16, 3))
    sh[0, 0] = [0.8, 0.2, -0.3]
    P, n = _scene(np.zeros((1, 3)), np.array([[math.log(0.15), math.log(0.04), math.log(0.08)]]),
                  quats=np.array([[q[3], q[0], q[1], q[2]]]), logits=[1.5], sh=sh)
    pr = oracle.project(P, n, cam, 64)
    rd = oracle.render(pr, W, H, prec=64)
    a, b, c = pr["cov2d"][0]
    assert abs(b) > 0.2 * math.sqrt(a * c)                          # clearly anisotropic, tilted
    Sinv = np.linalg.inv(np.array([[a, b], [b, c]]))
    ys, xs = np.mgrid[0:H, 0:W] + 0.5
    d = np.stack([xs - pr["mean2d"][0, 0], ys - pr["mean2d"][0, 1]], -1)
    alpha = float(pr["opacity"][0]) * np.exp(-0.5 * np.einsum("...i,ij,...j->...", d, Sinv, d))
    alpha = np.minimum(alpha, 0.99)
    alpha[alpha < 1 / 255] = 0.0
    tx0, ty0, tx1, ty1 = pr["rect"][0]
    tile_x, tile_y = np.floor((xs - 0.5) / 16), np.floor((ys - 0.5) / 16)
    alpha[~((tile_x >= tx0) & (tile_x <= tx1) & (tile_y >= ty0) & (tile_y <= ty1))] = 0.0
    assert (alpha > 0).sum() > 50
    np.testing.assert_allclose(rd["image"], pr["rgb"][0][:, None, None] * alpha[None], atol=1e-12)
    np.testing.assert_allclose(rd["T_final"], 1.0 - alpha, atol=1e-12)


def test_alpha_sum_and_colour_bounds():
    """Accumulated alpha 1 - T lies in [0, 1 - 1e-4]; each channel is at most
    max colour x (1 - T) with a black background."""
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg)
    cam = gi.cameras_for(cfg)[0]
    pr = oracle.project(P, cfg.n, cam, 32)
    rd = oracle.render(pr, 128, 128, count_used=True)
    T = rd["T_final"].astype(np.float64)
    assert T.max() <= 1.0 and T.min() >= 1e-4 * (1 - 1e-6)
    # composited entries: at most those iterated, the last iterated one among them, and
    # each takes at least 1/255 of the remaining transmittance
    nu, nc = rd["n_used"].astype(np.int64), rd["n_contrib"].astype(np.int64)
    assert np.all(nu <= nc) and np.array_equal(nu == 0, nc == 0)
    assert np.all(T <= (1 - 1 / 255) ** nu * (1 + 1e-5))
    assert nu.max() > 1
    cmax = pr["rgb"][pr["visible"]].max()
    assert np.all(rd["image"] <= cmax * (1 - T)[None] * (1 + 1e-5) + 1e-6)
    assert np.all(rd["image"] >= 0)


def test_permutation_invariance_distinct_depths():
    """Reordering the Gaussians in memory leaves the fp32 image, T and n_contrib
    bit-identical when depths are distinct (order comes from depth, not index)."""
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg, n=1500)
    cam = gi.camera((0.0, 0.0, 3.0), 96, 80)
    n = 1500
    # drop (put behind the camera) all but one member of any group of equal fp32 depth
    z0 = oracle.project(P, n, cam, 32)["depth"]
    _, first = np.unique(z0, return_index=True)
    dup = np.setdiff1d(np.arange(n), first)
    P[0:3, dup] = np.array([[0.0], [0.0], [10.0]], np.float32)
    perm = np.random.default_rng(1).permutation(n)
    P2 = P.copy()
    P2[:, :n] = P[:, :n][:, perm]
    a = oracle.project(P, n, cam, 32)
    b = oracle.project(P2, n, cam, 32)
    assert len(np.unique(a["depth"][a["visible"]])) == a["visible"].sum()
    ra, rb = oracle.render(a, 96, 80), oracle.render(b, 96, 80)
    for k in ("image", "T_final", "n_contrib"):
        np.testing.assert_array_equal(ra[k], rb[k])


def test_equal_depth_order_invariance():
    """Coincident Gaussians at equal depth with equal colours: swapping their order
    leaves colour and transmittance unchanged (products commute)."""
    rgb = np.array([0.2, 0.8, 0.5])
    cam = _cam(32, 32)
    means = np.zeros((3, 3))
    logits = np.array([0.5, -0.3, 1.1])
    sh = np.zeros((3, 16, 3))
    sh[:, 0, :] = (rgb - 0.5) * 2 * math.sqrt(math.pi)
    P1, n = _scene(means, math.log(0.07), logits=logits, sh=sh)
    P2, _ = _scene(means, math.log(0.07), logits=logits[::-1].copy(), sh=sh)
    r1 = oracle.render(oracle.project(P1, n, cam, 64), 32, 32, prec=64)
    r2 = oracle.render(oracle.project(P2, n, cam, 64), 32, 32, prec=64)
    np.testing.assert_allclose(r1["T_final"], r2["T_final"], atol=1e-14)
    np.testing.assert_allclose(r1["image"], r2["image"], atol=1e-14)


# ----------------------------------------------------------------------------- gradients

def _fd_scene(n=6, seed=11, W=32, H=32):
    rng = np.random.default_rng(seed)
    means = np.column_stack([rng.uniform(-0.35, 0.35, n), rng.uniform(-0.35, 0.35, n), rng.uniform(-0.3, 0.3, n)])
    ls = rng.normal(-2.2, 0.25, (n, 3))
    q = rng.normal(size=(n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    logits = rng.normal(0.0, 0.8, n)
    sh = np.zeros((n, 16, 3))
    sh[:, 0, :] = rng.uniform(-1, 1, (n, 3))
    sh[:, 1:, :] = rng.normal(0, 0.3, (n, 15, 3))
    P, _ = _scene(means, ls, quats=q, logits=logits, sh=sh)
    cam = gi.camera((0.4, -0.3, 2.9), W, H)
    return P, n, cam


def _clamped_pixels(pr, i, W=32, H=32):
    """Pixels where Gaussian i alone reaches the 0.99 opacity clamp (o e^power >= 0.99)."""
    ys, xs = np.mgrid[0:H, 0:W] + 0.5
    mx, my = pr["mean2d"][i]
    A, B, C = pr["conic"][i]
    dx, dy = xs - mx, ys - my
    power = -0.5 * (A * dx * dx + C * dy * dy) - B * dx * dy
    return int((pr["opacity"][i] * np.exp(power) >= 0.99).sum())


@pytest.mark.parametrize("hot,bg", [(None, (0.0, 0.0, 0.0)), (2, (0.0, 0.0, 0.0)), (None, (0.3, 0.6, 0.1))])
def test_render_backward_matches_finite_differences(hot, bg):
    """The suffix-sum backward equals central differences (fp64) of the L1 loss with
    respect to each projected quantity (mean2d, conic, opacity, colour), with
    tile rects held fixed and every residual sign far from zero.  With ``hot``, that
    Gaussian is nearly opaque (logit 12) and about 12 px wide: its alpha sits at the
    0.99 clamp over a disc of pixels, where alpha no longer depends on its opacity or
    its power.  With a coloured background, what shows through (T_final bg) depends
    on every entry's alpha too."""
    P, n, cam = _fd_scene()
    if hot is not None:
        P = P.copy()
        P[10, hot] = 12.0
        P[3:6, hot] += 3.0
    pr = oracle.project(P, n, cam, 64)
    if hot is not None:
        assert _clamped_pixels(pr, hot) >= 20
    base = oracle.render(pr, 32, 32, bg=bg, prec=64)
    tgt = gi.offset_target(base["image"], seed=3)
    rd = oracle.render(pr, 32, 32, bg=bg, target=tgt, prec=64)
    g2 = rd["grad2d"]
    assert np.abs(g2).max() > 0
    cols = [0, 1, 2, 3, 4, 5, 6, 7, 8]
    for i in range(n):
        if not pr["visible"][i]:
            continue
        for q, col in enumerate(cols):
            x0 = pr["proj16"][i, col]
            h = 1e-6 * max(1.0, abs(x0))
            vals = []
            for sgn in (1, -1):
                p2 = dict(pr)
                p2["proj16"] = pr["proj16"].copy()
                p2["proj16"][i, col] = x0 + sgn * h
                r = oracle.render(p2, 32, 32, bg=bg, target=tgt, prec=64)
                np.testing.assert_array_equal(r["n_contrib"], rd["n_contrib"])
                vals.append(r["loss"])
            fd = (vals[0] - vals[1]) / (2 * h)
            assert abs(fd - g2[q, i]) <= 1e-6 * abs(fd) + 1e-10, (i, q, fd, g2[q, i])


def _beyond_clamp_scene(W=64, H=64, sig=0.9):
    """Two isotropic Gaussians at depth 3 whose camera-space abscissa x / z (first) or
    ordinate y / z (second) is twice 1.3 x the half field of view, so the EWA
    Jacobian takes the clamped value; wide enough that their footprints still reach
    the image."""
    cam = _cam(W, H)
    z = 3.0
    limx = 1.3 * (0.5 * W) / float(cam["fx"])
    limy = 1.3 * (0.5 * H) / float(cam["fy"])
    c = np.array([[2 * limx * z, 0.0, z], [0.0, -2 * limy * z, z]])
    R = cam["R"].astype(np.float64)
    t = cam["t"].astype(np.float64)
    means = (c - t) @ R                              # world = R^T (c - t)
    P, n = _scene(means, math.log(sig), logits=[1.0, -0.5])
    return P, n, cam, limx, limy


def test_projection_jacobian_clamp_closed_form():
    """Beyond 1.3 x the half field of view the EWA Jacobian uses the clamped
    abscissa (cited method): for an isotropic Gaussian of scale s at (x, 0, z) with
    x / z past the limit L, J J^T = (f / z)^2 [[1 + L^2, 0], [0, 1]], so
    Sigma_2 = s^2 (f / z)^2 diag(1 + L^2, 1) + 0.3 I; likewise along y.  The mean
    itself projects unclamped."""
    P, n, cam, limx, limy = _beyond_clamp_scene()
    pr = oracle.project(P, n, cam, 64)
    assert pr["visible"].all()
    s = np.exp(P[3, :n].astype(np.float64))
    fx, fy = float(cam["fx"]), float(cam["fy"])
    z = (P[:3, :n].T.astype(np.float64) @ cam["R"].astype(np.float64).T + cam["t"].astype(np.float64))[:, 2]
    a = (s * fx / z) ** 2
    b = (s * fy / z) ** 2
    np.testing.assert_allclose(pr["cov2d"][0], [a[0] * (1 + limx ** 2) + 0.3, 0.0, b[0] + 0.3], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(pr["cov2d"][1], [a[1] + 0.3, 0.0, b[1] * (1 + limy ** 2) + 0.3], rtol=1e-9, atol=1e-9)
    # the means as the fp32 planes hold them, in camera space
    c = P[:3, :n].T.astype(np.float64) @ cam["R"].astype(np.float64).T + cam["t"].astype(np.float64)
    assert c[0, 0] / c[0, 2] > 1.9 * limx and c[1, 1] / c[1, 2] < -1.9 * limy
    np.testing.assert_allclose(pr["mean2d"][:, 0], fx * c[:, 0] / c[:, 2] + float(cam["cx"]), rtol=1e-12)
    np.testing.assert_allclose(pr["mean2d"][:, 1], fy * c[:, 1] / c[:, 2] + float(cam["cy"]), rtol=1e-12, atol=1e-12)


def _project_bwd_fd(P, n, cam, w):
    """Central differences (fp64) of sum(w * the nine projected outputs) against the
    analytic chain rule, for all 59 parameters of each Gaussian."""
    an = oracle.project_bwd(P, n, cam, w, prec=64)

    def func(Pm):
        r = oracle.project(Pm, n, cam, 64)
        return float((r["proj16"][:, :9].T * w).sum())

    for i in range(n):
        for pl in range(59):
            x0 = float(P[pl, i])
            h = 1e-3 * max(abs(x0), 0.05)
            Pp, Pm_ = P.copy(), P.copy()
            Pp[pl, i] = np.float32(x0 + h)
            Pm_[pl, i] = np.float32(x0 - h)
            he = (float(Pp[pl, i]) - float(Pm_[pl, i])) / 2
            fd = (func(Pp) - func(Pm_)) / (2 * he)
            assert abs(fd - an[pl, i]) <= 2e-5 * abs(fd) + 1e-7 * np.abs(an[:, i]).max() + 1e-9, (i, pl, fd, an[pl, i])


def test_project_backward_matches_finite_differences():
    """The projection chain rule equals central differences (fp64) of a random
    linear functional of the nine projected outputs with respect to all 59
    parameters of each Gaussian (SH, quaternion normalisation, scales, mean)."""
    P, n, cam = _fd_scene(n=4, seed=2)
    assert oracle.project(P, n, cam, 64)["visible"].all()
    _project_bwd_fd(P, n, cam, np.random.default_rng(4).normal(size=(9, n)))


def test_project_backward_through_the_jacobian_clamp():
    """Past the clamp the Jacobian no longer follows the mean's abscissa, so that
    path passes no gradient; central differences of the clamped forward agree."""
    P, n, cam, _, _ = _beyond_clamp_scene()
    assert oracle.project(P, n, cam, 64)["visible"].all()
    _project_bwd_fd(P, n, cam, np.random.default_rng(6).normal(size=(9, n)))


def test_whole_step_gradient_matches_finite_differences():
    """End to end: d loss / d params from render backward then projection backward
    equals central differences of the whole fp64 forward (all 59 planes)."""
    P, n, cam = _fd_scene(n=3, seed=9)
    pr = oracle.project(P, n, cam, 64)
    tgt = gi.offset_target(oracle.render(pr, 32, 32, prec=64)["image"], seed=5)
    rd = oracle.render(pr, 32, 32, target=tgt, prec=64)
    an = oracle.project_bwd(P, n, cam, rd["grad2d"], prec=64)

    def loss(Pm):
        return oracle.render(oracle.project(Pm, n, cam, 64), 32, 32, target=tgt, prec=64)["loss"]

    checked = 0
    for i in range(n):
        for pl in range(59):
            x0 = float(P[pl, i])
            h = 1e-3 * max(abs(x0), 0.05)
            Pp, Pm_ = P.copy(), P.copy()
            Pp[pl, i] = np.float32(x0 + h)
            Pm_[pl, i] = np.float32(x0 - h)
            he = (float(Pp[pl, i]) - float(Pm_[pl, i])) / 2
            fd = (loss(Pp) - loss(Pm_)) / (2 * he)
            assert abs(fd - an[pl, i]) <= 2e-4 * abs(fd) + 2e-7 * np.abs(an).max(), (i, pl, fd, an[pl, i])
            checked += 1
    assert checked == 3 * 59


# ----------------------------------------------------------------------------- Adam

def test_adam_constant_gradient_closed_form():
    """With a constant gradient g the bias-corrected moments are exactly g and g^2,
    so after t steps p = p0 - t lr g / (|g| + eps)."""
    rng = np.random.default_rng(0)
    planes, stride = 59, 64
    p0 = rng.normal(size=(planes, stride))
    g = rng.normal(size=(planes, stride)) * 10.0 ** rng.integers(-6, 1, (planes, stride))
    lr = gi.lr_planes()
    p, m, v = p0, np.zeros_like(p0), np.zeros_like(p0)
    T = 7
    for t in range(1, T + 1):
        p, m, v = oracle.adam(p, g, m, v, lr, 0.9, 0.999, 1e-15, t)
    np.testing.assert_allclose(p, p0 - T * lr[:, None] * g / (np.abs(g) + 1e-15), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(m, g * (1 - 0.9 ** T), rtol=1e-12)
    np.testing.assert_allclose(v, g * g * (1 - 0.999 ** T), rtol=1e-12)


def test_adam_first_step_is_signed_lr():
    """One step from zero moments moves each parameter by lr sign(g) (|g| >> eps),
    whatever beta1 and beta2 are."""
    rng = np.random.default_rng(1)
    p0 = rng.normal(size=(59, 32))
    g = rng.normal(size=(59, 32))
    lr = gi.lr_planes()
    for b1, b2 in ((0.9, 0.999), (0.0, 0.5)):
        p, _, _ = oracle.adam(p0, g, np.zeros_like(p0), np.zeros_like(p0), lr, b1, b2, 1e-15, 1)
        np.testing.assert_allclose(p, p0 - lr[:, None] * np.sign(g), rtol=1e-12)


# ----------------------------------------------------------------------------- SSIM

def _ssim_stats_scipy(x, y):
    """Local means and (co)variances from scipy: 11x11 window from scipy's Gaussian
    (std 1.5, normalised), zero padding outside the image."""
    nd = pytest.importorskip("scipy.ndimage")
    windows = pytest.importorskip("scipy.signal.windows")
    g = windows.gaussian(11, std=1.5)
    w = np.outer(g, g)
    w /= w.sum()
    f = lambda a: nd.correlate(a, w, mode="constant", cval=0.0)
    mx, my = f(x), f(y)
    return mx, my, f(x * x) - mx * mx, f(y * y) - my * my, f(x * y) - mx * my


def test_ssim_identity_and_symmetry():
    """SSIM(x, x) = 1 with zero gradient (its maximum); SSIM(x, y) = SSIM(y, x)."""
    rng = np.random.default_rng(0)
    x = rng.uniform(0, 1, (3, 30, 26))
    y = rng.uniform(0, 1, (3, 30, 26))
    s, g = oracle.ssim(x, x)
    assert abs(s - 1.0) < 1e-14 and np.abs(g).max() < 1e-14
    assert abs(oracle.ssim(x, y)[0] - oracle.ssim(y, x)[0]) < 1e-14


def test_ssim_reduces_to_library_statistics():
    """With y = 0 the index is C1/(mu_x^2 + C1) * C2/(s_xx + C2); with y = a x it is
    (2a mu^2 + C1)/((1+a^2) mu^2 + C1) * (2a s + C2)/((1+a^2) s + C2); local statistics
    from scipy's correlate with zero padding."""
    rng = np.random.default_rng(1)
    x = rng.uniform(0, 1, (3, 33, 29))
    C1, C2 = 0.01 ** 2, 0.03 ** 2
    for a in (0.0, 0.6, 1.7):
        y = a * x
        ref = []
        for c in range(3):
            mx, _, sxx, _, _ = _ssim_stats_scipy(x[c], y[c])
            ref.append((2 * a * mx * mx + C1) / ((1 + a * a) * mx * mx + C1)
                       * (2 * a * sxx + C2) / ((1 + a * a) * sxx + C2))
        assert abs(oracle.ssim(x, y)[0] - np.mean(ref)) < 1e-12, a


def test_ssim_gradient_matches_finite_differences():
    """d/dx of lambda (1 - SSIM) against central differences at every pixel of a small
    image (borders included)."""
    rng = np.random.default_rng(2)
    x = rng.uniform(0.1, 0.9, (3, 14, 12))
    y = np.clip(x + rng.normal(0, 0.2, x.shape), 0, 1)
    lam = 0.2
    _, g = oracle.ssim(x, y, lam)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = lam * ((1 - oracle.ssim(xp, y)[0]) - (1 - oracle.ssim(xm, y)[0])) / (2 * h)
    np.testing.assert_allclose(g, fd, rtol=1e-5, atol=1e-9 * np.abs(g).max())


def test_whole_step_gradient_with_dssim_matches_finite_differences():
    """(1 - lambda) L1 + lambda (1 - SSIM): the render backward with the SSIM image
    gradient added, then the projection backward, equals central differences of the
    whole fp64 forward.  The steps change no compositing decision (n_contrib is the
    same at +h and -h), so the loss is smooth across each difference."""
    P, n, cam = _fd_scene(n=3, seed=9)
    lam = 0.2
    pr = oracle.project(P, n, cam, 64)
    img = oracle.render(pr, 32, 32, prec=64)["image"]
    tgt = gi.offset_target(img, seed=6)
    _, extra = oracle.ssim(img, tgt, lam)
    assert np.abs(extra).max() > 0
    rd = oracle.render(pr, 32, 32, target=tgt, prec=64, l1_weight=1 - lam, dLdC_extra=extra)
    an = oracle.project_bwd(P, n, cam, rd["grad2d"], prec=64)

    def loss(Pm):
        p = oracle.project(Pm, n, cam, 64)
        r = oracle.render(p, 32, 32, target=tgt, prec=64, l1_weight=1 - lam)
        np.testing.assert_array_equal(r["n_contrib"], rd["n_contrib"])
        return r["loss"] + lam * (1 - oracle.ssim(r["image"], tgt)[0])

    def central(i, pl, h):
        x0 = float(P[pl, i])
        Pp, Pm_ = P.copy(), P.copy()
        Pp[pl, i] = np.float32(x0 + h)
        Pm_[pl, i] = np.float32(x0 - h)
        he = (float(Pp[pl, i]) - float(Pm_[pl, i])) / 2
        return (loss(Pp) - loss(Pm_)) / (2 * he), he

    for i in range(n):
        for pl in (0, 1, 2, 3, 6, 10, 11, 14, 20, 58):
            h = 1e-3 * max(abs(float(P[pl, i])), 0.05)
            # Richardson: the central difference is D + c he^2 + O(he^4); two step
            # sizes remove the he^2 term
            d1, e1 = central(i, pl, h)
            d2, e2 = central(i, pl, h / 2)
            fd = (d2 * e1 * e1 - d1 * e2 * e2) / (e1 * e1 - e2 * e2)
            assert abs(fd - an[pl, i]) <= 2e-4 * abs(fd) + 2e-7 * np.abs(an).max(), (i, pl, fd, an[pl, i])


def test_step_composes_the_objective():
    """The whole step with lambda in {0, 0.2}: its loss is (1 - lambda) mean |C - C*| +
    lambda (1 - SSIM(C, C*)) of its own render, and its parameter gradients are those
    of the composition the test above checks against finite differences (render
    backward with weight 1 - lambda plus the SSIM image gradient, then the projection
    backward), up to the fp32 decisions and image the step uses."""
    P, n, cam = _fd_scene(n=3, seed=9)
    pr = oracle.project(P, n, cam, 64)
    img = oracle.render(pr, 32, 32, prec=64)["image"]
    tgt = gi.offset_target(img, seed=6)
    z = np.zeros((59, P.shape[1]))
    for lam in (0.0, 0.2):
        r = oracle.step(P, n, cam, tgt, z, z, 1, gi.lr_planes(), dssim=lam)
        c = r["render"]["image"].astype(np.float64)
        want = (1 - lam) * np.abs(c - tgt).mean() + lam * (1 - oracle.ssim(c, tgt)[0])
        assert r["render"]["loss"] == pytest.approx(want, rel=1e-9)
        extra = oracle.ssim(img, tgt, lam)[1] if lam > 0 else None
        rd = oracle.render(pr, 32, 32, target=tgt, prec=64, l1_weight=1 - lam, dLdC_extra=extra)
        an = oracle.project_bwd(P, n, cam, rd["grad2d"], prec=64)
        g = r["grads"][:, :n]
        scale = np.abs(an).max(axis=1, keepdims=True)
        assert np.all(np.abs(g - an) <= 1e-3 * np.abs(an) + 1e-4 * scale)


# ----------------------------------------------------------------------------- batched step

def test_batch_hyperparameters_follow_the_pages():
    """"Scaling 3D Gaussian Splatting with Distributed Compute", batch-size section:
    learning rates grow as sqrt(BS), epsilon shrinks as 1/sqrt(BS), and the momentum
    linearisation takes beta1 = 0.9 to zero at BS = 10 (held at zero beyond)."""
    lr = np.full(59, 1e-3)
    for B, b1, b2 in ((1, 0.9, 0.999), (4, 0.6, 0.996), (10, 0.0, 0.99)):
        lr_b, c1, c2, e = oracle.batch_hyper(B, lr, 0.9, 0.999, 1e-15)
        np.testing.assert_allclose(lr_b, 1e-3 * np.sqrt(B), rtol=1e-15)
        assert abs(c1 - b1) < 1e-12 and abs(c2 - b2) < 1e-12, (B, c1, c2)
        assert abs(e - 1e-15 / np.sqrt(B)) < 1e-30
    assert oracle.batch_hyper(12, lr, 0.9, 0.999, 1e-15)[1] == 0.0


def _two_views(seed=11):
    P, n, cam = _fd_scene(n=6, seed=seed)
    cam2 = gi.camera((-0.5, 0.35, 2.8), 32, 32)
    pr1, pr2 = oracle.project(P, n, cam, 32), oracle.project(P, n, cam2, 32)
    t1 = gi.offset_target(oracle.render(pr1, 32, 32)["image"], seed=21)
    t2 = gi.offset_target(oracle.render(pr2, 32, 32)["image"], seed=22)
    return P, n, [cam, cam2], [t1, t2]


def test_batch_of_one_is_the_single_view_step():
    P, n, cams, targets = _two_views()
    z = np.zeros((59, P.shape[1]))
    a = oracle.step(P, n, cams[0], targets[0], z, z, 1, gi.lr_planes())
    b = oracle.step_batch(P, n, cams[:1], targets[:1], z, z, 1, gi.lr_planes())
    np.testing.assert_array_equal(b["grads"], a["grads"])
    for k in ("params", "m", "v"):
        np.testing.assert_allclose(b[k], a[k], rtol=1e-15, atol=0)


@pytest.mark.parametrize("lam", [0.0, 0.2])
def test_batch_gradient_is_the_mean_of_view_gradients(lam):
    """The batch loss is the mean of the view losses, so its gradient is the mean of
    the single-view gradients (a dropped 1/BS or a missing view fails), with or
    without the D-SSIM term."""
    P, n, cams, targets = _two_views()
    z = np.zeros((59, P.shape[1]))
    s1 = oracle.step(P, n, cams[0], targets[0], z, z, 1, gi.lr_planes(), dssim=lam)
    s2 = oracle.step(P, n, cams[1], targets[1], z, z, 1, gi.lr_planes(), dssim=lam)
    g1, g2 = s1["grads"], s2["grads"]
    r = oracle.step_batch(P, n, cams, targets, z, z, 1, gi.lr_planes(), dssim=lam)
    assert np.abs(g1 - g2).max() > 1e-3 * np.abs(g1).max()
    np.testing.assert_allclose(r["grads"], 0.5 * (g1 + g2), rtol=1e-9, atol=1e-18)
    assert abs(r["loss"] - 0.5 * (s1["render"]["loss"] + s2["render"]["loss"])) < 1e-12


def test_batch_first_step_moves_by_sqrt_batch_lr():
    """Four identical views: the gradient is the single view's, and the first Adam
    step from zero moments moves each parameter by lr sqrt(4) sign(g) where |g| is
    far above epsilon / sqrt(4)."""
    P, n, cams, targets = _two_views()
    z = np.zeros((59, P.shape[1]))
    g = oracle.step(P, n, cams[0], targets[0], z, z, 1, gi.lr_planes())["grads"]
    r = oracle.step_batch(P, n, [cams[0]] * 4, [targets[0]] * 4, z, z, 1, gi.lr_planes())
    np.testing.assert_allclose(r["grads"], g, rtol=1e-12, atol=1e-18)
    lr = np.asarray(gi.lr_planes(), np.float64)[:, None]
    big = np.abs(g) > 1e-6  # epsilon / sqrt(4) is below 1e-9 of these
    expect = P.astype(np.float64) - 2.0 * lr * np.sign(g)
    assert big.sum() > 50
    np.testing.assert_allclose(r["params"][big], expect[big], rtol=0, atol=1e-11)  # a flip moves by >= 2.5e-4


# ----------------------------------------------------------------------------- density control

def _dscene(n=8, seed=0):
    rng = np.random.default_rng(seed)
    means = rng.uniform(-0.5, 0.5, (n, 3))
    ls = np.full((n, 3), -5.0)  # scale 0.0067: below 0.01 x extent 1
    q = rng.normal(size=(n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    P, _ = _scene(means, ls, quats=q, logits=np.zeros(n))
    return P


def test_densify_thresholds_are_the_stated_ones():
    """fp32 thresholds formed in fp64: sigmoid(logit_prune) = 0.005, exp(log scale) =
    0.01 x extent, the reset logit is that of 2 x 0.005, and the split shrink is 1.6."""
    th = oracle.densify.thresholds(extent=3.3)
    # fp32 rounding of a logit near -5 moves the sigmoid by at most ~3e-9
    assert abs(1.0 / (1.0 + math.exp(-float(th["logit_prune"]))) - 0.005) < 5e-9
    assert abs(math.exp(float(th["log_grow_scale"])) - 0.033) < 1e-8
    assert abs(math.exp(float(th["log_prune_scale"])) - 0.33) < 1e-7
    assert abs(1.0 / (1.0 + math.exp(-float(th["logit_reset"]))) - 0.01) < 5e-9
    assert abs(math.exp(float(th["log_shrink"])) - 1.6) < 1e-6
    assert th["grad"] == np.float32(2e-4)


def test_densify_decisions_on_constructed_gaussians():
    D = oracle.densify
    th = D.thresholds(extent=1.0)
    P = _dscene()
    n = 8
    acc = np.zeros(n, np.float32)
    cnt = np.zeros(n, np.int64)
    P[10, 0] = -6.0                              # sigmoid 0.0025 < 0.005: prune
    acc[1], cnt[1] = 9e-4, 3                      # mean 3e-4 > 2e-4, small: clone
    acc[2], cnt[2] = 9e-4, 3
    P[3:6, 2] = [-4.0, -2.0, -4.0]                # max scale e^-2 = 0.135 > 0.01: split
    acc[3], cnt[3] = 3e-4, 3                      # mean 1e-4: keep
    P[10, 4] = float(th["logit_prune"])           # exactly at the threshold: not below, keep
    acc[5], cnt[5] = np.float32(2e-4), 1          # mean equals the threshold (strict >): keep
    acc[6], cnt[6] = 6e-4, 2                      # mean 3e-4 and max log-scale exactly at the
    P[3:6, 6] = [float(th["log_grow_scale"]), -5.0, -5.0]  # clone threshold (<=): clone
    P[10, 7] = -5.3                               # sigmoid 0.00497 < 0.005: prune
    action, offset, n_out = D.plan(P, n, acc, cnt, th)
    assert action.tolist() == [D.PRUNE, D.CLONE, D.SPLIT, D.KEEP, D.KEEP, D.KEEP, D.CLONE, D.PRUNE]
    assert offset.tolist() == [0, 0, 2, 4, 5, 6, 7, 9]
    assert n_out == 9
    # the optional large-Gaussian prune also removes Gaussian 2: its largest log-scale
    # -2 exceeds ln(0.1 x extent) = -2.303
    a2, _, _ = D.plan(P, n, acc, cnt, th, prune_big=True)
    assert a2[2] == D.PRUNE and (a2 == D.PRUNE).sum() == 3


def test_split_children_follow_the_rotated_axes():
    """With xi = (e_a, e_b) the children sit at mu + s_a r_a and mu + s_b r_b, where r_k
    is column k of the rotation (scipy's, from the same quaternion) and s_k the scale;
    children's log-scales are shrunk by ln 1.6, every other plane is copied and their
    Adam moments start at zero."""
    Rot = pytest.importorskip("scipy.spatial.transform").Rotation
    D = oracle.densify
    th = D.thresholds()
    P = _dscene(n=4, seed=3)
    P[3:6, :4] = np.array([[-1.0, -1.5, -2.0]] * 4).T
    n = 4
    acc = np.full(n, 1e-3, np.float32)
    cnt = np.ones(n, np.int64)
    action, offset, n_out = D.plan(P, n, acc, cnt, th)
    assert (action == D.SPLIT).all() and n_out == 8
    randn = np.zeros((n, 6), np.float32)
    for i in range(n):
        randn[i, i % 3] = 1.0              # child 0 along axis i % 3
        randn[i, 3 + (i + 1) % 3] = -2.0   # child 1 along axis (i + 1) % 3, twice, reversed
    m = np.random.default_rng(0).normal(size=(59, P.shape[1])).astype(np.float32)
    v = np.abs(m)
    out_p, out_m, out_v = D.apply(P, m, v, n, action, offset, n_out, randn, th)
    for i in range(n):
        q = P[6:10, i].astype(np.float64)
        rot = Rot.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()
        s = np.exp(P[3:6, i].astype(np.float64))
        a, b = i % 3, (i + 1) % 3
        np.testing.assert_allclose(out_p[0:3, 2 * i], P[0:3, i] + s[a] * rot[:, a], rtol=0, atol=1e-6)
        np.testing.assert_allclose(out_p[0:3, 2 * i + 1], P[0:3, i] - 2.0 * s[b] * rot[:, b], rtol=0, atol=1e-6)
        for k in (0, 1):
            np.testing.assert_array_equal(out_p[3:6, 2 * i + k], (P[3:6, i] - np.float32(np.log(1.6))))
            np.testing.assert_array_equal(out_p[6:, 2 * i + k], P[6:, i])
    assert not out_m[:, :8].any() and not out_v[:, :8].any()
    assert not out_p[:, 8:].any()


def test_clone_keeps_the_original_moments_and_copies_it():
    D = oracle.densify
    th = D.thresholds()
    P = _dscene(n=3, seed=4)
    n = 3
    acc = np.array([1e-3, 0.0, 1e-3], np.float32)
    cnt = np.array([2, 0, 2])
    action, offset, n_out = D.plan(P, n, acc, cnt, th)
    assert action.tolist() == [D.CLONE, D.KEEP, D.CLONE] and offset.tolist() == [0, 2, 3] and n_out == 5
    rng = np.random.default_rng(1)
    m = rng.normal(size=P.shape).astype(np.float32)
    v = np.abs(rng.normal(size=P.shape)).astype(np.float32)
    out_p, out_m, out_v = D.apply(P, m, v, n, action, offset, n_out, np.zeros((n, 6), np.float32), th)
    for src, dst in ((0, 0), (1, 2), (2, 3)):
        np.testing.assert_array_equal(out_p[:, dst], P[:, src])
        np.testing.assert_array_equal(out_m[:, dst], m[:, src])
        np.testing.assert_array_equal(out_v[:, dst], v[:, src])
    for src, dst in ((0, 1), (2, 4)):
        np.testing.assert_array_equal(out_p[:, dst], P[:, src])
        assert not out_m[:, dst].any() and not out_v[:, dst].any()


def test_densify_count_identity_and_offsets():
    """N_out = N - pruned - split + cloned + 2 split, offsets strictly increase over
    the Gaussians that produce output, and every output column is written once."""
    D = oracle.densify
    th = D.thresholds(extent=3.3)
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg).copy()
    n = cfg.n
    P[10, :n:40] = -7.0  # some transparent Gaussians to prune
    rng = np.random.default_rng(7)
    acc = rng.exponential(3e-4, n).astype(np.float32)
    cnt = rng.integers(0, 4, n)
    action, offset, n_out = D.plan(P, n, acc, cnt, th, prune_big=True)
    c = np.bincount(action, minlength=4)
    assert min(c) > 0
    assert n_out == n - c[D.PRUNE] - c[D.SPLIT] + c[D.CLONE] + 2 * c[D.SPLIT]
    live = action != D.PRUNE
    assert np.all(np.diff(offset[live].astype(np.int64)) > 0)
    out_p, _, _ = D.apply(P, P, P, n, action, offset, n_out, rng.normal(size=(n, 6)).astype(np.float32), th)
    assert out_p.shape[1] % 256 == 0 and out_p.shape[1] >= n_out
    written = np.zeros(out_p.shape[1], bool)
    for i in np.nonzero(live)[0]:
        written[offset[i]:offset[i] + (1 if action[i] == D.KEEP else 2)] = True
    assert written[:n_out].all() and not written[n_out:].any()


def test_opacity_reset_clamps_to_twice_the_prune_opacity():
    D = oracle.densify
    th = D.thresholds()
    P = _dscene(n=4, seed=5)
    P[10, :4] = [-6.0, -4.0, 0.0, 3.0]
    m = np.ones_like(P)
    v = np.ones_like(P)
    D.opacity_reset(P, m, v, 4, th)
    sig = 1.0 / (1.0 + np.exp(-P[10, :4].astype(np.float64)))
    np.testing.assert_allclose(sig, np.minimum([0.0024726, 0.0179862, 0.5, 0.9525741], 0.01), rtol=1e-5)
    assert not m[10, :4].any() and not v[10, :4].any() and m[9, 0] == 1.0


def test_accumulate_is_the_ndc_scaled_norm():
    """A gradient of (2a / W, 2b / H) on the projected mean is (a, b) in NDC units:
    the accumulator gains sqrt(a^2 + b^2) for visible Gaussians and nothing else."""
    D = oracle.densify
    W, H = 64, 48
    g = np.zeros((9, 3), np.float32)
    g[0] = [2 * 3.0 / W, 2 * 0.5 / W, 1.0]
    g[1] = [2 * 4.0 / H, 2 * 1.2 / H, 1.0]
    acc = np.zeros(3, np.float32)
    cnt = np.zeros(3, np.int64)
    D.accumulate(g, np.array([True, True, False]), W, H, acc, cnt)
    D.accumulate(g, np.array([True, False, False]), W, H, acc, cnt)
    np.testing.assert_allclose(acc, [10.0, 1.3, 0.0], rtol=1e-6)
    assert cnt.tolist() == [2, 1, 0]
