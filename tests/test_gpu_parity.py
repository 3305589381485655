"""GPU <-> oracle parity, stage by stage, through the C ABI.

Both sides get identical seeded inputs from gs_inputs.  Tolerances (tests/_tol.py):
  * integer, index and key outputs (radius, rect, count, keys, ids, ranges,
    n_contrib): bit-exact;
  * projected records, images, T_final: bit-exact (the frozen fp32 sequence; the
    stated 1e-5 absolute is asserted too);
  * 2D and parameter gradients: within 1e-4 relative with an absolute floor of
    1e-6 x the largest magnitude of the same plane (the quaternion planes of an
    isotropic scene take the covariance chain's floor, see tests/_tol.py);
  * Adam: |dp| <= 1e-5 |p_ref| + 1e-7.
"""
import numpy as np
import pytest

import gs_inputs as gi
import oracle
from _grad2d import moments_to_partials
from _tol import DSSIM_FLOOR, adam_close, adam_defined, grad_close, isotropic

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"


# ----------------------------------------------------------------------------- helpers

def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _partials(tr, n, conic):
    """The GPU's grad2d of Gaussians [0, n) as the nine 2D partials (header layout)."""
    return moments_to_partials(gs.grad2d_planes(tr.grad2d, n), conic[:n])


def _grad_close(got, ref, what="", iso=False, **kw):
    return grad_close(got, ref, isotropic_scene=iso, what=what, **kw)


def _scene(name, n=None, seed=0):
    cfg = gi.CONFIGS[name]
    P = gi.scene_for(cfg, seed=seed, n=n)
    return cfg, P, (n or cfg.n)


def _cam_for(cfg, view=0, W=None, H=None):
    if cfg.kind == "cube":
        return gi.camera((0.0, 0.0, 3.0), W or cfg.width, H or cfg.height)
    cams = gi.fibonacci_cameras(cfg.n_views, W or cfg.width, H or cfg.height)
    return cams[view]


def _gpu_forward(P, n, cam, capacity=1 << 20):
    W, H = cam["width"], cam["height"]
    tr = gs.Trainer(P, n, W, H, capacity=capacity, lr_plane=gi.lr_planes())
    tr.forward(cam)
    torch.cuda.synchronize()
    return tr


CASES = [
    ("tiny", None, None, None),          # 4,096 Gaussians, 128x128
    ("tiny", 3000, 72, 56),              # ragged tiles on both axes, n not a multiple of 256
    ("iso1m_512", 60_000, 256, 192),     # isosurface generator at reduced size
]


@pytest.fixture(scope="module", params=CASES, ids=[f"{c[0]}-{c[1]}-{c[2]}x{c[3]}" for c in CASES])
def case(request):
    name, n, W, H = request.param
    cfg, P, n = _scene(name, n)
    cam = _cam_for(cfg, 3 if cfg.kind != "cube" else 0, W, H)
    ref_proj = oracle.project(P, n, cam, 32)
    tr = _gpu_forward(P, n, cam)
    return {"cfg": cfg, "P": P, "n": n, "cam": cam, "ref_proj": ref_proj, "tr": tr, "iso": isotropic(P, n)}


# ----------------------------------------------------------------------------- exp

def test_expf_bitwise_equal_to_oracle():
    x = np.concatenate([np.linspace(-90, 90, 200_001, dtype=np.float32),
                        np.random.default_rng(0).uniform(-6, 0, 100_000).astype(np.float32),
                        np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 88.0, -87.0], np.float32)])
    xd = torch.from_numpy(x).to(DEV)
    yd = torch.empty_like(xd)
    gs.util_expf(xd, yd)
    y = yd.cpu().numpy()
    yr = oracle.expf(x)
    same = (y.view(np.uint32) == yr.view(np.uint32)) | (np.isnan(y) & np.isnan(yr))
    assert same.all(), x[~same][:10]


# ----------------------------------------------------------------------------- projection

def test_project_parity(case):
    tr, ref, n = case["tr"], case["ref_proj"], case["n"]
    assert tr.check_status() == 0
    count = _u32(tr.proj.count)[:n]
    np.testing.assert_array_equal(count, ref["count"])
    vis = ref["count"] > 0
    assert vis.sum() > 0.5 * n
    np.testing.assert_array_equal(tr.proj.radius.cpu().numpy()[:n][vis], ref["radius"][vis])
    rect = _u32(tr.proj.rect)[:n]
    r = ref["rect"]
    np.testing.assert_array_equal(rect[vis, 0], (r[vis, 0] | (r[vis, 1] << 16)).astype(np.uint32))
    np.testing.assert_array_equal(rect[vis, 1], (r[vis, 2] | (r[vis, 3] << 16)).astype(np.uint32))
    depth = tr.proj.depth.cpu().numpy()[:n]
    np.testing.assert_array_equal(depth[vis].view(np.uint32), ref["depth"][vis].view(np.uint32))
    rec = tr.proj.rec.cpu().numpy()[:n]
    exp = np.stack([ref["mean2d"][:, 0], ref["mean2d"][:, 1], -0.5 * ref["conic"][:, 0], -ref["conic"][:, 1],
                    -0.5 * ref["conic"][:, 2], ref["opacity"], ref["rgb"][:, 0], ref["rgb"][:, 1],
                    ref["rgb"][:, 2]], 1).astype(np.float32)
    got = rec[:, :9]
    assert np.max(np.abs(got[vis] - exp[vis])) <= 1e-5 * np.maximum(1, np.abs(exp[vis])).max()
    exact = np.mean(got[vis].view(np.uint32) == exp[vis].view(np.uint32))
    assert exact == 1.0, f"only {exact:.6f} of projected record values are bit-exact"
    np.testing.assert_array_equal(rec[vis, 9].view(np.uint32), np.nonzero(vis)[0].astype(np.uint32))
    # the record's last slot carries the depth (the binning's sort keys read it there)
    np.testing.assert_array_equal(rec[vis, 11].view(np.uint32), ref["depth"][vis].view(np.uint32))


# ----------------------------------------------------------------------------- binning

def test_bin_sort_parity(case):
    tr, ref, cam = case["tr"], case["ref_proj"], case["cam"]
    tl = oracle.tile_lists(ref, cam["width"], cam["height"])
    K = tr.n_isect()
    assert K == tl["K"]
    keys = tr.bins.keys.cpu().numpy()[:K].view(np.uint64)
    ids = _u32(tr.bins.ids)[:K]
    np.testing.assert_array_equal(keys, tl["keys"])
    np.testing.assert_array_equal(ids, tl["ids"])
    # non-empty tiles: identical [start, end); empty tiles: [0, 0) by the ABI's convention
    rg = _u32(tr.bins.ranges)
    nonempty = tl["ranges"][:, 1] > tl["ranges"][:, 0]
    np.testing.assert_array_equal(rg[nonempty], tl["ranges"][nonempty])
    assert np.all(rg[~nonempty] == 0)
    # records gathered into key order are the projected records of those ids
    srec = tr.bins.rec.cpu().numpy()[:K]
    prec = tr.proj.rec.cpu().numpy()
    np.testing.assert_array_equal(srec.view(np.uint32), prec[ids].view(np.uint32))


def test_bin_sort_deterministic(case):
    tr, cam = case["tr"], case["cam"]
    keys0 = tr.bins.keys.clone()
    ids0 = tr.bins.ids.clone()
    img0 = tr.image.clone()
    tr.forward(cam)
    torch.cuda.synchronize()
    K = tr.n_isect()
    assert torch.equal(tr.bins.keys[:K], keys0[:K])
    assert torch.equal(tr.bins.ids[:K], ids0[:K])
    assert torch.equal(tr.image, img0)


def _depth_scene(depths, seed):
    """The tiny scene with its means moved to the given camera depths, inside the
    field of view, for the camera at (0, 0, 3) looking at the origin."""
    cfg = gi.CONFIGS["tiny"]
    n = len(depths)
    P = gi.scene_for(cfg, n=n, seed=seed).copy()
    cam = gi.camera((0.0, 0.0, 3.0), 128, 128)
    rng = np.random.default_rng(seed)
    xy = rng.uniform(-0.4, 0.4, (n, 2)) * depths[:, None]
    c = np.stack([xy[:, 0], xy[:, 1], depths], 1)
    R = cam["R"].astype(np.float64)
    t = cam["t"].astype(np.float64)
    P[0:3, :n] = ((c - t) @ R).T.astype(np.float32)  # world = R^T (c - t)
    P[3:6, :n] = np.log(0.004 * depths)[None, :].astype(np.float32)  # a few pixels wide at any depth
    return P, n, cam


@pytest.mark.parametrize("span", ["wide", "narrow"])
def test_bin_sort_depth_ranges(span):
    """Depths over four decades make every depth digit vary; depths within a few
    ulps of 3 leave the upper three digits constant, so those passes are identities.
    Both must give the oracle's keys and ids."""
    rng = np.random.default_rng(5)
    if span == "wide":
        d = np.exp(rng.uniform(np.log(0.05), np.log(500.0), 3000))
    else:
        d = 3.0 + rng.integers(-40, 40, 3000) * 2.4e-7  # +-40 ulps of 3
    P, n, cam = _depth_scene(d, 6)
    ref = oracle.project(P, n, cam, 32)
    vis = ref["count"] > 0
    assert vis.sum() > 2000
    bits = ref["depth"][vis].view(np.uint32).astype(np.int64)
    spread = int(bits.max() - bits.min())
    assert spread >= (1 << 24) if span == "wide" else spread < (1 << 8)
    tr = _gpu_forward(P, n, cam)
    tl = oracle.tile_lists(ref, cam["width"], cam["height"])
    K = tr.n_isect()
    assert K == tl["K"] and tr.check_status() == 0
    np.testing.assert_array_equal(tr.bins.keys.cpu().numpy()[:K].view(np.uint64), tl["keys"])
    np.testing.assert_array_equal(_u32(tr.bins.ids)[:K], tl["ids"])


# ----------------------------------------------------------------------------- forward

def test_render_fwd_parity(case):
    tr, ref, cam = case["tr"], case["ref_proj"], case["cam"]
    rd = oracle.render(ref, cam["width"], cam["height"])
    img = tr.image.cpu().numpy()
    assert np.max(np.abs(img - rd["image"])) <= 1e-5
    assert np.max(np.abs(tr.T_final.cpu().numpy() - rd["T_final"])) <= 1e-5
    np.testing.assert_array_equal(_u32(tr.n_contrib), rd["n_contrib"])
    assert np.array_equal(img.view(np.uint32), rd["image"].view(np.uint32)), "image not bit-exact"


def test_render_fwd_counted_parity(case):
    """The counting forward: the same image, T_final and n_contrib bit for bit, and
    each pixel's count of composited entries equal to the oracle's."""
    tr, ref, cam = case["tr"], case["ref_proj"], case["cam"]
    W, H = cam["width"], cam["height"]
    rd = oracle.render(ref, W, H, count_used=True)
    img = torch.empty_like(tr.image)
    T = torch.empty_like(tr.T_final)
    nc = torch.empty_like(tr.n_contrib)
    nu = torch.full_like(tr.n_contrib, -1)
    st = _status()
    gs.render_fwd_counted(cam, tr.bins, tr.bg, img, T, nc, nu, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(_u32(img), rd["image"].view(np.uint32))
    np.testing.assert_array_equal(_u32(T), rd["T_final"].view(np.uint32))
    np.testing.assert_array_equal(_u32(nc), rd["n_contrib"])
    np.testing.assert_array_equal(_u32(nu), rd["n_used"])
    assert (rd["n_used"] <= rd["n_contrib"]).all() and rd["n_used"].sum() > 0


def test_render_fwd_overflowing_colour():
    """A Gaussian whose SH coefficients are finite but whose colour sum overflows to
    +inf (every coefficient of the red channel 3e38 with the sign of its basis value):
    the projection flags nothing, the pixels that composite it turn to inf, and every
    other pixel, the entry's neighbours in the same walk included, is untouched, bit
    for bit as the oracle renders it."""
    cfg = gi.CONFIGS["tiny"]
    n = 300
    P = gi.scene_for(cfg, n=n, seed=3).copy()
    cam = gi.camera((0.0, 0.0, 3.0), 128, 128)
    P[0:3, 0] = [0.02, -0.01, 0.0]
    P[3:6, 0] = np.log(0.05)
    P[10, 0] = 3.0
    d = P[0:3, 0].astype(np.float64) - cam["campos"].astype(np.float64)
    Y = oracle.sh_basis((d / np.linalg.norm(d))[None, :].astype(np.float32))[0]
    for k in range(16):
        P[11 + 3 * k, 0] = np.float32(3.0e38) * (1.0 if Y[k] >= 0 else -1.0) if abs(Y[k]) > 1e-3 else 0.0
    ref = oracle.project(P, n, cam, 32)
    assert np.isinf(ref["rgb"][0, 0]) and ref["visible"][0]
    rd = oracle.render(ref, 128, 128)
    assert np.isinf(rd["image"]).sum() > 50 and np.isfinite(rd["image"]).sum() > 40000
    tr = _gpu_forward(P, n, cam)
    assert tr.check_status() == 0
    np.testing.assert_array_equal(_u32(tr.image), rd["image"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.T_final), rd["T_final"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.n_contrib), rd["n_contrib"])


# ----------------------------------------------------------------------------- backward

def _target_for(case):
    cam = case["cam"]
    rd = oracle.render(case["ref_proj"], cam["width"], cam["height"])
    return gi.offset_target(rd["image"], seed=7)


def test_render_bwd_parity(case):
    tr, ref, cam, n = case["tr"], case["ref_proj"], case["cam"], case["n"]
    W, H = cam["width"], cam["height"]
    target = _target_for(case)
    rd = oracle.render(ref, W, H, target=target)
    tgt = torch.from_numpy(target).to(DEV)
    tr.forward(cam)
    tr.backward(cam, tgt)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    _grad_close(_partials(tr, n, ref["conic"]), rd["grad2d"], what="grad2d")
    assert abs(float(tr.loss.item()) - rd["loss"]) <= 1e-5 * rd["loss"]
    # padding gets no gradient
    assert not tr.grad2d[n:].any()


def test_project_bwd_parity(case):
    """Seeded stand-in 2D sums fed to both sides isolate the chain rule (the oracle
    gets them as the partials the header's layout defines)."""
    tr, P, cam, n = case["tr"], case["P"], case["cam"], case["n"]
    g2 = gi.random_grad2d(11, n, P.shape[1])
    ref = oracle.project_bwd(P, n, cam, moments_to_partials(g2[:, :n], case["ref_proj"]["conic"][:n]), prec=32)
    g2d = torch.from_numpy(gs.grad2d_interleaved(g2)).to(DEV)
    st = _status()
    gs.project(n, tr.params, cam, tr.proj, st)
    gs.project_bwd(n, tr.params, cam, tr.proj, g2d, tr.grads, st)
    torch.cuda.synchronize()
    got = tr.grads.cpu().numpy()
    _grad_close(got[:, :n], ref, what="param grads", iso=case["iso"])
    assert not np.any(got[:, n:])


def test_adam_parity():
    rng = np.random.default_rng(5)
    n, n_pad = 1000, 1024
    p = rng.normal(size=(59, n_pad)).astype(np.float32)
    g = (rng.normal(size=(59, n_pad)) * 10.0 ** rng.integers(-7, 0, (59, n_pad))).astype(np.float32)
    m = (rng.normal(size=(59, n_pad)) * 1e-3).astype(np.float32)
    v = (rng.uniform(size=(59, n_pad)) * 1e-6).astype(np.float32)
    lr = gi.lr_planes()
    t = 5
    pr, mr, vr = oracle.adam(p.astype(np.float64), g.astype(np.float64), m.astype(np.float64),
                             v.astype(np.float64), lr, 0.9, 0.999, 1e-15, t)
    pd, gd, md, vd = (torch.from_numpy(a.copy()).to(DEV) for a in (p, g, m, v))
    gs.adam_step(n, pd, gd, md, vd, lr, 0.9, 0.999, 1e-15, t)
    torch.cuda.synchronize()
    adam_close(pd.cpu().numpy(), pr)
    # where the 1e-7 floor is below 1e-5 |p| (|p| >= 0.01, almost every entry), the
    # relative bound holds on its own
    big = np.abs(pr) >= 1e-2
    assert big.mean() > 0.9
    rel = np.abs(pd.cpu().numpy().astype(np.float64) - pr)[big] / np.abs(pr)[big]
    assert rel.max() <= 1e-5, rel.max()
    # moments: one fp32 multiply-add each, so the error is bounded by a few ulp of the
    # larger of the two terms (the result itself may cancel to near zero)
    g64, m64, v64 = g.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    assert np.all(np.abs(md.cpu().numpy() - mr) <= 1e-6 * (np.abs(0.9 * m64) + np.abs(0.1 * g64)) + 1e-30)
    assert np.all(np.abs(vd.cpu().numpy() - vr) <= 1e-6 * (np.abs(0.999 * v64) + np.abs(0.001 * g64 * g64)) + 1e-30)


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_whole_step_end_to_end(case, fused):
    """The whole chain from the same parameters: every stage against the oracle's
    chain; Adam is compared where the gradient is not within its tolerance of 0
    (at t = 1 an update is lr sign(g), so a near-zero g has no defined sign).
    ``fused`` runs the projection backward and Adam as gs_project_bwd_adam."""
    P, cam, n = case["P"], case["cam"], case["n"]
    W, H = cam["width"], cam["height"]
    target = _target_for(case)
    z = np.zeros((59, P.shape[1]))
    ref = oracle.step(P, n, cam, target, z, z, 1, gi.lr_planes())
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes(), fused=fused)
    tr.step(cam, torch.from_numpy(target).to(DEV))
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    _grad_close(_partials(tr, n, case["ref_proj"]["conic"]), ref["render"]["grad2d"], what="grad2d")
    gref = ref["grads"][:, :n]
    if fused:
        # the fused kernel writes no gradient planes; at t = 1 from zero moments
        # m = (1 - beta1) g, with 1 - beta1 rounded to fp32 once
        _grad_close(tr.m.cpu().numpy()[:, :n] / np.float64(np.float32(0.1)), gref, what="fused m = 0.1 g",
                    iso=case["iso"])
    else:
        _grad_close(tr.grads.cpu().numpy()[:, :n], gref, what="param grads", iso=case["iso"])
    # the sign of g (hence the t = 1 update) is certain where |g| exceeds the gradient
    # tolerance many times over
    defined = adam_defined(gref, case["iso"])
    assert defined.mean() > 0.2
    adam_close(tr.params.cpu().numpy()[:, :n], ref["params"][:, :n], defined)
    # padding is never moved
    assert not tr.params[:, n:].any()


def test_fused_project_bwd_adam_equals_separate_calls(case):
    """gs_project_bwd_adam applies the same fp32 arithmetic as gs_project_bwd then
    gs_adam_step: parameters and moments agree to an ulp or so, over three steps
    with nonzero moments (seeded 2D gradients as input)."""
    P, cam, n = case["P"], case["cam"], case["n"]
    n_pad = P.shape[1]
    W, H = cam["width"], cam["height"]
    lr = gi.lr_planes()
    a = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=lr, fused=False)
    b = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=lr, fused=True)
    st = _status()
    for t in range(1, 4):
        g2 = torch.from_numpy(gs.grad2d_interleaved(gi.random_grad2d(100 + t, n, n_pad))).to(DEV)
        gs.project(n, a.params, cam, a.proj, st)
        gs.project_bwd(n, a.params, cam, a.proj, g2, a.grads, st)
        gs.adam_step(n, a.params, a.grads, a.m, a.v, lr, 0.9, 0.999, 1e-15, t)
        gs.project(n, b.params, cam, b.proj, st)
        gs.project_bwd_adam(n, b.params, cam, b.proj, g2, b.m, b.v, lr, 0.9, 0.999, 1e-15, t, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y in ((a.params, b.params), (a.m, b.m), (a.v, b.v)):
        x, y = x.cpu().numpy().astype(np.float64), y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(x - y) <= 4e-7 * np.abs(x) + 1e-30)


# ----------------------------------------------------------------------------- D-SSIM

def _ssim_gpu(x, y, lam):
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(DEV)
    yd = torch.from_numpy(np.ascontiguousarray(y, np.float32)).to(DEV)
    _, H, W = x.shape
    maps = torch.full((gs.SSIM_MAPS, H, W), float("nan"), dtype=torch.float32, device=DEV)
    s = torch.full((1,), float("nan"), dtype=torch.float32, device=DEV)
    g = torch.full((3, H, W), float("nan"), dtype=torch.float32, device=DEV)
    gs.ssim_fwd(xd, yd, lam, maps, s)
    gs.ssim_bwd(xd, yd, maps, g)
    torch.cuda.synchronize()
    return float(s.item()), g.cpu().numpy().astype(np.float64)


def _ssim_grad_close(got, ref, lam, P):
    """fp32 against fp64.  The gradient's natural unit is lambda / (3 P).  The kernels
    take the window moments about a per-tile shift and fold the local means in about
    a shift too, so flat regions cancel exactly.  Elsewhere single terms of the
    filtered sums are large: the luminance factor divides by mu_x^2 + mu_y^2 + C1 >=
    1e-4 and the contrast-structure factor by the variances + C2 >= 9e-4, so in dark
    or smooth regions a term reaches hundreds of units while their sum is far smaller,
    and 121-tap fp32 sums of them keep about 1e-5 of the image's largest gradient.
    Allowed: 1e-4 relative plus 1e-4 of the larger of the unit and the largest
    gradient magnitude (the 2D-gradient tests scale their floor with the group's
    largest value the same way)."""
    unit = lam / (3.0 * P)
    tol = 1e-4 * np.abs(ref) + 1e-4 * max(unit, float(np.abs(ref).max()))
    bad = ~(np.abs(got - ref) <= tol)
    assert not bad.any(), (int(bad.sum()), float(np.nanmax(np.abs(got - ref) / unit)), float(np.abs(ref).max() / unit))


SSIM_SHAPES = [(37, 53), (128, 128), (5, 7), (1, 1), (300, 200)]


@pytest.mark.parametrize("H,W", SSIM_SHAPES, ids=[f"{h}x{w}" for h, w in SSIM_SHAPES])
def test_ssim_parity_random_images(H, W):
    """Mean SSIM within 1e-5 and the gradient of lambda (1 - SSIM) per value, on
    seeded images with ragged 16x16 tiles, images smaller than the window and a
    single pixel."""
    rng = np.random.default_rng(H * 1000 + W)
    x = rng.uniform(0, 1, (3, H, W)).astype(np.float32)
    y = np.clip(x + rng.normal(0, 0.15, x.shape), 0, 1).astype(np.float32)
    s_ref, g_ref = oracle.ssim(x, y, 0.2)
    s, g = _ssim_gpu(x, y, 0.2)
    assert abs(s - s_ref) <= 1e-5, (s, s_ref)
    _ssim_grad_close(g, g_ref, 0.2, H * W)


def test_ssim_identical_and_flat_images():
    """SSIM(x, x) = 1 with zero gradient (its maximum), on a textured image and on a
    flat one (variances exactly zero); a flat image against a different flat image."""
    rng = np.random.default_rng(3)
    x = rng.uniform(0, 1, (3, 40, 24)).astype(np.float32)
    for a, b in ((x, x), (np.full_like(x, 0.3), np.full_like(x, 0.3)), (np.full_like(x, 0.3), np.full_like(x, 0.7))):
        s_ref, g_ref = oracle.ssim(a, b, 0.2)
        s, g = _ssim_gpu(a, b, 0.2)
        assert abs(s - s_ref) <= 1e-5, (s, s_ref)
        _ssim_grad_close(g, g_ref, 0.2, a.shape[1] * a.shape[2])


def test_ssim_parity_on_renders(case):
    """The images the step feeds it: a render against its offset target."""
    cam = case["cam"]
    W, H = cam["width"], cam["height"]
    img = oracle.render(case["ref_proj"], W, H)["image"]
    tgt = _target_for(case)
    s_ref, g_ref = oracle.ssim(img, tgt, 0.2)
    s, g = _ssim_gpu(img, tgt, 0.2)
    assert abs(s - s_ref) <= 1e-5, (s, s_ref)
    _ssim_grad_close(g, g_ref, 0.2, W * H)


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_whole_step_with_dssim_end_to_end(case, fused):
    """(1 - lambda) L1 + lambda (1 - SSIM) with lambda = 0.2: loss, 2D gradients and
    the Adam update against the oracle's step with the same objective."""
    P, cam, n = case["P"], case["cam"], case["n"]
    W, H = cam["width"], cam["height"]
    target = _target_for(case)
    z = np.zeros((59, P.shape[1]))
    ref = oracle.step(P, n, cam, target, z, z, 1, gi.lr_planes(), dssim=0.2)
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes(), fused=fused, dssim=0.2)
    tr.step(cam, torch.from_numpy(target).to(DEV))
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    assert abs(tr.total_loss() - ref["render"]["loss"]) <= 1e-5 * abs(ref["render"]["loss"])
    assert abs(float(tr.ssim_val.item()) - ref["render"]["ssim"]) <= 1e-5
    _grad_close(_partials(tr, n, case["ref_proj"]["conic"]), ref["render"]["grad2d"], what="grad2d")
    gref = ref["grads"][:, :n]
    # the parameter gradients inherit the SSIM image gradient's fp32 error (tests/_tol.py)
    if fused:
        _grad_close(tr.m.cpu().numpy()[:, :n] / np.float64(np.float32(0.1)), gref, what="fused m = 0.1 g",
                    iso=case["iso"], floor=DSSIM_FLOOR)
    else:
        _grad_close(tr.grads.cpu().numpy()[:, :n], gref, what="param grads", iso=case["iso"], floor=DSSIM_FLOOR)
    defined = adam_defined(gref, case["iso"])
    assert defined.mean() > 0.2
    adam_close(tr.params.cpu().numpy()[:, :n], ref["params"][:, :n], defined)


def test_render_bwd_extra_image_gradient(case):
    """The render backward driven only by a given dL/dC image (L1 weight 0): the 2D
    gradients are the oracle's for the same image gradient, and the loss is 0."""
    tr, ref, cam, n = case["tr"], case["ref_proj"], case["cam"], case["n"]
    W, H = cam["width"], cam["height"]
    target = _target_for(case)
    extra = np.random.default_rng(21).normal(0.0, 1.0 / (3 * W * H), (3, H, W)).astype(np.float32)
    rd = oracle.render(ref, W, H, target=target, l1_weight=0.0, dLdC_extra=extra)
    tr.forward(cam)
    st = _status()
    gs.render_bwd(n, tr.n_pad, cam, tr.bins, tr.bg, tr.image, torch.from_numpy(target).to(DEV), tr.T_final,
                  tr.n_contrib, tr.grad2d, tr.loss, st, l1_weight=0.0,
                  dLdC_extra=torch.from_numpy(extra).to(DEV))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert float(tr.loss.item()) == 0.0
    _grad_close(_partials(tr, n, ref["conic"]), rd["grad2d"], what="grad2d")


@pytest.mark.parametrize("order", ["before", "after_backward"])
def test_staged_host_targets_feed_the_right_step(case, order):
    """Targets uploaded from pinned host memory through HostTargets (copy stream,
    two slots, the next upload overlapping the current step) drive the same steps as
    targets already on the device: per-step losses agree over four steps with four
    different targets, so every step read its own upload.  The next upload is enqueued
    before the current step, or after it and waiting on the step's after_backward event
    (the bench's end-to-end order)."""
    P, cam, n = case["P"], case["cam"], case["n"]
    W, H = cam["width"], cam["height"]
    base = _target_for(case)
    targets = [gi.offset_target(base, seed=40 + k) for k in range(4)]
    a = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    b = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    la, lb = [], []
    for t in targets:
        a.step(cam, torch.from_numpy(t).to(DEV))
        la.append(float(a.loss.item()))
    host = [torch.from_numpy(t).pin_memory() for t in targets]
    staged = gs.HostTargets((3, H, W), DEV)
    slot = staged.put(host[0])
    loss_b = torch.empty((4,), dtype=torch.float32).pin_memory()
    for k in range(4):
        if order == "before":
            nxt = staged.put(host[k + 1]) if k + 1 < 4 else None
            b.step_staged(cam, staged, slot)
        else:
            b.step_staged(cam, staged, slot)
            nxt = staged.put(host[k + 1], after=b.after_backward) if k + 1 < 4 else None
        loss_b[k:k + 1].copy_(b.loss, non_blocking=True)
        slot = nxt
    torch.cuda.synchronize()
    lb = loss_b.tolist()
    assert a.check_status() == 0 and b.check_status() == 0
    assert len(set(round(x, 6) for x in la)) == 4
    np.testing.assert_allclose(lb, la, rtol=1e-5)


def _batch_cams(case, B=3):
    cfg, cam = case["cfg"], case["cam"]
    W, H = cam["width"], cam["height"]
    if cfg.kind == "cube":
        return [gi.camera(pos, W, H) for pos in ((0.0, 0.0, 3.0), (0.6, -0.4, 2.8), (-0.5, 0.5, 2.9))][:B]
    cams = gi.fibonacci_cameras(cfg.n_views, W, H)
    return [cams[k] for k in (3, 9, 20)][:B]


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_batch_step_matches_oracle(case, fused):
    """A step over three views ("Scaling 3D Gaussian Splatting with Distributed
    Compute", batch-size section): the mean of the view losses, gradients summed
    through gs_project_bwd_accumulate (or, fused, added inside gs_project_bwd_adam),
    one Adam step with lr sqrt(3), eps / sqrt(3) and betas 1 - 3 (1 - beta)."""
    P, n = case["P"], case["n"]
    cams = _batch_cams(case)
    targets = [gi.offset_target(oracle.render(oracle.project(P, n, c, 32), c["width"], c["height"])["image"],
                                seed=60 + k) for k, c in enumerate(cams)]
    z = np.zeros((59, P.shape[1]))
    ref = oracle.step_batch(P, n, cams, targets, z, z, 1, gi.lr_planes())
    W, H = cams[0]["width"], cams[0]["height"]
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes(), fused=fused)
    tr.step_batch(cams, [torch.from_numpy(t).to(DEV) for t in targets])
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    assert abs(tr.batch_loss() - ref["loss"]) <= 1e-5 * ref["loss"]
    gref = ref["grads"][:, :n]
    if not fused:
        _grad_close(tr.grads.cpu().numpy()[:, :n], gref, what="batch grads", iso=case["iso"])
    defined = adam_defined(gref, case["iso"])
    assert defined.mean() > 0.2
    adam_close(tr.params.cpu().numpy()[:, :n], ref["params"][:, :n], defined)
    assert not tr.params[:, n:].any()


def test_batch_of_one_is_the_single_view_step(case):
    """step_batch with one view runs the same calls as step: the same loss, and the
    same parameters wherever the gradient's sign is certain (elsewhere the first Adam
    step, lr sign(g), follows the atomics' summation order)."""
    P, cam, n = case["P"], case["cam"], case["n"]
    W, H = cam["width"], cam["height"]
    target = _target_for(case)
    tgt = torch.from_numpy(target).to(DEV)
    a = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    b = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    a.step(cam, tgt)
    b.step_batch([cam], [tgt])
    torch.cuda.synchronize()
    # the loss is summed with one fp32 atomic per warp, in no fixed order: two runs of
    # the same step agree to a few ulps of the sum of 512 warp partials, within the
    # 1e-5 relative the oracle comparisons allow
    assert abs(b.batch_loss() - float(a.loss.item())) <= 1e-5 * float(a.loss.item())
    z = np.zeros((59, P.shape[1]))
    gref = oracle.step(P, n, cam, target, z, z, 1, gi.lr_planes())["grads"][:, :n]
    defined = adam_defined(gref, case["iso"])
    assert defined.mean() > 0.2
    x = a.params.cpu().numpy()[:, :n].astype(np.float64)
    y = b.params.cpu().numpy()[:, :n].astype(np.float64)
    bad = (np.abs(x - y) > 1e-6 * np.abs(x) + 1e-7) & defined
    assert not bad.any(), bad.sum()


def test_device_step_count_equals_host_step_count(case):
    """gs_project_bwd_adam_tdev forms lr / (1 - beta1^t) and 1 / sqrt(1 - beta2^t)
    from a step count in device memory in fp64, as gs_project_bwd_adam does on the
    host: on identical seeded 2D gradients over three steps (t = 1, 2, 3) the
    parameters and moments agree to an ulp."""
    P, cam, n = case["P"], case["cam"], case["n"]
    n_pad = P.shape[1]
    W, H = cam["width"], cam["height"]
    lr = gi.lr_planes()
    a = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=lr)
    b = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=lr)
    st = _status()
    t_dev = torch.zeros(1, dtype=torch.int64, device=DEV)
    for t in range(1, 4):
        g2 = torch.from_numpy(gs.grad2d_interleaved(gi.random_grad2d(200 + t, n, n_pad))).to(DEV)
        gs.project(n, a.params, cam, a.proj, st)
        gs.project_bwd_adam(n, a.params, cam, a.proj, g2, a.m, a.v, lr, 0.9, 0.999, 1e-15, t, st)
        gs.project(n, b.params, cam, b.proj, st)
        gs.step_counter_add(t_dev, 1)
        gs.project_bwd_adam_tdev(n, b.params, cam, b.proj, g2, b.m, b.v, lr, 0.9, 0.999, 1e-15, t_dev, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(t_dev.item()) == 3
    for x, y in ((a.params, b.params), (a.m, b.m), (a.v, b.v)):
        x, y = x.cpu().numpy().astype(np.float64), y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(x - y) <= 2.5e-7 * np.abs(x) + 1e-30)


def test_graph_replayed_steps_match_eager_steps(case):
    """Steps captured as CUDA graphs (camera, target and hyperparameters fixed at
    capture, the step count advanced and read on the device) replay the eager steps:
    four steps over three views after one eager step give the same losses (each
    step's loss depends on all parameters the earlier steps moved)."""
    P, n = case["P"], case["n"]
    cams = _batch_cams(case)
    W, H = cams[0]["width"], cams[0]["height"]
    tg = [torch.from_numpy(gi.offset_target(oracle.render(oracle.project(P, n, c, 32), W, H)["image"],
                                            seed=80 + k)).to(DEV) for k, c in enumerate(cams)]
    a = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    b = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    a.step(cams[0], tg[0])
    b.step(cams[0], tg[0])
    graphs = [b.capture_step(c, t) for c, t in zip(cams, tg)]
    order = [1, 2, 0, 1]
    la, lb = [], []
    for k in order:
        a.step(cams[k], tg[k])
        la.append(float(a.loss.item()))
        b.replay(graphs[k])
        lb.append(float(b.loss.item()))
    assert a.check_status() == 0 and b.check_status() == 0
    assert b.t == a.t == 5 and int(b.t_dev.item()) == 5
    np.testing.assert_allclose(lb, la, rtol=1e-5)


def test_render_on_a_coloured_background():
    """Forward and backward on a coloured background against the oracle: image,
    T_final and n_contrib bit for bit, the loss and the 2D gradients within tolerance.
    What shows through (T_final bg) depends on every composited alpha, and the
    backward's carried colour starts at the background."""
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg)
    n, W, H = cfg.n, cfg.width, cfg.height
    cam = _cam_for(cfg)
    bg = (0.3, 0.6, 0.1)
    ref = oracle.project(P, n, cam, 32)
    target = gi.offset_target(oracle.render(ref, W, H, bg=bg)["image"], seed=7)
    rd = oracle.render(ref, W, H, bg=bg, target=target)
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes(), bg=bg)
    tr.forward(cam)
    tr.loss_backward(cam, torch.from_numpy(target).to(DEV))
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    np.testing.assert_array_equal(_u32(tr.image), rd["image"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.T_final), rd["T_final"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.n_contrib), rd["n_contrib"])
    assert abs(float(tr.loss.item()) - rd["loss"]) <= 1e-5 * rd["loss"]
    _grad_close(_partials(tr, n, ref["conic"]), rd["grad2d"], what="grad2d (coloured background)")


# ----------------------------------------------------------------------------- edge cases

def test_empty_scene_all_culled():
    """Every Gaussian behind the camera: K = 0, background image, zero gradients."""
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg, n=500)
    P[2, :500] = 50.0          # far behind the camera at z = +3 looking down -z
    cam = gi.camera((0.0, 0.0, 3.0), 64, 48)
    tgt = torch.zeros((3, 48, 64), device=DEV)
    for fused in (False, True):
        tr = gs.Trainer(P, 500, 64, 48, capacity=1024, lr_plane=gi.lr_planes(), bg=(0.2, 0.4, 0.6), fused=fused)
        p0 = tr.params.clone()
        tr.step(cam, tgt)
        torch.cuda.synchronize()
        assert tr.check_status() == 0
        assert tr.n_isect() == 0
        img = tr.image.cpu().numpy()
        np.testing.assert_array_equal(img[0], np.float32(0.2))
        np.testing.assert_array_equal(img[2], np.float32(0.6))
        if not fused:
            assert not tr.grads.any()
        # zero gradients: zero moments, parameters unchanged
        assert not tr.m.any() and not tr.v.any()
        assert torch.equal(tr.params, p0)


def test_capacity_overflow_is_flagged_not_written():
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg)
    cam = _cam_for(cfg)
    tr = gs.Trainer(P, cfg.n, 128, 128, capacity=1000, lr_plane=gi.lr_planes())
    guard = torch.full((4096,), -7, dtype=torch.int64, device=DEV)   # allocated after the bins
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() & gs.GS_ERR_CAPACITY
    assert tr.n_isect() > 1000
    assert torch.all(guard == -7)


def test_nonfinite_parameters_are_flagged_and_culled():
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg, n=600)
    P[0, 5] = np.nan
    P[4, 9] = np.inf
    P[20, 11] = np.nan     # an SH coefficient
    cam = _cam_for(cfg)
    tr = _gpu_forward(P, 600, cam)
    assert tr.check_status() & gs.GS_ERR_NONFINITE
    count = _u32(tr.proj.count)
    assert count[5] == 0 and count[9] == 0 and count[11] == 0
    ref = oracle.project(P, 600, cam, 32)
    np.testing.assert_array_equal(count[:600], ref["count"])
    assert np.isfinite(tr.image.cpu().numpy()).all()


def test_large_gaussian_spanning_many_tiles():
    """One Gaussian covering the whole image plus small ones: long per-Gaussian key
    runs and a tile list longer than one shared-memory batch."""
    cam = gi.camera((0.0, 0.0, 3.0), 200, 120)
    rng = np.random.default_rng(3)
    n = 900
    means = np.column_stack([rng.uniform(-0.8, 0.8, n), rng.uniform(-0.5, 0.5, n), rng.uniform(-0.1, 0.1, n)])
    ls = np.full((n, 3), -2.6)
    ls[0] = 0.3      # huge
    q = np.tile([1.0, 0, 0, 0], (n, 1))
    logits = rng.normal(-1.5, 0.3, n)       # low opacity: long lists before termination
    sh = np.zeros((n, 16, 3))
    sh[:, 0] = rng.uniform(-1, 1, (n, 3))
    P = gi.pack(means, ls, q, logits, sh)
    ref = oracle.project(P, n, cam, 32)
    assert ref["count"][0] == gs.n_tiles(200, 120)
    tr = _gpu_forward(P, n, cam)
    tl = oracle.tile_lists(ref, 200, 120)
    assert (np.diff(tl["ranges"], axis=1).max()) > 256
    K = tr.n_isect()
    np.testing.assert_array_equal(tr.bins.keys.cpu().numpy()[:K].view(np.uint64), tl["keys"])
    rd = oracle.render(ref, 200, 120, target=gi.offset_target(oracle.render(ref, 200, 120)["image"], 2))
    assert np.array_equal(tr.image.cpu().numpy().view(np.uint32), rd["image"].view(np.uint32))
    tgt = torch.from_numpy(gi.offset_target(oracle.render(ref, 200, 120)["image"], 2)).to(DEV)
    tr.backward(cam, tgt)
    torch.cuda.synchronize()
    _grad_close(_partials(tr, n, ref["conic"]), rd["grad2d"], what="grad2d")


# ----------------------------------------------------------------------------- bounded waits

@pytest.mark.parametrize("which", ["lookback", "mbarrier"])
def test_bounded_wait_runs_out_and_the_context_stays_usable(which):
    """A wait on a flag nothing sets (a look-back word never published, an mbarrier
    nothing arrives at) gives up after its limit: GS_ERR_TIMEOUT in the status word, the
    kernel returns, and the next calls on the device run normally."""
    lib = gs.load()
    st = _status()
    s = torch.cuda.current_stream().cuda_stream
    if which == "lookback":
        scratch = torch.empty(lib.gs_util_lookback_probe_bytes(), dtype=torch.uint8, device=DEV)
        r = lib.gs_util_lookback_probe(2000, scratch.data_ptr(), scratch.numel(), st.data_ptr(), s)
    else:
        r = lib.gs_util_mbarrier_probe(2000, st.data_ptr(), s)
    assert r == gs.GS_OK
    torch.cuda.synchronize()
    assert int(st.item()) & gs.GS_ERR_TIMEOUT
    # the context is usable: a forward pass runs and matches the oracle
    cfg, P, n = _scene("tiny")
    cam = _cam_for(cfg)
    tr = _gpu_forward(P, n, cam)
    rd = oracle.render(oracle.project(P, n, cam, 32), cam["width"], cam["height"])
    assert tr.check_status() == 0
    np.testing.assert_array_equal(tr.image.cpu().numpy().view(np.uint32), rd["image"].view(np.uint32))
