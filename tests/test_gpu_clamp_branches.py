"""GPU <-> oracle parity on the two branches of the method that the seeded scenes
never reach, stage by stage through the C ABI:

* alpha at the 0.99 clamp.  The compositing rule caps alpha = min(0.99, o e^power)
  (the cited 3DGS method's rule, which "Scaling 3D Gaussian Splatting with
  Distributed Compute" composites with); where the cap is active alpha depends on
  neither the opacity nor the power, so those entries pass no gradient to them.  The
  scene puts wide, nearly opaque Gaussians (logit 12) in front of the tiny scene so
  that their alpha sits at the cap over discs of pixels.
* the EWA Jacobian clamp.  The perspective Jacobian is taken at the mean with its
  abscissa and ordinate clamped to 1.3 x the half field of view; past that the
  Jacobian no longer follows the mean, and that path passes no gradient.  The scene
  puts Gaussians well beyond the limit on both axes, wide enough that their
  footprints still reach the image.

Each stage is compared as in test_gpu_parity.py: integer outputs, records, keys,
ids and images bit-exact, gradients and Adam within the tolerances of tests/_tol.py.
"""
import math

import numpy as np
import pytest

import gs_inputs as gi
import oracle
from _grad2d import moments_to_partials
from _tol import adam_close, adam_defined, grad_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"
W = H = 128


def _cam():
    return gi.camera((0.0, 0.0, 3.0), W, H)


def _world_of(cam, c):
    """World positions of camera-space points c (rows), for world = R^T (c - t)."""
    R = cam["R"].astype(np.float64)
    t = cam["t"].astype(np.float64)
    return (np.asarray(c, np.float64) - t) @ R


def _hot_scene(n_base=2000, n_hot=3):
    """The tiny scene's generator, plus n_hot isotropic Gaussians of logit 12 (o =
    0.999994) and world scale 0.26 (about 24 px sigma) at camera depth 1.5, in front of
    every other Gaussian (the base scene lies at depth 2 to 4).  With o that close to 1,
    o e^power >= 0.99 holds where power >= ln(o / 0.99), about -0.01: a disc of radius
    0.14 sigma, about 3.4 px, around each mean."""
    cam = _cam()
    base = gi.scene_for(gi.CONFIGS["tiny"], n=n_base, seed=4)
    rng = np.random.default_rng(8)
    z = 1.5
    xy = rng.uniform(-0.25, 0.25, (n_hot, 2)) * z
    c = np.column_stack([xy, np.full(n_hot, z)])
    sh = np.zeros((n_hot, 16, 3))
    sh[:, 0, :] = rng.uniform(-1, 1, (n_hot, 3))
    q = np.tile([1.0, 0.0, 0.0, 0.0], (n_hot, 1))
    hot = gi.pack(_world_of(cam, c), np.full((n_hot, 3), math.log(0.26)), q, np.full(n_hot, 12.0), sh)
    n = n_base + n_hot
    P = np.zeros((59, gi.n_pad_of(n)), np.float32)
    P[:, :n_base] = base[:, :n_base]
    P[:, n_base:n] = hot[:, :n_hot]
    return P, n, cam, np.arange(n_base, n)


def _beyond_scene(n_base=2000):
    """The tiny scene's generator, plus four isotropic Gaussians at depth 3 whose
    camera-space x / z or y / z is 1.6 x the clamp limit 1.3 tan(fov / 2), on each
    side, with world scale 0.6 (about 27 px sigma, 95 px radius) so that their
    footprints reach about 25 px into the image."""
    cam = _cam()
    base = gi.scene_for(gi.CONFIGS["tiny"], n=n_base, seed=5)
    z = 3.0
    limx = 1.3 * (0.5 * W) / float(cam["fx"])
    limy = 1.3 * (0.5 * H) / float(cam["fy"])
    c = np.array([[1.6 * limx * z, 0.1, z], [-1.6 * limx * z, -0.2, z],
                  [0.15, 1.6 * limy * z, z], [-0.1, -1.6 * limy * z, z]])
    m = c.shape[0]
    rng = np.random.default_rng(9)
    sh = np.zeros((m, 16, 3))
    sh[:, 0, :] = rng.uniform(-1, 1, (m, 3))
    sh[:, 1:, :] = rng.normal(0, 0.05, (m, 15, 3))
    q = rng.normal(size=(m, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    extra = gi.pack(_world_of(cam, c), np.full((m, 3), math.log(0.6)), q, np.array([1.0, 0.5, 0.8, 1.2]), sh)
    n = n_base + m
    P = np.zeros((59, gi.n_pad_of(n)), np.float32)
    P[:, :n_base] = base[:, :n_base]
    P[:, n_base:n] = extra[:, :m]
    return P, n, cam, np.arange(n_base, n), (limx, limy)


def _stagewise(P, n, cam, seed):
    """Every stage on the GPU against the oracle; returns the oracle projection."""
    ref = oracle.project(P, n, cam, 32)
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    # projection
    cnt = tr.proj.count.cpu().numpy().view(np.uint32)[:n]
    np.testing.assert_array_equal(cnt, ref["count"])
    vis = ref["count"] > 0
    np.testing.assert_array_equal(tr.proj.radius.cpu().numpy()[:n][vis], ref["radius"][vis])
    rec = tr.proj.rec.cpu().numpy()[:n]
    exp = np.stack([ref["mean2d"][:, 0], ref["mean2d"][:, 1], -0.5 * ref["conic"][:, 0], -ref["conic"][:, 1],
                    -0.5 * ref["conic"][:, 2], ref["opacity"], ref["rgb"][:, 0], ref["rgb"][:, 1],
                    ref["rgb"][:, 2]], 1).astype(np.float32)
    np.testing.assert_array_equal(rec[vis, :9].view(np.uint32), exp[vis].view(np.uint32))
    # binning
    tl = oracle.tile_lists(ref, W, H)
    K = tr.n_isect()
    assert K == tl["K"]
    np.testing.assert_array_equal(tr.bins.keys.cpu().numpy()[:K].view(np.uint64), tl["keys"])
    np.testing.assert_array_equal(tr.bins.ids.cpu().numpy()[:K].view(np.uint32), tl["ids"])
    # forward
    rd = oracle.render(ref, W, H)
    np.testing.assert_array_equal(tr.image.cpu().numpy().view(np.uint32), rd["image"].view(np.uint32))
    np.testing.assert_array_equal(tr.T_final.cpu().numpy().view(np.uint32), rd["T_final"].view(np.uint32))
    np.testing.assert_array_equal(tr.n_contrib.cpu().numpy().view(np.uint32), rd["n_contrib"])
    # backward
    target = gi.offset_target(rd["image"], seed=seed)
    rb = oracle.render(ref, W, H, target=target)
    tr.backward(cam, torch.from_numpy(target).to(DEV))
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    g2 = gs.grad2d_planes(tr.grad2d, n)
    grad_close(moments_to_partials(g2, ref["conic"]), rb["grad2d"], what="grad2d")
    assert abs(float(tr.loss.item()) - rb["loss"]) <= 1e-5 * rb["loss"]
    # projection backward on the GPU's own 2D sums (identical inputs on both sides)
    gs.project_bwd(n, tr.params, cam, tr.proj, tr.grad2d, tr.grads, tr.status)
    torch.cuda.synchronize()
    gref = oracle.project_bwd(P, n, cam, moments_to_partials(g2, ref["conic"]), prec=32)
    grad_close(tr.grads.cpu().numpy()[:, :n], gref, what="param grads")
    # the whole fused step from the same parameters, against the oracle's chain
    st = oracle.step(P, n, cam, target, np.zeros((59, P.shape[1])), np.zeros((59, P.shape[1])), 1, gi.lr_planes())
    tf = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes(), fused=True)
    tf.step(cam, torch.from_numpy(target).to(DEV))
    torch.cuda.synchronize()
    assert tf.check_status() == 0
    g_end = st["grads"][:, :n]
    grad_close(tf.m.cpu().numpy()[:, :n] / np.float64(np.float32(0.1)), g_end, what="fused m = 0.1 g")
    adam_close(tf.params.cpu().numpy()[:, :n], st["params"][:, :n], adam_defined(g_end), what="fused params")
    return ref, rb


def test_alpha_clamp_branch():
    P, n, cam, hot = _hot_scene()
    ref = oracle.project(P, n, cam, 32)
    assert ref["visible"][hot].all()
    # the hot Gaussians are the nearest of all, so every pixel composites them first;
    # count the pixels where one of them alone reaches the cap
    ys, xs = np.mgrid[0:H, 0:W] + 0.5
    capped = 0
    for i in hot:
        mx, my = ref["mean2d"][i]
        A, B, C = ref["conic"][i]
        dx, dy = xs - mx, ys - my
        power = -0.5 * (A * dx * dx + C * dy * dy) - B * dx * dy
        capped += int((ref["opacity"][i] * np.exp(power) >= 0.99).sum())
    assert ref["depth"][hot].max() < ref["depth"][ref["visible"]][:hot[0]].min()
    assert capped >= 60, capped
    _, rb = _stagewise(P, n, cam, seed=31)
    # a capped entry passes no opacity gradient from its capped pixels, but the
    # Gaussians still get gradients from their uncapped rims
    assert np.all(np.abs(rb["grad2d"][5, hot]) > 0)


def test_jacobian_clamp_branch():
    P, n, cam, out, (limx, limy) = _beyond_scene()
    ref = oracle.project(P, n, cam, 32)
    assert ref["visible"][out].all(), ref["count"][out]
    c = P[:3, out].T.astype(np.float64) @ cam["R"].astype(np.float64).T + cam["t"].astype(np.float64)
    past = (np.abs(c[:, 0] / c[:, 2]) > 1.5 * limx) | (np.abs(c[:, 1] / c[:, 2]) > 1.5 * limy)
    assert past.all()
    _, rb = _stagewise(P, n, cam, seed=32)
    # their footprints reach the image: they composite at some pixels and get gradients
    assert np.all(np.abs(rb["grad2d"][6:9, out]).sum(axis=0) > 0)
