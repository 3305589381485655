"""GPU <-> oracle parity at the configs' full sizes, in the launch configuration the
bench uses (the library picks every launch shape from the sizes).

* 1M Gaussians at 512x512, 4M at 1024x1024 and 4M at 2048x2048 (the bench's
  workload): the whole view.  Every Gaussian's projection, the key and id of every
  intersection, every gathered record and every pixel's colour, T_final and
  n_contrib bit-exact; every Gaussian's nine 2D gradients; and the fused projection
  backward + Adam of every Gaussian (its first moment m = 0.1 g against the oracle's
  gradient of the whole chain, the updated parameters against the oracle's Adam).
* 18M Gaussians (turbulence isosurface), 2048x2048: the oracle on samples it can
  compute one by one (projection and the fused backward + Adam of sampled
  Gaussians; compositing and its backward on the tile block that the most rects
  cover, given every Gaussian whose rect meets the block), and for the sort the
  properties that fix its output uniquely at any size.

Tolerances are those of tests/_tol.py: integer/key/index work and the images
bit-exact, gradients 1e-4 relative with the per-plane floor, Adam 1e-5.
"""
import numpy as np
import pytest

import gs_inputs as gi
import oracle
from _grad2d import moments_to_partials
from _tol import adam_close, adam_defined, grad_close, isotropic

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _trainer_for(P, n, cam):
    """A trainer whose intersection capacity fits this view (read once, before the step)."""
    W, H = cam["width"], cam["height"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    params = torch.from_numpy(P).to(DEV)
    pb = gs.ProjBuffers(P.shape[1], DEV)
    gs.project(n, params, cam, pb, st)
    K = int(pb.count[:n].to(torch.int64).sum().item())
    del pb
    return gs.Trainer(params, n, W, H, capacity=K + 4096, lr_plane=gi.lr_planes())


def _check_projection(tr, P, n, cam, idx, ref=None):
    """Projection of the Gaussians idx bit-exact against the oracle's (``ref``: the
    oracle's projection of exactly those Gaussians, computed here if not given)."""
    if ref is None:
        ref = oracle.project(np.ascontiguousarray(P[:, idx]), len(idx), cam, 32)
    count = _u32(tr.proj.count)[idx]
    np.testing.assert_array_equal(count, ref["count"])
    vis = ref["count"] > 0
    np.testing.assert_array_equal(tr.proj.radius.cpu().numpy()[idx][vis], ref["radius"][vis])
    np.testing.assert_array_equal(tr.proj.depth.cpu().numpy()[idx][vis].view(np.uint32),
                                  ref["depth"][vis].view(np.uint32))
    rec = tr.proj.rec.cpu().numpy()[idx]
    exp = np.stack([ref["mean2d"][:, 0], ref["mean2d"][:, 1], -0.5 * ref["conic"][:, 0], -ref["conic"][:, 1],
                    -0.5 * ref["conic"][:, 2], ref["opacity"], ref["rgb"][:, 0], ref["rgb"][:, 1],
                    ref["rgb"][:, 2]], 1).astype(np.float32)
    np.testing.assert_array_equal(rec[vis, :9].view(np.uint32), exp[vis].view(np.uint32))
    return vis.sum()


def _check_sort_properties(tr, n, TX):
    """The sorted (key, id) sequence is fixed by: keys non-decreasing, equal keys in
    increasing id, every key's tile inside its Gaussian's rect with that Gaussian's
    depth bits, and each Gaussian appearing exactly count times; ranges follow."""
    K = tr.n_isect()
    keys = tr.bins.keys[:K].cpu().numpy().view(np.uint64)
    ids = _u32(tr.bins.ids)[:K].astype(np.int64)
    assert K == int(_u32(tr.proj.count)[:n].astype(np.int64).sum())
    dk = np.diff(keys.astype(np.uint64))
    assert np.all(keys[1:] >= keys[:-1])
    same = keys[1:] == keys[:-1]
    assert np.all(ids[1:][same] > ids[:-1][same])
    tile = (keys >> np.uint64(32)).astype(np.int64)
    zb = (keys & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    np.testing.assert_array_equal(zb, tr.proj.depth.cpu().numpy().view(np.uint32)[ids])
    rect = _u32(tr.proj.rect)[ids]
    tx, ty = tile % TX, tile // TX
    assert np.all((tx >= (rect[:, 0] & 0xFFFF)) & (tx <= (rect[:, 1] & 0xFFFF)))
    assert np.all((ty >= (rect[:, 0] >> 16)) & (ty <= (rect[:, 1] >> 16)))
    np.testing.assert_array_equal(np.bincount(ids, minlength=n)[:n], _u32(tr.proj.count)[:n])
    rg = _u32(tr.bins.ranges).astype(np.int64)
    T = rg.shape[0]
    start = np.searchsorted(tile, np.arange(T), side="left")
    end = np.searchsorted(tile, np.arange(T), side="right")
    ne = end > start
    np.testing.assert_array_equal(rg[ne, 0], start[ne])
    np.testing.assert_array_equal(rg[ne, 1], end[ne])
    assert np.all(rg[~ne] == 0)
    sample = np.random.default_rng(0).integers(0, K, 20000)
    np.testing.assert_array_equal(tr.bins.rec[sample].cpu().numpy().view(np.uint32),
                                  tr.proj.rec[torch.from_numpy(ids[sample]).to(DEV)].cpu().numpy().view(np.uint32))
    del dk
    return K


def _block_subset(ref, tx0, ty0, nt):
    """Gaussians (oracle projection) whose rect meets the block of nt x nt tiles, and
    those whose rect lies inside it."""
    r = ref["rect"]
    vis = ref["count"] > 0
    meets = vis & (r[:, 0] <= tx0 + nt - 1) & (r[:, 2] >= tx0) & (r[:, 1] <= ty0 + nt - 1) & (r[:, 3] >= ty0)
    inside = vis & (r[:, 0] >= tx0) & (r[:, 2] <= tx0 + nt - 1) & (r[:, 1] >= ty0) & (r[:, 3] <= ty0 + nt - 1)
    return np.nonzero(meets)[0], inside


def _sub(ref, idx):
    return {"proj16": np.ascontiguousarray(ref["proj16"][idx]), "iproj6": np.ascontiguousarray(ref["iproj6"][idx])}


def _check_block(tr, ref, cam, tx0, ty0, nt, backward=True):
    """Forward (bit-exact) and backward (Gaussians inside the block) on a tile block."""
    W, H = cam["width"], cam["height"]
    idx, inside = _block_subset(ref, tx0, ty0, nt)
    sub = _sub(ref, idx)
    rd = oracle.render(sub, W, H)
    ys, xs = slice(16 * ty0, 16 * (ty0 + nt)), slice(16 * tx0, 16 * (tx0 + nt))
    img = tr.image.cpu().numpy()
    np.testing.assert_array_equal(img[:, ys, xs].view(np.uint32), rd["image"][:, ys, xs].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.n_contrib)[ys, xs], rd["n_contrib"][ys, xs])
    if not backward:
        return
    target = np.full((3, H, W), 0.5, np.float32)
    target[:, ys, xs] = gi.offset_target(rd["image"][:, ys, xs], seed=11)
    rb = oracle.render(sub, W, H, target=target)
    gs.render_bwd(tr.n, tr.n_pad, cam, tr.bins, tr.bg, tr.image, torch.from_numpy(target).to(DEV), tr.T_final,
                  tr.n_contrib, tr.grad2d, tr.loss, tr.status)
    torch.cuda.synchronize()
    sel = inside[idx]
    assert sel.sum() > 50
    got = moments_to_partials(gs.grad2d_planes(tr.grad2d, tr.n_pad)[:, idx[sel]], ref["conic"][idx[sel]])
    grad_close(got, rb["grad2d"][:, sel], what="grad2d (block)")


def _check_fused_sample(tr, P, n, cam, idx):
    """Fused projection backward + Adam (t = 1) on seeded 2D sums, against the
    oracle's projection backward (fed the partials they define) and Adam for sampled
    Gaussians."""
    n_pad = P.shape[1]
    g2 = gi.random_grad2d(21, n, n_pad)
    lr = gi.lr_planes()
    gs.project(n, tr.params, cam, tr.proj, tr.status)
    tr.m.zero_()
    tr.v.zero_()
    gs.project_bwd_adam(n, tr.params, cam, tr.proj, torch.from_numpy(gs.grad2d_interleaved(g2)).to(DEV), tr.m, tr.v,
                        lr, 0.9, 0.999, 1e-15, 1, tr.status)
    torch.cuda.synchronize()
    Ps = np.ascontiguousarray(P[:, idx])
    conic = oracle.project(Ps, len(idx), cam, 32)["conic"]
    gref = oracle.project_bwd(Ps, len(idx), cam, moments_to_partials(g2[:, idx], conic), prec=32)
    pr, mr, vr = oracle.adam(Ps.astype(np.float64), gref, np.zeros_like(gref), np.zeros_like(gref), lr, 0.9, 0.999,
                             1e-15, 1)
    m = tr.m.cpu().numpy()[:, idx]
    iso = isotropic(P, n)
    grad_close(m / np.float64(np.float32(0.1)), gref, isotropic_scene=iso, what="fused m = 0.1 g")
    defined = adam_defined(gref, iso)
    assert defined.mean() > 0.2
    adam_close(tr.params.cpu().numpy()[:, idx], pr, defined)


def _densest_block(ref, TX, TY, nt):
    """Block of nt x nt tiles around the tile that the most Gaussians' rects cover
    (per-tile coverage from the oracle's rects by a 2D difference array)."""
    r = ref["rect"][ref["count"] > 0]
    d = np.zeros((TY + 1, TX + 1), np.int64)
    np.add.at(d, (r[:, 1], r[:, 0]), 1)
    np.add.at(d, (r[:, 1], r[:, 2] + 1), -1)
    np.add.at(d, (r[:, 3] + 1, r[:, 0]), -1)
    np.add.at(d, (r[:, 3] + 1, r[:, 2] + 1), 1)
    cover = d.cumsum(0).cumsum(1)[:TY, :TX]
    ty, tx = divmod(int(np.argmax(cover)), TX)
    return min(max(0, tx - nt // 2), TX - nt), min(max(0, ty - nt // 2), TY - nt)


# ----------------------------------------------------------------------------- whole views

def _full_view_parity(name, view, seed):
    cfg = gi.CONFIGS[name]
    P = gi.scene_for(cfg, device=DEV)
    n, W, H = cfg.n, cfg.width, cfg.height
    cam = gi.cameras_for(cfg)[view]
    iso = isotropic(P, n)
    assert iso
    tr = _trainer_for(P, n, cam)
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    ref = oracle.project(P, n, cam, 32)
    assert _check_projection(tr, P, n, cam, np.arange(n), ref) > 0.9 * n
    # binning: every key, id and range; every gathered record
    tl = oracle.tile_lists(ref, W, H)
    K = tr.n_isect()
    assert K == tl["K"]
    np.testing.assert_array_equal(tr.bins.keys[:K].cpu().numpy().view(np.uint64), tl["keys"])
    ids = _u32(tr.bins.ids)[:K]
    np.testing.assert_array_equal(ids, tl["ids"])
    rg = _u32(tr.bins.ranges)
    nonempty = tl["ranges"][:, 1] > tl["ranges"][:, 0]
    np.testing.assert_array_equal(rg[nonempty], tl["ranges"][nonempty])
    assert np.all(rg[~nonempty] == 0)
    del tl
    gathered = tr.proj.rec[tr.bins.ids[:K].to(torch.int64)]
    assert torch.equal(tr.bins.rec[:K].view(torch.int32), gathered.view(torch.int32))
    del gathered
    # compositing: every pixel; the backward: every Gaussian
    target = gi.uniform_target(seed, W, H)
    rb = oracle.render(ref, W, H, target=target)
    np.testing.assert_array_equal(_u32(tr.image), rb["image"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.T_final), rb["T_final"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.n_contrib), rb["n_contrib"])
    gs.render_bwd(n, tr.n_pad, cam, tr.bins, tr.bg, tr.image, torch.from_numpy(target).to(DEV), tr.T_final,
                  tr.n_contrib, tr.grad2d, tr.loss, tr.status)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    assert abs(float(tr.loss.item()) - rb["loss"]) <= 1e-5 * rb["loss"]
    grad_close(moments_to_partials(gs.grad2d_planes(tr.grad2d, n), ref["conic"]), rb["grad2d"], what="grad2d")
    # the fused projection backward + Adam (t = 1 from zero moments) of every Gaussian
    lr = gi.lr_planes()
    tr.m.zero_()
    tr.v.zero_()
    gs.project_bwd_adam(n, tr.params, cam, tr.proj, tr.grad2d, tr.m, tr.v, lr, 0.9, 0.999, 1e-15, 1, tr.status)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    gref = oracle.project_bwd(P, n, cam, rb["grad2d"], 32)
    del rb
    grad_close(tr.m.cpu().numpy()[:, :n] / np.float64(np.float32(0.1)), gref, isotropic_scene=iso,
               what="fused m = 0.1 g")
    pr, _, _ = oracle.adam(P[:, :n].astype(np.float64), gref, np.zeros_like(gref), np.zeros_like(gref), lr, 0.9,
                           0.999, 1e-15, 1)
    defined = adam_defined(gref, iso)
    # most Gaussians of a whole orbit view are hidden behind the surface's front and
    # get no gradient; several percent of the 59 n parameters still have a defined sign
    assert defined.mean() > 0.05
    adam_close(tr.params.cpu().numpy()[:, :n], pr, defined)
    assert not tr.params[:, n:].any()


def test_iso1m_512_full_parity():
    """1M Gaussians, 512x512, orbit view 5."""
    _full_view_parity("iso1m_512", 5, seed=3)


def test_iso4m_1024_full_parity():
    """4M Gaussians, 1024x1024 (the config with about 10-40 Gaussians per pixel),
    orbit view 0."""
    _full_view_parity("iso4m_1024", 0, seed=4)


def test_iso4m_2048_full_parity():
    """4M Gaussians, 2048x2048: the bench's workload, orbit view 0."""
    _full_view_parity("iso4m_2048", 0, seed=5)


def test_iso4m_2048_sort_properties_late_view():
    """A second view of the bench's workload (orbit view 300) through the sort's
    uniqueness properties and a sampled projection."""
    cfg = gi.CONFIGS["iso4m_2048"]
    P = gi.scene_for(cfg, device=DEV)
    n = cfg.n
    cam = gi.cameras_for(cfg)[300]
    tr = _trainer_for(P, n, cam)
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    _check_projection(tr, P, n, cam, np.sort(np.random.default_rng(2).choice(n, 40_000, replace=False)))
    _check_sort_properties(tr, n, cfg.width // 16)


# ----------------------------------------------------------------------------- 18M, 2048x2048

def test_turb18m_2048_sampled_parity():
    cfg = gi.CONFIGS["turb18m_2048"]
    P = gi.scene_for(cfg, device=DEV)
    n = cfg.n
    cam = gi.cameras_for(cfg)[100]
    tr = _trainer_for(P, n, cam)
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    rng = np.random.default_rng(3)
    _check_projection(tr, P, n, cam, np.sort(rng.choice(n, 40_000, replace=False)))
    TX, TY = cfg.width // 16, cfg.height // 16
    _check_sort_properties(tr, n, TX)
    ref = oracle.project(P, n, cam, 32)
    tx0, ty0 = _densest_block(ref, TX, TY, 3)
    _check_block(tr, ref, cam, tx0, ty0, 3)
    _check_fused_sample(tr, P, n, cam, np.sort(rng.choice(n, 40_000, replace=False)))
    assert tr.check_status() == 0
