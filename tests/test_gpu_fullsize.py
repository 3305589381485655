"""GPU <-> oracle parity at the configs' full sizes, in the launch configuration the
bench uses (the library picks every launch shape from the sizes).

* 1M Gaussians, 512x512: every stage against the oracle over the whole image.
* 4M Gaussians, 2048x2048 (the bench's workload): the oracle on samples it can
  compute one by one (projection and the fused backward + Adam of sampled
  Gaussians; compositing and its backward on a block of tiles, given every
  Gaussian whose rect meets the block), and for the sort the properties that fix
  its output uniquely at any size.
* 18M Gaussians (turbulence isosurface), 2048x2048: the same sort properties,
  sampled projection and a sampled tile block.

Tolerances are those of test_gpu_parity.py: integer/key/index work and the
images bit-exact, gradients 1e-4 relative with the group floor, Adam 1e-5.
"""
import numpy as np
import pytest

import gs_inputs as gi
import oracle
from _grad2d import moments_to_partials

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"
GROUPS_59 = [(0, 3), (3, 10), (10, 11), (11, 59)]
GROUPS_9 = [(0, 2), (2, 5), (5, 6), (6, 9)]


def _grad_close(got, ref, rtol=1e-4, floor=1e-6, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    groups = GROUPS_59 if ref.shape[0] == 59 else GROUPS_9
    scale = np.zeros((ref.shape[0], 1))
    for a, b in groups:
        scale[a:b] = max(np.abs(ref[a:b]).max(), 1e-30)
    tol = rtol * np.abs(ref) + floor * scale
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


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


def _check_projection(tr, P, n, cam, idx):
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
    _grad_close(got, rb["grad2d"][:, sel], what="grad2d (block)")


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
    _grad_close(m / 0.1, mr / 0.1, what="fused m = 0.1 g")
    p = tr.params.cpu().numpy()[:, idx].astype(np.float64)
    gscale = np.zeros((59, 1))
    for a, b in GROUPS_59:
        gscale[a:b] = np.abs(gref[a:b]).max()
    defined = np.abs(gref) > 1e-3 * gscale
    assert defined.mean() > 0.2
    assert not ((np.abs(p - pr) > 1e-5 * np.abs(pr) + 1e-7) & defined).any()


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


# ----------------------------------------------------------------------------- 1M, 512x512

def test_iso1m_512_full_parity():
    cfg = gi.CONFIGS["iso1m_512"]
    P = gi.scene_for(cfg, device=DEV)
    n = cfg.n
    cam = gi.cameras_for(cfg)[5]
    tr = _trainer_for(P, n, cam)
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    ref = oracle.project(P, n, cam, 32)
    assert _check_projection(tr, P, n, cam, np.arange(n)) > 0.9 * n
    tl = oracle.tile_lists(ref, cfg.width, cfg.height)
    K = tr.n_isect()
    assert K == tl["K"]
    np.testing.assert_array_equal(tr.bins.keys[:K].cpu().numpy().view(np.uint64), tl["keys"])
    np.testing.assert_array_equal(_u32(tr.bins.ids)[:K], tl["ids"])
    rd = oracle.render(ref, cfg.width, cfg.height)
    np.testing.assert_array_equal(tr.image.cpu().numpy().view(np.uint32), rd["image"].view(np.uint32))
    np.testing.assert_array_equal(_u32(tr.n_contrib), rd["n_contrib"])
    target = gi.offset_target(rd["image"], seed=3)
    rb = oracle.render(ref, cfg.width, cfg.height, target=target)
    gs.render_bwd(n, tr.n_pad, cam, tr.bins, tr.bg, tr.image, torch.from_numpy(target).to(DEV), tr.T_final,
                  tr.n_contrib, tr.grad2d, tr.loss, tr.status)
    torch.cuda.synchronize()
    _grad_close(moments_to_partials(gs.grad2d_planes(tr.grad2d, n), ref["conic"]), rb["grad2d"], what="grad2d")
    assert abs(float(tr.loss.item()) - rb["loss"]) <= 1e-5 * rb["loss"]
    _check_fused_sample(tr, P, n, cam, np.random.default_rng(1).choice(n, 50_000, replace=False))
    assert tr.check_status() == 0


# ----------------------------------------------------------------------------- 4M, 2048x2048

def test_iso4m_2048_sampled_parity():
    cfg = gi.CONFIGS["iso4m_2048"]
    P = gi.scene_for(cfg, device=DEV)
    n = cfg.n
    cam = gi.cameras_for(cfg)[0]
    tr = _trainer_for(P, n, cam)
    tr.forward(cam)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    rng = np.random.default_rng(2)
    _check_projection(tr, P, n, cam, np.sort(rng.choice(n, 40_000, replace=False)))
    TX, TY = cfg.width // 16, cfg.height // 16
    _check_sort_properties(tr, n, TX)
    ref = oracle.project(P, n, cam, 32)
    tx0, ty0 = _densest_block(ref, TX, TY, 4)
    _check_block(tr, ref, cam, tx0, ty0, 4)
    _check_block(tr, ref, cam, TX // 2 - 2, TY // 2 - 2, 4, backward=False)
    _check_fused_sample(tr, P, n, cam, np.sort(rng.choice(n, 40_000, replace=False)))
    assert tr.check_status() == 0


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
    _check_block(tr, ref, cam, tx0, ty0, 3, backward=False)
