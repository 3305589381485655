"""The Morton storage order (gs_spatial_order, gs_permute_planes) through the C ABI.

The codes are written out here from the header's definition (IEEE fp32 operations in
its order, so numpy reproduces them bit for bit) and the permutation must be their
stable sort, exactly.  Reordering changes a step only where two Gaussians of a tile
have equal fp32 depths, whose order the index decides: such ties are not rare (about
200 among the 57K visible Gaussians of the view below), and swapping them moves a few
pixels by up to about 1e-4.  So the reordered trainer is compared bit for bit with a
trainer built from the same permutation applied on the host."""
import numpy as np
import pytest

import gs_inputs as gi

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"


def _spread10(x):
    x = x.astype(np.uint32) & np.uint32(0x3FF)
    x = (x | (x << np.uint32(16))) & np.uint32(0x030000FF)
    x = (x | (x << np.uint32(8))) & np.uint32(0x0300F00F)
    x = (x | (x << np.uint32(4))) & np.uint32(0x030C30C3)
    x = (x | (x << np.uint32(2))) & np.uint32(0x09249249)
    return x


def _codes(P, n):
    code = np.zeros(n, np.uint32)
    for a in range(3):
        v = P[a, :n].astype(np.float32)
        fin = np.isfinite(v)
        if fin.any():
            lo, hi = v[fin].min(), v[fin].max()
            ext = np.float32(hi - lo)
            sc = np.float32(np.float32(1023.0) / ext) if ext > 0 else np.float32(0.0)
        else:
            lo, sc = np.float32(0.0), np.float32(0.0)
        with np.errstate(invalid="ignore"):
            t = ((v - lo).astype(np.float32) * sc).astype(np.float32) + np.float32(0.5)
        t = np.where(fin, t, np.float32(0.0)).astype(np.float32)
        q = np.clip(np.floor(t), 0, 1023).astype(np.uint32)
        code |= _spread10(q) << np.uint32(a)
    return code


def _order(P, n):
    Pd = torch.from_numpy(P).to(DEV)
    perm = torch.empty(max(n, 1), dtype=torch.int32, device=DEV)
    ws = torch.empty(max(gs.spatial_order_workspace_bytes(n, P.shape[1]), 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gs.spatial_order(n, Pd, perm, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return perm.cpu().numpy()[:n].astype(np.int64)


@pytest.mark.parametrize("n", [1, 300, 4096, 70_000])
def test_perm_is_the_stable_sort_of_the_codes(n):
    P = gi.scene_for(gi.CONFIGS["tiny"], n=n, seed=3).copy()
    if n >= 300:
        P[0, 7] = np.nan            # a non-finite coordinate counts as lo
        P[1, 11] = np.inf
        P[:3, 20:40] = P[:3, 40:60]  # equal codes: ties by index
    got = _order(P, n)
    want = np.argsort(_codes(P, n), kind="stable")
    np.testing.assert_array_equal(got, want)


def test_flat_axis_and_isosurface_scene():
    """An axis with a single value (hi = lo) and a level-set scene of 60K Gaussians;
    in the second, consecutive Gaussians in the new order are far closer in space."""
    P = gi.scene_for(gi.CONFIGS["tiny"], n=2000, seed=4).copy()
    P[2, :2000] = 0.25
    np.testing.assert_array_equal(_order(P, 2000), np.argsort(_codes(P, 2000), kind="stable"))
    cfg = gi.CONFIGS["iso1m_512"]
    n = 60_000
    P = gi.scene_for(cfg, n=n)
    perm = _order(P, n)
    np.testing.assert_array_equal(perm, np.argsort(_codes(P, n), kind="stable"))
    mu = P[:3, :n].T.astype(np.float64)
    step_before = np.linalg.norm(np.diff(mu, axis=0), axis=1).mean()
    step_after = np.linalg.norm(np.diff(mu[perm], axis=0), axis=1).mean()
    assert step_after < 0.1 * step_before


@pytest.mark.parametrize("dtype", [torch.float32, torch.int32])
def test_permute_planes(dtype):
    n, n_pad, planes = 3000, 3072, 5
    rng = np.random.default_rng(1)
    perm = rng.permutation(n).astype(np.int32)
    src = rng.integers(-2**31, 2**31 - 1, (planes, n_pad), dtype=np.int64).astype(np.int32)
    src_t = torch.from_numpy(src).to(DEV)
    if dtype == torch.float32:
        src_t = src_t.view(torch.float32)
    dst = torch.empty_like(src_t)
    gs.permute_planes(n, torch.from_numpy(perm).to(DEV), src_t, dst)
    torch.cuda.synchronize()
    want = src.copy()
    want[:, :n] = src[:, perm]
    np.testing.assert_array_equal(dst.view(torch.int32).cpu().numpy(), want)


def test_render_invariant_and_state_permuted():
    cfg = gi.CONFIGS["iso1m_512"]
    n, W, H = 60_000, 256, 192
    P = gi.scene_for(cfg, n=n)
    cam = gi.fibonacci_cameras(cfg.n_views, W, H)[3]
    perm = np.argsort(_codes(P, n), kind="stable")
    Pm = P.copy()
    Pm[:, :n] = P[:, perm]
    a = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    b = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    c = gs.Trainer(Pm, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    np.testing.assert_array_equal(b.reorder_spatially().cpu().numpy(), perm)
    for t in (a, b, c):
        t.forward(cam)
    torch.cuda.synchronize()
    # reordered on the device = reordered on the host, bit for bit
    assert b.n_isect() == c.n_isect() == a.n_isect()
    for name in ("image", "T_final", "n_contrib"):
        assert torch.equal(getattr(b, name), getattr(c, name)), name
    # against the generated order only tied depths differ
    assert float((a.image - b.image).abs().max().item()) < 1e-3
    # after a step with density control on, every per-Gaussian array follows its
    # Gaussian
    b.enable_density_control(3.0)
    tgt = torch.from_numpy(gi.offset_target(np.zeros((3, H, W), np.float32), seed=2)).to(DEV)
    b.step(cam, tgt)
    torch.cuda.synchronize()
    before = {k: getattr(b, k).clone() for k in ("params", "m", "v", "grad_acc", "vis_cnt")}
    assert int(before["vis_cnt"].max().item()) == 1 and float(before["m"].abs().max().item()) > 0
    pi = b.reorder_spatially().to(torch.int64)
    torch.cuda.synchronize()
    for k, x in before.items():
        y = getattr(b, k)
        assert torch.equal(y[..., :n], x[..., :n].index_select(-1, pi)), k
        assert torch.equal(y[..., n:], x[..., n:]), k
    b.step(cam, tgt)
    torch.cuda.synchronize()
    assert b.check_status() == 0
