"""Adaptive density control through the C ABI against the oracle (oracle/densify.py),
on identical inputs: the accumulation and every decision bit-exact, the new planes
bit-exact except split children's means (fp32 rotation against the oracle's fp64,
within 2e-6 of the parameters' scale), and a short training run with a refinement."""
import numpy as np
import pytest

import gs_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gaussian_splatting_differentiable_project_gb300 as gs  # noqa: E402

DEV = "cuda"
D = oracle.densify


def _scene(n):
    cfg = gi.CONFIGS["tiny"]
    P = gi.scene_for(cfg, n=n).copy()
    P[10, :n:37] = -7.0  # some transparent Gaussians
    return P, gi.camera((0.0, 0.0, 3.0), 128, 128)


@pytest.mark.parametrize("n", [4096, 3000])
def test_accumulate_matches_oracle(n):
    """Seeded sums in grad2d's layout on the GPU; the oracle accumulates the mean
    gradients they define (the header's formula with the Gaussian's conic, each fp32
    product and sum rounded once, as stated there)."""
    P, cam = _scene(n)
    W, H = cam["width"], cam["height"]
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    tr.enable_density_control(3.3)
    pr = oracle.project(P, n, cam, 32)
    tr.forward(cam)
    S = gi.random_grad2d(5, n, tr.n_pad)
    tr.grad2d.copy_(torch.from_numpy(gs.grad2d_interleaved(S)))
    vis = pr["count"] > 0
    A, B, C = (np.where(vis, pr["conic"][:, k], 0).astype(np.float32) for k in range(3))
    g2 = np.zeros((9, n), np.float32)
    g2[0] = (A * S[0, :n]).astype(np.float32) + (B * S[1, :n]).astype(np.float32)
    g2[1] = (B * S[0, :n]).astype(np.float32) + (C * S[1, :n]).astype(np.float32)
    acc = np.zeros(n, np.float32)
    cnt = np.zeros(n, np.int64)
    for _ in range(2):
        gs.densify_accumulate(n, tr.n_pad, tr.proj, tr.grad2d, W, H, tr.grad_acc, tr.vis_cnt)
        D.accumulate(g2, vis, W, H, acc, cnt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tr.vis_cnt.cpu().numpy()[:n], cnt)
    np.testing.assert_array_equal(tr.grad_acc.cpu().numpy()[:n].view(np.uint32), acc.view(np.uint32))
    assert (cnt > 0).mean() > 0.5 and acc.max() > 0


@pytest.mark.parametrize("n,prune_big", [(4096, False), (3000, True)])
def test_plan_and_apply_match_oracle(n, prune_big):
    P, cam = _scene(n)
    n_pad = P.shape[1]
    rng = np.random.default_rng(n)
    acc = np.zeros(n_pad, np.float32)
    cnt = np.zeros(n_pad, np.int32)
    acc[:n] = rng.exponential(3e-4, n).astype(np.float32)
    cnt[:n] = rng.integers(0, 4, n)
    m = rng.normal(0, 1e-3, P.shape).astype(np.float32)
    v = np.abs(rng.normal(0, 1e-6, P.shape)).astype(np.float32)
    randn = rng.normal(size=(n, 6)).astype(np.float32)
    extent = 3.3
    cfg, log_shrink, _ = gs.densify_thresholds(extent, prune_big=prune_big)
    th = D.thresholds(extent=extent)
    # the product's thresholds are its own fp64 formation; they round to the oracle's
    assert np.float32(cfg.logit_prune) == th["logit_prune"] and np.float32(log_shrink) == th["log_shrink"]
    Pd, Md, Vd = (torch.from_numpy(x).to(DEV) for x in (P, m, v))
    accd, cntd = torch.from_numpy(acc).to(DEV), torch.from_numpy(cnt).to(DEV)
    action = torch.empty(n, dtype=torch.uint8, device=DEV)
    offset = torch.empty(n, dtype=torch.int32, device=DEV)
    n_out = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gs.densify_workspace_bytes(n, n_pad), dtype=torch.uint8, device=DEV)
    gs.densify_plan(n, Pd, accd, cntd, cfg, action, offset, n_out, ws)
    a_ref, off_ref, n_ref = D.plan(P, n, acc, cnt, th, prune_big=prune_big)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(action.cpu().numpy(), a_ref)
    np.testing.assert_array_equal(offset.cpu().numpy().astype(np.uint32), off_ref)
    assert int(n_out.item()) == n_ref
    assert min(np.bincount(a_ref, minlength=4)) > 0
    n_pad_new = -(-n_ref // 256) * 256
    out = [torch.full((59, n_pad_new), float("nan"), device=DEV) for _ in range(3)]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gs.densify_apply(n, Pd, Md, Vd, action, offset, n_out, torch.from_numpy(randn).to(DEV), log_shrink, *out, st)
    ref_p, ref_m, ref_v = D.apply(P, m, v, n, a_ref, off_ref, n_ref, randn, th, n_pad_new)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got_p, got_m, got_v = (x.cpu().numpy() for x in out)
    np.testing.assert_array_equal(got_m.view(np.uint32), ref_m.view(np.uint32))
    np.testing.assert_array_equal(got_v.view(np.uint32), ref_v.view(np.uint32))
    child = np.zeros(n_pad_new, bool)
    sp = np.nonzero(a_ref == D.SPLIT)[0]
    child[off_ref[sp]] = True
    child[off_ref[sp] + 1] = True
    np.testing.assert_array_equal(got_p[3:].view(np.uint32), ref_p[3:].view(np.uint32))
    np.testing.assert_array_equal(got_p[:3, ~child].view(np.uint32), ref_p[:3, ~child].view(np.uint32))
    scale = np.abs(ref_p[:3, child]).max()
    assert np.abs(got_p[:3, child] - ref_p[:3, child]).max() <= 2e-6 * max(scale, 1.0)
    assert not got_p[:, n_ref:].any()


def test_apply_refuses_a_small_destination():
    """n_out above n_pad_dst: GS_ERR_CAPACITY on the device, nothing written."""
    n = 4096
    P, _ = _scene(n)
    n_pad = P.shape[1]
    cfg, log_shrink, _ = gs.densify_thresholds(3.3)
    Pd = torch.from_numpy(P).to(DEV)
    acc = torch.full((n_pad,), 1e-3, dtype=torch.float32, device=DEV)  # everything grows
    cnt = torch.ones(n_pad, dtype=torch.int32, device=DEV)
    action = torch.empty(n, dtype=torch.uint8, device=DEV)
    offset = torch.empty(n, dtype=torch.int32, device=DEV)
    n_out = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gs.densify_workspace_bytes(n, n_pad), dtype=torch.uint8, device=DEV)
    gs.densify_plan(n, Pd, acc, cnt, cfg, action, offset, n_out, ws)
    out = [torch.zeros((59, n_pad), device=DEV) for _ in range(3)]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gs.densify_apply(n, Pd, Pd, Pd, action, offset, n_out, torch.zeros((n, 6), device=DEV), log_shrink, *out, st)
    torch.cuda.synchronize()
    assert int(n_out.item()) > n_pad
    assert int(st.item()) & gs.GS_ERR_CAPACITY
    assert not any(x.any() for x in out)


def test_opacity_reset_matches_oracle():
    n = 3000
    P, _ = _scene(n)
    rng = np.random.default_rng(9)
    P[10, :n] = rng.normal(-3.0, 2.0, n).astype(np.float32)
    m = rng.normal(size=P.shape).astype(np.float32)
    v = np.abs(m)
    _, _, logit_reset = gs.densify_thresholds(3.3)
    th = D.thresholds(extent=3.3)
    assert np.float32(logit_reset) == th["logit_reset"]
    Pd, Md, Vd = (torch.from_numpy(x.copy()).to(DEV) for x in (P, m, v))
    gs.opacity_reset(n, Pd, Md, Vd, logit_reset)
    D.opacity_reset(P, m, v, n, th)
    torch.cuda.synchronize()
    for got, ref in ((Pd, P), (Md, m), (Vd, v)):
        np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_training_with_refinement():
    """Six steps with the gradient accumulated, a refinement whose counts are the
    oracle plan of the same accumulators, then three more steps at the new size."""
    n = 4096
    P, cam = _scene(n)
    W, H = cam["width"], cam["height"]
    tgt = torch.from_numpy(gi.offset_target(oracle.render(oracle.project(P, n, cam, 32), W, H)["image"],
                                            seed=4)).to(DEV)
    tr = gs.Trainer(P, n, W, H, capacity=1 << 20, lr_plane=gi.lr_planes())
    tr.enable_density_control(1.0)  # a small extent: many Gaussians count as large and split
    for _ in range(6):
        tr.step(cam, tgt)
    torch.cuda.synchronize()
    Pn = tr.params.cpu().numpy()
    acc = tr.grad_acc.cpu().numpy()
    cnt = tr.vis_cnt.cpu().numpy()
    assert cnt[:n].max() == 6
    a_ref, _, n_ref = D.plan(Pn, n, acc, cnt, D.thresholds(extent=1.0))
    counts = tr.refine(seed=1)
    assert tr.n == n_ref == counts["n"]
    assert counts["cloned"] + counts["split"] > 0 and counts["pruned"] > 0
    assert tr.params.shape[1] % 256 == 0 and not tr.grad_acc.any()
    for _ in range(3):
        tr.step(cam, tgt)
    torch.cuda.synchronize()
    assert tr.check_status() == 0
    assert np.isfinite(float(tr.loss.item())) and int(tr.vis_cnt.max().item()) == 3
