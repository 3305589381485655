"""The trainer's host logic, without a GPU: checkpoints (save and load round-trip the
parameter planes, the Adam moments, the step count and the Gaussian count bit for bit;
the trainer only holds buffers until a step runs, so CPU tensors serve), the Adam
hyperparameters of a batch step and the density-control thresholds."""
import numpy as np
import pytest
import torch

import gs_inputs as gi
from gaussian_splatting_differentiable_project_gb300.trainer import Trainer


def test_save_load_round_trip(tmp_path):
    cfg = gi.CONFIGS["tiny"]
    n = 3000
    P = gi.scene_for(cfg, n=n, seed=2)
    rng = np.random.default_rng(4)
    tr = Trainer(P, n, 72, 56, capacity=1 << 12, lr_plane=gi.lr_planes(), device="cpu")
    m = rng.normal(size=P.shape).astype(np.float32)
    v = np.abs(rng.normal(size=P.shape)).astype(np.float32)
    tr.m.copy_(torch.from_numpy(m))
    tr.v.copy_(torch.from_numpy(v))
    tr.t = 17
    path = tmp_path / "state.npz"
    tr.save(path)
    back = Trainer.load(path, 72, 56, 1 << 12, gi.lr_planes(), device="cpu")
    assert back.n == n and back.t == 17 and back.n_pad == P.shape[1]
    for name, want in (("params", P), ("m", m), ("v", v)):
        np.testing.assert_array_equal(getattr(back, name).numpy().view(np.uint32), want.view(np.uint32))


def test_batch_hyperparameters_on_the_host():
    """The library's batch-step Adam hyperparameters (gs_batch_hyper, a host call) follow
    the batch-size section of
    "Scaling 3D Gaussian Splatting with Distributed Compute": learning rates times
    sqrt(B), epsilon over sqrt(B), beta -> 1 - B (1 - beta) with beta1 = 0.9 reaching
    zero at B = 10 and held there beyond; one view leaves everything unchanged.  The
    oracle's own statement of the rule agrees at every batch size."""
    from gaussian_splatting_differentiable_project_gb300 import batch_hyper as batch_adam_hyper
    lr = gi.lr_planes()
    l1, b1, b2, e1 = batch_adam_hyper(1, lr, 0.9, 0.999, 1e-15)
    np.testing.assert_array_equal(l1, np.asarray(lr, np.float64))
    assert (b1, b2, e1) == (0.9, 0.999, 1e-15)
    l4, b1, b2, e4 = batch_adam_hyper(4, lr, 0.9, 0.999, 1e-15)
    np.testing.assert_allclose(l4, 2.0 * np.asarray(lr, np.float64), rtol=1e-15)
    assert e4 == 0.5e-15 and abs(b1 - 0.6) < 1e-15 and abs(b2 - 0.996) < 1e-15
    _, b1, _, _ = batch_adam_hyper(10, lr, 0.9, 0.999, 1e-15)
    assert abs(b1) < 1e-15
    _, b1, b2, _ = batch_adam_hyper(16, lr, 0.9, 0.999, 1e-15)
    assert b1 == 0.0 and abs(b2 - 0.984) < 1e-15
    import oracle
    for B in (1, 2, 3, 7, 10, 11, 64):
        got = batch_adam_hyper(B, lr, 0.9, 0.999, 1e-15)
        want = oracle.batch_hyper(B, lr, 0.9, 0.999, 1e-15)
        np.testing.assert_allclose(got[0], want[0], rtol=1e-15)
        for a, b in zip(got[1:], want[1:]):
            assert abs(a - b) <= 1e-15 * max(1.0, abs(b)), (B, got[1:], want[1:])
    import gaussian_splatting_differentiable_project_gb300 as gs
    with pytest.raises(gs.GsError):
        batch_adam_hyper(0, lr, 0.9, 0.999, 1e-15)


def test_density_thresholds_on_the_host():
    """The density-control thresholds (gs_densify_thresholds, a host call), formed in
    fp64 and rounded to fp32 once: grow above a mean 2D gradient of 2e-4; clone at most 0.01 x
    the extent in scale (compared as a log-scale); prune below opacity 0.005 (as a
    logit) or, optionally, above 0.1 x the extent; split children shrink by 1.6 (as a
    log); the opacity reset clamps to twice the prune opacity (as a logit)."""
    import math
    import gaussian_splatting_differentiable_project_gb300 as gs
    extent = 3.3
    cfg, log_shrink, logit_reset = gs.densify_thresholds(extent, prune_big=True)
    f32 = lambda x: float(np.float32(x))  # noqa: E731
    assert f32(cfg.grad_threshold) == f32(2e-4)
    assert f32(cfg.log_grow_scale) == f32(math.log(0.01 * extent))
    assert f32(cfg.log_prune_scale) == f32(math.log(0.1 * extent))
    assert f32(cfg.logit_prune) == f32(math.log(0.005 / 0.995))
    assert cfg.prune_big == 1
    assert log_shrink == f32(math.log(1.6))
    assert logit_reset == f32(math.log(0.01 / 0.99))
    # the logit threshold decides exactly where the sigmoid crosses 0.005
    assert 1 / (1 + math.exp(-f32(cfg.logit_prune))) == pytest.approx(0.005, rel=1e-6)
    # the oracle's own thresholds agree
    import oracle
    th = oracle.densify.thresholds(extent=extent)
    for k in ("logit_prune", "log_grow_scale", "log_prune_scale"):
        assert f32(getattr(cfg, k)) == f32(th[k]), k
    assert log_shrink == f32(th["log_shrink"]) and logit_reset == f32(th["logit_reset"])
    with pytest.raises(gs.GsError):
        gs.densify_thresholds(-1.0)
