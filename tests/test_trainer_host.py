"""The trainer's host logic, without a GPU: checkpoints (save and load round-trip the
parameter planes, the Adam moments, the step count and the Gaussian count bit for bit;
the trainer only holds buffers until a step runs, so CPU tensors serve) and the Adam
hyperparameters of a batch step."""
import numpy as np
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
    """The trainer's batch-step Adam hyperparameters follow the batch-size section of
    "Scaling 3D Gaussian Splatting with Distributed Compute": learning rates times
    sqrt(B), epsilon over sqrt(B), beta -> 1 - B (1 - beta) with beta1 = 0.9 reaching
    zero at B = 10 and held there beyond; one view leaves everything unchanged."""
    from gaussian_splatting_differentiable_project_gb300.trainer import batch_adam_hyper
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
