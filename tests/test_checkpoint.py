"""Trainer checkpoints: save and load round-trip the parameter planes, the Adam
moments, the step count and the Gaussian count bit for bit.  The trainer only holds
buffers until a step runs, so the round trip runs on CPU tensors without a GPU."""
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
