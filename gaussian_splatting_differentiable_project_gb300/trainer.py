"""Buffers and call order of one training step (one camera view per step).

The step is the six C-ABI calls in order: project -> bin_sort -> render_fwd ->
render_bwd -> project_bwd -> adam_step, all enqueued on one CUDA stream with no
host synchronisation inside the step.  With a D-SSIM weight lambda > 0 the loss is
(1 - lambda) L1 + lambda (1 - SSIM): ssim_fwd and ssim_bwd run between render_fwd
and render_bwd, and render_bwd adds their image gradient to the weighted L1 one.  Parameters, Adam moments and every
transient buffer stay resident on the device; the device status word is read
only when the caller asks for it.
"""
from __future__ import annotations

import numpy as np

from . import (BinBuffers, ProjBuffers, GRAD2D_STRIDE, SSIM_MAPS, adam_step, batch_hyper, bin_sort, densify_accumulate,
               densify_apply, densify_plan, densify_thresholds, densify_workspace_bytes, opacity_reset,
               permute_planes, project, project_bwd, project_bwd_accumulate, project_bwd_adam,
               project_bwd_adam_tdev, render_bwd, render_fwd, spatial_order, spatial_order_workspace_bytes,
               ssim_bwd, ssim_fwd, status_str, step_counter_add)


class HostTargets:
    """Double-buffered upload of per-step targets (3 x H x W fp32, pinned host memory).

    ``put`` starts the upload of a host target into a free device slot on a copy
    stream of its own and returns the slot; ``get`` orders a compute stream after that
    upload; ``release`` marks the slot free once the work enqueued so far on the
    compute stream is done.  The upload for the next step thus runs while the current
    step computes.  With ``after`` (an event on the compute stream) the upload waits for
    it: ``Trainer.step_staged`` records one after its backward, so that the upload's
    writes pass through L2 during the streaming projection-backward and Adam pass
    rather than while the rasterisers' working set is there."""

    def __init__(self, shape, device="cuda", slots: int = 2):
        import torch
        self.bufs = [torch.empty(shape, dtype=torch.float32, device=device) for _ in range(slots)]
        self.copied = [torch.cuda.Event() for _ in range(slots)]
        self.consumed = [torch.cuda.Event() for _ in range(slots)]
        self.used = [False] * slots
        self.stream = torch.cuda.Stream(device=device)
        self.next = 0

    def put(self, host, after=None) -> int:
        import torch
        k = self.next
        self.next = (k + 1) % len(self.bufs)
        with torch.cuda.stream(self.stream):
            if self.used[k]:
                self.stream.wait_event(self.consumed[k])
            if after is not None:
                self.stream.wait_event(after)
            self.bufs[k].copy_(host, non_blocking=True)
            self.copied[k].record(self.stream)
        self.used[k] = True
        return k

    def get(self, k: int, stream=None):
        import torch
        (stream or torch.cuda.current_stream()).wait_event(self.copied[k])
        return self.bufs[k]

    def release(self, k: int, stream=None) -> None:
        import torch
        self.consumed[k].record(stream or torch.cuda.current_stream())


class Trainer:
    def __init__(self, params, n: int, width: int, height: int, capacity: int, lr_plane, betas=(0.9, 0.999),
                 eps: float = 1e-15, bg=(0.0, 0.0, 0.0), device="cuda", fused: bool = True, dssim: float = 0.0):
        import torch
        if isinstance(params, np.ndarray):
            params = torch.from_numpy(np.ascontiguousarray(params, np.float32))
        self.params = params.to(device=device, dtype=torch.float32).contiguous()
        self.n = int(n)
        self.n_pad = int(self.params.shape[1])
        self.width, self.height = int(width), int(height)
        self.m = torch.zeros_like(self.params)
        self.v = torch.zeros_like(self.params)
        self.grads = torch.empty_like(self.params)
        self.grad2d = torch.empty((self.n_pad, GRAD2D_STRIDE), dtype=torch.float32, device=device)
        self.proj = ProjBuffers(self.n_pad, device)
        self.bins = BinBuffers(self.n, capacity, width, height, device)
        self.image = torch.empty((3, height, width), dtype=torch.float32, device=device)
        self.T_final = torch.empty((height, width), dtype=torch.float32, device=device)
        self.n_contrib = torch.empty((height, width), dtype=torch.int32, device=device)
        self.loss = torch.zeros(1, dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.lr_plane = np.asarray(lr_plane, np.float64)
        self.beta1, self.beta2 = float(betas[0]), float(betas[1])
        self.eps = float(eps)
        self.bg = tuple(float(x) for x in bg)
        self.fused = bool(fused)
        self.dssim = float(dssim)
        if not (0.0 <= self.dssim <= 1.0):
            raise ValueError(f"D-SSIM weight must lie in [0, 1], got {dssim}")
        if self.dssim > 0.0:
            self.ssim_maps = torch.empty((SSIM_MAPS, height, width), dtype=torch.float32, device=device)
            self.dLdC = torch.empty((3, height, width), dtype=torch.float32, device=device)
            self.ssim_val = torch.zeros(1, dtype=torch.float32, device=device)
        self.t = 0
        self.capacity = int(capacity)
        self.device = device
        self.density = None

    # the stages ------------------------------------------------------------------
    def forward(self, cam: dict, stream=None) -> None:
        project(self.n, self.params, cam, self.proj, self.status, stream)
        bin_sort(self.n, self.n_pad, self.proj, cam, self.bins, self.status, stream)
        render_fwd(cam, self.bins, self.bg, self.image, self.T_final, self.n_contrib, self.status, stream)

    def loss_backward(self, cam: dict, target, stream=None, weight: float = 1.0, loss_out=None,
                      ssim_out=None) -> None:
        """The loss and its gradient with respect to the projected quantities
        (grad2d): the D-SSIM term first when lambda > 0, then the render backward.
        ``weight`` scales the whole loss (1 / batch for a view of a batch step);
        ``loss_out`` / ``ssim_out`` default to the trainer's own scalars."""
        extra = None
        if self.dssim > 0.0:
            ssim_fwd(self.image, target, self.dssim * weight, self.ssim_maps,
                     self.ssim_val if ssim_out is None else ssim_out, stream)
            ssim_bwd(self.image, target, self.ssim_maps, self.dLdC, stream)
            extra = self.dLdC
        render_bwd(self.n, self.n_pad, cam, self.bins, self.bg, self.image, target, self.T_final, self.n_contrib,
                   self.grad2d, self.loss if loss_out is None else loss_out, self.status, stream,
                   l1_weight=(1.0 - self.dssim) * weight, dLdC_extra=extra)

    def backward(self, cam: dict, target, stream=None) -> None:
        self.loss_backward(cam, target, stream)
        self.accumulate_density(cam, stream)
        project_bwd(self.n, self.params, cam, self.proj, self.grad2d, self.grads, self.status, stream)

    def optimizer_step(self, stream=None) -> None:
        self.t += 1
        adam_step(self.n, self.params, self.grads, self.m, self.v, self.lr_plane, self.beta1, self.beta2, self.eps,
                  self.t, stream)

    def step(self, cam: dict, target, stream=None) -> None:
        """One optimisation step for one view: forward, backward, Adam.  With
        ``fused`` the projection backward and Adam run as one call and the gradient
        planes (``grads``) are not written."""
        self.forward(cam, stream)
        if not self.fused:
            self.backward(cam, target, stream)
            self.optimizer_step(stream)
            return
        self.loss_backward(cam, target, stream)
        self.accumulate_density(cam, stream)
        self.t += 1
        project_bwd_adam(self.n, self.params, cam, self.proj, self.grad2d, self.m, self.v, self.lr_plane, self.beta1,
                         self.beta2, self.eps, self.t, self.status, stream)

    def step_batch(self, cams, targets, stream=None) -> None:
        """One optimisation step over a batch of views: the loss is the mean of the
        view losses.  The first view writes the gradient planes, later ones
        accumulate into them, and the last view's projection backward runs fused with
        Adam (adding the accumulated planes) under the batch-scaled hyperparameters;
        with ``fused`` off the last view accumulates too and Adam runs on its own.
        Per-view losses (weighted by 1 / batch) land in ``batch_losses``."""
        import torch
        B = len(cams)
        if B < 1 or len(targets) != B:
            raise ValueError("step_batch needs one target per camera")
        if getattr(self, "batch_losses", None) is None or self.batch_losses.numel() != B:
            self.batch_losses = torch.zeros(B, dtype=torch.float32, device=self.params.device)
            if self.dssim > 0.0:
                self.batch_ssim = torch.zeros(B, dtype=torch.float32, device=self.params.device)
        lr_b, b1, b2, eps_b = batch_hyper(B, self.lr_plane, self.beta1, self.beta2, self.eps)
        self.t += 1
        for k, (cam, target) in enumerate(zip(cams, targets)):
            self.forward(cam, stream)
            self.loss_backward(cam, target, stream, weight=1.0 / B, loss_out=self.batch_losses[k:k + 1],
                               ssim_out=self.batch_ssim[k:k + 1] if self.dssim > 0.0 else None)
            self.accumulate_density(cam, stream)
            if self.fused and k == B - 1:
                project_bwd_adam(self.n, self.params, cam, self.proj, self.grad2d, self.m, self.v, lr_b, b1, b2,
                                 eps_b, self.t, self.status, stream, grads_in=self.grads if B > 1 else None)
            elif k == 0:
                project_bwd(self.n, self.params, cam, self.proj, self.grad2d, self.grads, self.status, stream)
            else:
                project_bwd_accumulate(self.n, self.params, cam, self.proj, self.grad2d, self.grads, self.status,
                                       stream)
        if not self.fused:
            adam_step(self.n, self.params, self.grads, self.m, self.v, lr_b, b1, b2, eps_b, self.t, stream)

    def batch_loss(self) -> float:
        """The mean view loss of the last batch step (synchronises)."""
        v = float(self.batch_losses.cpu().numpy().astype(np.float64).sum())
        if self.dssim > 0.0:
            s = self.batch_ssim.cpu().numpy().astype(np.float64)
            v += self.dssim * float((1.0 - s).mean())
        return v

    # adaptive density control ---------------------------------------------------------
    def enable_density_control(self, extent: float, prune_big: bool = False, **thresholds) -> None:
        """Accumulate each visible Gaussian's NDC-scaled 2D mean-gradient norm after
        every step's loss backward (for refine) with the cited method's thresholds,
        ``extent`` being the scene's extent (the cameras' radius x 1.1 there)."""
        import torch
        cfg, log_shrink, logit_reset = densify_thresholds(extent, prune_big=prune_big, **thresholds)
        self.density = {"cfg": cfg, "log_shrink": log_shrink, "logit_reset": logit_reset}
        self.grad_acc = torch.zeros(self.n_pad, dtype=torch.float32, device=self.device)
        self.vis_cnt = torch.zeros(self.n_pad, dtype=torch.int32, device=self.device)

    def accumulate_density(self, cam: dict, stream=None) -> None:
        if self.density is not None:
            densify_accumulate(self.n, self.n_pad, self.proj, self.grad2d, cam["width"], cam["height"],
                               self.grad_acc, self.vis_cnt, stream)

    def refine(self, randn=None, seed: int = 0) -> dict:
        """Clone, split and prune by the accumulated gradients (synchronises to read
        the new count), rebuild the parameter, moment and per-Gaussian buffers at the
        new size, and clear the accumulators.  ``randn``: (n, 6) fp32 normals for the
        split children (drawn from ``seed`` when not given).  Returns the counts."""
        import torch
        if self.density is None:
            raise RuntimeError("enable_density_control first")
        n, dev = self.n, self.device
        action = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        offset = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
        n_out = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.empty(densify_workspace_bytes(n, self.n_pad), dtype=torch.uint8, device=dev)
        densify_plan(n, self.params, self.grad_acc, self.vis_cnt, self.density["cfg"], action, offset, n_out, ws)
        n_new = int(n_out.item())
        n_pad_new = max(256, -(-n_new // 256) * 256)
        if randn is None:
            gen = torch.Generator(device=dev)
            gen.manual_seed(int(seed))
            randn = torch.randn((max(n, 1), 6), generator=gen, device=dev, dtype=torch.float32)
        P = torch.empty((self.params.shape[0], n_pad_new), dtype=torch.float32, device=dev)
        M = torch.empty_like(P)
        V = torch.empty_like(P)
        densify_apply(n, self.params, self.m, self.v, action, offset, n_out, randn, self.density["log_shrink"], P, M,
                      V, self.status)
        counts = torch.bincount(action[:n].to(torch.int64), minlength=4).tolist() if n else [0, 0, 0, 0]
        self.params, self.m, self.v = P, M, V
        self.n, self.n_pad = n_new, n_pad_new
        self.grads = torch.empty_like(P)
        self.grad2d = torch.empty((n_pad_new, GRAD2D_STRIDE), dtype=torch.float32, device=dev)
        self.proj = ProjBuffers(n_pad_new, dev)
        self.bins = BinBuffers(n_new, self.capacity, self.width, self.height, dev)
        self.grad_acc = torch.zeros(n_pad_new, dtype=torch.float32, device=dev)
        self.vis_cnt = torch.zeros(n_pad_new, dtype=torch.int32, device=dev)
        return {"n": n_new, "pruned": counts[0], "kept": counts[1], "cloned": counts[2], "split": counts[3]}

    def reorder_spatially(self, stream=None):
        """Store the Gaussians in Morton order of their means (``gs_spatial_order``):
        the parameters, the Adam moments and any density accumulators are permuted
        together, so training continues unchanged but for the index that breaks ties
        between equal fp32 depths.  Gaussians near each other in space then sit near each other in memory,
        which the record gather and the backward's gradient atomics feel on scenes
        larger than L2.  Returns perm (perm[j] = the index before of the Gaussian now at
        j).  CUDA graphs captured before refer to the old buffers: capture again."""
        import torch
        n, dev = self.n, self.device
        perm = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
        ws = torch.empty(max(spatial_order_workspace_bytes(n, self.n_pad), 256), dtype=torch.uint8, device=dev)
        spatial_order(n, self.params, perm, ws, self.status, stream)
        names = ["params", "m", "v"] + (["grad_acc", "vis_cnt"] if self.density is not None else [])
        for name in names:
            src = getattr(self, name)
            dst = torch.empty_like(src)
            permute_planes(n, perm, src, dst, stream)
            setattr(self, name, dst)
        return perm[:n]

    def reset_opacity(self, stream=None) -> None:
        """Clamp opacities to 2 x the prune opacity and zero their Adam moments."""
        if self.density is None:
            raise RuntimeError("enable_density_control first")
        opacity_reset(self.n, self.params, self.m, self.v, self.density["logit_reset"], stream)

    # CUDA graphs --------------------------------------------------------------------
    def capture_step(self, cam: dict, target):
        """A CUDA graph of one fused step for this camera against ``target`` (a device
        tensor the caller keeps alive): the step counter advance, forward, loss
        backward and the fused projection backward + Adam reading the step count
        from device memory.  Replay it with ``replay``; eager and replayed steps may
        be mixed (the device step count follows ``t``)."""
        import torch
        if not self.fused:
            raise ValueError("graph capture runs the fused step")
        if getattr(self, "t_dev", None) is None:
            self.t_dev = torch.zeros(1, dtype=torch.int64, device=self.params.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_counter_add(self.t_dev, 1)
            self.forward(cam)
            self.loss_backward(cam, target)
            project_bwd_adam_tdev(self.n, self.params, cam, self.proj, self.grad2d, self.m, self.v, self.lr_plane,
                                  self.beta1, self.beta2, self.eps, self.t_dev, self.status)
        return g

    def replay(self, graph) -> None:
        """One step from a graph of ``capture_step`` (on the current stream)."""
        if int(self._t_dev_synced) != self.t:
            self.t_dev.fill_(self.t)
        graph.replay()
        self.t += 1
        self._t_dev_synced = self.t

    _t_dev_synced = -1

    def step_staged(self, cam: dict, targets: HostTargets, slot: int, stream=None) -> None:
        """``step`` against the target uploaded into ``slot`` of ``targets``.  The step
        waits for that upload only before its loss backward (projection, binning and
        the forward do not read the target), and records ``after_backward`` once the
        rasterisers are done: pass it to ``targets.put`` for the next step's upload."""
        import torch
        s = stream or torch.cuda.current_stream()
        if getattr(self, "after_backward", None) is None:
            self.after_backward = torch.cuda.Event()
        self.forward(cam, stream)
        target = targets.get(slot, s)
        if not self.fused:
            self.backward(cam, target, stream)
            self.after_backward.record(s)
            self.optimizer_step(stream)
        else:
            self.loss_backward(cam, target, stream)
            self.accumulate_density(cam, stream)
            self.after_backward.record(s)
            self.t += 1
            project_bwd_adam(self.n, self.params, cam, self.proj, self.grad2d, self.m, self.v, self.lr_plane,
                             self.beta1, self.beta2, self.eps, self.t, self.status, stream)
        targets.release(slot, s)

    # checkpoint ----------------------------------------------------------------------
    def save(self, path) -> None:
        """Write the state a run resumes from to one ``.npz`` file (host copies;
        synchronises): the parameter and Adam moment planes, the Adam step count and
        the Gaussian count."""
        np.savez(path, params=self.params.cpu().numpy(), m=self.m.cpu().numpy(), v=self.v.cpu().numpy(),
                 t=np.int64(self.t), n=np.int64(self.n))

    @classmethod
    def load(cls, path, width: int, height: int, capacity: int, lr_plane, **kwargs) -> "Trainer":
        """A trainer resumed from ``save``'s file.  Image size, capacity, learning rates
        and the other constructor options are the caller's, as for a new trainer;
        density control, if wanted, is enabled again (its accumulators start at zero,
        as after a refinement)."""
        import torch
        with np.load(path) as z:
            tr = cls(z["params"], int(z["n"]), width, height, capacity, lr_plane, **kwargs)
            tr.m.copy_(torch.from_numpy(z["m"]))
            tr.v.copy_(torch.from_numpy(z["v"]))
            tr.t = int(z["t"])
        return tr

    # host-side reads (synchronise) -----------------------------------------------
    def total_loss(self) -> float:
        """(1 - lambda) L1 + lambda (1 - SSIM) of the last step (L1 alone for lambda = 0)."""
        v = float(self.loss[0].item())
        if self.dssim > 0.0:
            v += self.dssim * (1.0 - float(self.ssim_val[0].item()))
        return v

    def n_isect(self) -> int:
        return int(self.bins.n_isect[0].item()) & 0xFFFFFFFF

    def check_status(self) -> int:
        s = int(self.status[0].item()) & 0xFFFFFFFF
        return s

    def raise_on_status(self) -> None:
        s = self.check_status()
        if s:
            raise RuntimeError(f"device status {s}: {status_str(s)}")
