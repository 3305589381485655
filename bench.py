#!/usr/bin/env python
"""Train steps/s of the GB300 3DGS step (fwd + bwd + Adam, one view per step).

Workload (default): 4M-Gaussian blob isosurface at 2048x2048 with 448 orbit views,
SH degree 3, fp32; step s trains view s mod 448 against that view's target image
(a render of the same surface sampled with another seed).  Every input is seeded
and synthetic and resident on the GPU before the timed region; parameters, Adam
state and targets (22.5 GB) exceed L2 many times over, so no flush is needed.  Before
the warm-up the Gaussians are stored in Morton order of their means (a layout that
changes a step's result only through the index that breaks ties between equal fp32
depths; ``--order generated`` keeps the generator's order).

One JSON line is printed (rank 0).  Besides the device-timed value it carries:
  e2e           the same steps (from the same model state) through the public API
                with each step's target copied from pinned host memory (on a copy
                stream, overlapping the previous step) and its loss read back;
  roofline      for the kernel with the largest share of step time;
  cpu_baseline  one whole, unsampled CPU oracle step timed on this host's cores;
  stages_ms     per-stage device time per step (CUDA events on the stream);
  clocks        SM clocks and throttle reasons sampled during the timed region.

``--impl reference`` times the CPU oracle instead (the reference arm of this
build): whole unsampled oracle steps over the same orbit views.
Multi-GPU runs are independent replicas (the step does not shard).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gs_inputs as gi  # noqa: E402

METRIC = "train steps/s (fwd+bwd+Adam, 1 view) at 4M Gaussians 2048²; % of roofline"
METRIC_BATCH = "train steps/s ({B} views per step: fwd+bwd per view, one Adam) at 4M Gaussians 2048²"
STAGES_SEPARATE = ["project", "bin_sort", "render_fwd", "render_bwd", "project_bwd", "adam"]
STAGES_FUSED = ["project", "bin_sort", "render_fwd", "render_bwd", "project_bwd_adam"]


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=448)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="iso4m_2048", choices=sorted(gi.CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--capacity-slack", type=float, default=1.15)
    ap.add_argument("--separate", action="store_true",
                    help="run the projection backward and Adam as two calls instead of gs_project_bwd_adam")
    ap.add_argument("--views", type=int, default=0,
                    help="use only the first N orbit views (profiling runs; 0 = all)")
    ap.add_argument("--batch", type=int, default=1,
                    help="views per optimisation step (batch-size scaling of the Adam hyperparameters); the "
                         "headline is one view per step")
    ap.add_argument("--graph", action="store_true",
                    help="replay each view's step from a CUDA graph captured after the warm-up (one view per step)")
    ap.add_argument("--order", choices=["morton", "generated"], default="morton",
                    help="storage order of the Gaussians, set once before the warm-up: Morton order of the means "
                         "(gs_spatial_order) or the order the scene generator wrote them in")
    ap.add_argument("--dssim", type=float, default=0.0,
                    help="D-SSIM weight lambda: the loss becomes (1 - lambda) L1 + lambda (1 - SSIM) (0 = L1)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend="nccl"):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend)
    return dist


def max_over_ranks(dist, x: float, device=None) -> float:
    """The largest of every rank's x (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_replicas(dist, body, sync, device=None) -> float:
    """Milliseconds of ``body`` on the slowest rank.  Every rank synchronises its
    device and meets the others at a barrier before and after; ``body`` returns its
    own duration in ms (CUDA events on the GPU)."""
    sync()
    if dist:
        dist.barrier()
    ms = body()
    sync()
    if dist:
        dist.barrier()
    return max_over_ranks(dist, ms, device)


def whole_job_rate(ws: int, steps: int, ms: float) -> float:
    """Steps per second of the whole job: every rank runs ``steps`` independent
    steps, the job takes the slowest rank's ``ms``."""
    return ws * steps / (ms / 1e3)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = max((num(r[2]) for r in rows if num(r[2]) is not None), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        load = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ----------------------------------------------------------------------------- roofline model

def passes_for(width, height):
    """Radix passes of the tile sort: ceil(tile bits / 8)."""
    tiles = (-(-width // 16)) * (-(-height // 16))
    b = 0
    while (1 << b) < tiles:
        b += 1
    return (b + 7) // 8


def stage_bytes(N, n_pad, V, K, P, passes, dssim=False, E=0.0):
    """Algorithmic DRAM bytes of each stage per step (the traffic the method needs
    with the data layout used: SoA planes, 48-byte records, 8+4-byte keys).  E is the
    number of iterated (pixel, entry) pairs: the composited-entry masks hold 4 bytes
    per pixel and 32-entry chunk, E / 8 bytes in all."""
    return {
        # all N: 11 geometric planes + depth/radius/rect/count; visible: 48 SH + record
        "project": 64 * N + 240 * V,
        # counts twice; visible: depth read, (depth, index) written, 4 depth passes of
        # 16 bytes, sorted index + count read twice and rect once; per intersection
        # (tile, index) emitted, each tile pass reads and writes 16 bytes, then tile
        # key + index read, 48-byte record gathered and written, 64-bit key written
        "bin_sort": 8 * N + 100 * V + (8 + 16 * passes + 112) * K,
        # records once per tile, image + T + n_contrib written, the composited-entry
        # masks written
        "render_fwd": 48 * K + 20 * P + E / 8,
        # grad2d (12 floats per Gaussian) cleared, records once per tile,
        # image/target/T/n_contrib read (and the D-SSIM image gradient when that term is
        # on), the masks read
        "render_bwd": 48 * n_pad + 48 * K + (44 if dssim else 32) * P + E / 8,
        # D-SSIM: image + target read, 15 maps (3 partials, 2 means per channel)
        # written; the maps, image and target read again, the image gradient written
        "ssim": 180 * P,
        # all: count + 59 gradient planes written; visible: 59 params + the 48-byte
        # grad2d slot read
        "project_bwd": 240 * N + 284 * V,
        # p, g, m, v read; p, m, v written
        "adam": 59 * n_pad * 28,
    }


# Bytes the fused projection backward + Adam actually moves: count, the 48-byte grad2d slot of the
# visible, p, m, v read and written for every parameter (the gradient planes are
# never written).  The step roofline still charges rows a5 + a6 their own bytes.
def fused_bytes(N, n_pad, V):
    return 4 * N + 48 * V + 59 * n_pad * 24


# Rows of the step each measured stage covers.
STAGE_ROWS = {"project": ["project"], "bin_sort": ["bin_sort"], "render_fwd": ["render_fwd"],
              "render_bwd": ["render_bwd"], "project_bwd": ["project_bwd"], "adam": ["adam"],
              "project_bwd_adam": ["project_bwd", "adam"], "ssim": ["ssim"]}


# Algorithmic operations per iterated (pixel, entry) pair of the compositing rule as
# the method states it (per-pair partials of the mean and the conic), FMA = 2, the
# exponential and the reciprocal 1 each, FP32 compares, min and selects 1 each:
# forward 26 + exp = 27: offset 2; power -1/2 (A dx^2 + C dy^2) - B dx dy 9 (dx^2, dy^2,
#   A dx^2 + C dy^2, -1/2, dx dy, the last FMA); the skip test 1; power log2(e) 1;
#   o e^power 1; the 0.99 clamp 1; the 1/255 test 1; T (1 - alpha) 2; the stop test 1;
#   alpha T 1; three colour FMAs 6.
# backward 64 + exp + reciprocal = 66: the forward's evaluation up to the 1/255 test 16;
#   T recovered as T / (1 - alpha) 2; alpha T 1; three colour partials 3; dL/dalpha
#   (three colour differences from the carried colour, their dot product with dL/dC,
#   times T) 9; the carried colour's update 3 FMAs 6; dL/dpower and dL/do with their two
#   clamp selects 4; the mean partials (A dx + B dy, B dx + C dy, times dL/dpower) 8; the
#   conic partials (dx^2, dx dy, dy^2 reused, their factors, times dL/dpower) 6; the
#   nine partials added to the Gaussian's sums 9.
# The achieved rate is these figures over the measured time.  This implementation's
# exact exponential (two multiplies, a rounding and nine FMAs: 21 by this count) costs
# more than the 1 counted here; its moment form of the partials costs less.
FLOP_FWD_PAIR = 27
FLOP_BWD_PAIR = 66
# FP32 operations per pixel of the D-SSIM forward and backward over 3 channels.  Per
# channel, forward: horizontal pass 158 (42 staged rows per 32 output rows; per 4
# outputs 42 products and 5 moments x 44 FMAs), vertical 110, SSIM partials 35;
# backward: folding the means 14, horizontal 87, vertical 66, combine 6.
FLOP_SSIM_PIX = 3 * (158 + 110 + 35 + 14 + 87 + 66 + 6)


# Operations of an iterated pair that does not composite (the power is positive or
# alpha falls below 1/255): the rule's evaluation up to the 1/255 test, offset 2, power
# 9, skip test 1, power log2(e) 1, the exponential 1, o e^power 1, the 0.99 clamp 1,
# the 1/255 test 1.
FLOP_SKIP_PAIR = 17


def composited_flops(per_pair: int, iterated: float, composited: float) -> float:
    """Work of a rasteriser charging composited pairs the full per-pair count and the
    other iterated pairs only their evaluation."""
    return per_pair * composited + FLOP_SKIP_PAIR * max(0.0, iterated - composited)


def fp32_peak_tflops(sm_mhz, sms):
    # SMs x 128 FP32 lanes x 2 FLOP per FMA per clock
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------- CPU oracle leg

class OracleStep:
    """Whole oracle steps, nothing sampled or scaled: per view, the projection of every
    Gaussian, the tile lists and the compositing forward and backward of every pixel,
    the projection backward of every Gaussian and Adam over every parameter, with the
    parameters and moments carried from step to step.  The loss is L1 against a seeded
    U(0, 1) target per view (the work of a step does not depend on the target's
    values)."""

    def __init__(self, P, n, width, height, seed=0):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.P = np.ascontiguousarray(P, np.float32)
        self.n, self.W, self.H, self.seed = n, width, height, seed
        self.m = np.zeros(self.P.shape, np.float64)
        self.v = np.zeros(self.P.shape, np.float64)
        self.t = 0

    def target(self, view: int) -> np.ndarray:
        return gi.uniform_target(self.seed + 7919 * view, self.W, self.H)

    def seconds(self, cam, target) -> float:
        """One whole training step of the oracle for one view; returns its wall time."""
        t0 = time.perf_counter()
        r = self.oracle.step(self.P, self.n, cam, target, self.m, self.v, self.t + 1, gi.lr_planes())
        self.P = r["params"].astype(np.float32)
        self.m, self.v = r["m"], r["v"]
        self.t += 1
        return time.perf_counter() - t0

    def desc(self, what: str) -> str:
        return (f"{what}: whole oracle steps, every Gaussian and every pixel of the "
                f"{self.W}x{self.H} view (projection, tile lists, compositing forward and backward, "
                f"projection backward, Adam), nothing sampled or scaled; L1 against seeded U(0,1) targets")


def _torch_dev():
    try:
        import torch
        return "cuda" if torch.cuda.is_available() else "cpu"
    except ImportError:
        return None


def run_reference(args, cfg, rank):
    """Reference arm: the CPU oracle, whole unsampled steps over the orbit views in
    order (the same views as the GPU arm's steps)."""
    if rank != 0:
        return
    cams = gi.cameras_for(cfg)
    P = gi.scene_for(cfg, seed=args.seed, device=_torch_dev() if cfg.n >= 1_000_000 else None)
    ost = OracleStep(P, cfg.n, cfg.width, cfg.height, seed=args.seed)
    per = []
    for s in range(args.warmup + args.steps):
        v = s % len(cams)
        tgt = ost.target(v)
        sec = ost.seconds(cams[v], tgt)
        if s >= args.warmup:
            per.append(sec)
    val = len(per) / float(np.sum(per))
    desc = ost.desc(f"{args.warmup} warm-up and {args.steps} timed steps, orbit views in order")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / val, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 decisions)", "data": "synthetic",
        "config": _config_dict(cfg),
        "cpu_baseline": {"value": val, "unit": "steps/s", "cores": ost.oracle.threads(), "kind": "oracle",
                         "sample": desc, "extrapolated": False},
        "e2e": {"value": val, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "step_s": {"mean": float(np.mean(per)), "min": float(np.min(per)), "max": float(np.max(per))},
    }
    print(json.dumps(line), flush=True)


def _config_dict(cfg):
    return {"workload": f"{cfg.name}: {cfg.description}; one view per step, views in orbit order",
            "n_gaussians": cfg.n, "width": cfg.width, "height": cfg.height, "views": cfg.n_views,
            "sh_degree": 3, "l2": "inputs larger than L2 (parameters + Adam state + targets >> 129 MB); no flush"}


# ----------------------------------------------------------------------------- GPU arm

def run_gb300(args, cfg, ws, rank, local):
    import torch
    import gaussian_splatting_differentiable_project_gb300 as gs

    dist = dist_init(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t_setup = time.time()
    gs.load()
    P = gi.scene_for(cfg, seed=args.seed, device=dev)
    Pt = gi.target_scene_for(cfg, seed=args.seed, device=dev)
    cams = gi.cameras_for(cfg)
    if args.views > 0:
        cams = cams[: args.views]
    V_views = len(cams)
    W, H = cfg.width, cfg.height
    n, n_pad = cfg.n, P.shape[1]
    passes = passes_for(W, H)

    # capacity: project every view (model and target sets) and take the largest K
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    Pd = torch.from_numpy(P).to(dev)
    Ptd = torch.from_numpy(Pt).to(dev)
    proj = gs.ProjBuffers(n_pad, dev)
    kmax, Ks, Vs = 0, [], []
    for cam in cams:
        for which in (Ptd, Pd):
            gs.project(n, which, cam, proj, st)
            k = int(proj.count[:n].sum().item())
            kmax = max(kmax, k)
            if which is Pd:
                Ks.append(k)
                Vs.append(int((proj.count[:n] > 0).sum().item()))
    capacity = int(kmax * args.capacity_slack) + 4096
    del proj

    # targets: forward renders of the target set, one per view
    rend = gs.Trainer(Ptd, n, W, H, capacity, gi.lr_planes(), device=dev)
    targets = torch.empty((V_views, 3, H, W), dtype=torch.float32, device=dev)
    for v, cam in enumerate(cams):
        rend.forward(cam)
        targets[v].copy_(rend.image)
    torch.cuda.synchronize()
    rend.raise_on_status()
    del rend, Ptd

    tr = gs.Trainer(Pd, n, W, H, capacity, gi.lr_planes(), device=dev, fused=not args.separate, dssim=args.dssim)
    if args.order == "morton":
        tr.reorder_spatially()
    STAGES = list(STAGES_SEPARATE if args.separate else STAGES_FUSED)
    if args.dssim > 0:
        STAGES.insert(STAGES.index("render_bwd"), "ssim")
    del Pd
    # per-view work statistics (forward on the initial parameters): pairs iterated
    # (sum of n_contrib) and pairs composited (the counting forward's n_used)
    E, E_used = [], []
    n_used = torch.empty_like(tr.n_contrib)
    for cam in cams:
        gs.project(tr.n, tr.params, cam, tr.proj, tr.status)
        gs.bin_sort(tr.n, tr.n_pad, tr.proj, cam, tr.bins, tr.status)
        gs.render_fwd_counted(cam, tr.bins, tr.bg, tr.image, tr.T_final, tr.n_contrib, n_used, tr.status)
        E.append(int(tr.n_contrib.to(torch.int64).sum().item()))
        E_used.append(int(n_used.to(torch.int64).sum().item()))
    del n_used
    torch.cuda.synchronize()
    tr.raise_on_status()
    setup_s = time.time() - t_setup

    B = max(1, args.batch)

    def views_of(s):
        return [(s * B + k) % V_views for k in range(B)]

    def step(s, events=None):
        if B > 1:
            vs = views_of(s)
            tr.step_batch([cams[v] for v in vs], [targets[v] for v in vs])
            return
        v = s % V_views
        cam = cams[v]
        if events is None:
            tr.step(cam, targets[v])
            return
        e = events
        e[0].record()
        gs.project(tr.n, tr.params, cam, tr.proj, tr.status)
        e[1].record()
        gs.bin_sort(tr.n, tr.n_pad, tr.proj, cam, tr.bins, tr.status)
        e[2].record()
        gs.render_fwd(cam, tr.bins, tr.bg, tr.image, tr.T_final, tr.n_contrib, tr.status)
        e[3].record()
        k = 4
        extra = None
        if args.dssim > 0:
            gs.ssim_fwd(tr.image, targets[v], tr.dssim, tr.ssim_maps, tr.ssim_val)
            gs.ssim_bwd(tr.image, targets[v], tr.ssim_maps, tr.dLdC)
            extra = tr.dLdC
            e[k].record()
            k += 1
        gs.render_bwd(tr.n, tr.n_pad, cam, tr.bins, tr.bg, tr.image, targets[v], tr.T_final, tr.n_contrib,
                      tr.grad2d, tr.loss, tr.status, l1_weight=1.0 - tr.dssim, dLdC_extra=extra)
        e[k].record()
        if args.separate:
            gs.project_bwd(tr.n, tr.params, cam, tr.proj, tr.grad2d, tr.grads, tr.status)
            e[k + 1].record()
            tr.optimizer_step()
            e[k + 2].record()
        else:
            tr.t += 1
            gs.project_bwd_adam(tr.n, tr.params, cam, tr.proj, tr.grad2d, tr.m, tr.v, tr.lr_plane, tr.beta1,
                                tr.beta2, tr.eps, tr.t, tr.status)
            e[k + 1].record()

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    graphs = {}
    if args.graph:
        if B != 1 or args.separate:
            raise SystemExit("--graph replays the fused one-view step")
        for s in range(args.steps):
            v = (args.warmup + s) % V_views
            if v not in graphs:
                graphs[v] = tr.capture_step(cams[v], targets[v])
        torch.cuda.synchronize()

    # the model state the timed steps start from: the end-to-end leg restarts from it,
    # so that both legs time the same steps (training changes the per-step work)
    snap = (tr.params.clone(), tr.m.clone(), tr.v.clone(), tr.t) if not args.no_e2e else None

    # ---------------------------------------------------------------- timed region
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    def timed():
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("timed")
        t_start.record()
        for s in range(K):
            if graphs:
                tr.replay(graphs[(args.warmup + s) % V_views])
            else:
                step(args.warmup + s, ev[s] if B == 1 else None)
        t_end.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        return t_start.elapsed_time(t_end)

    ms = time_replicas(dist, timed, torch.cuda.synchronize, dev)
    clk = clocks.stop()
    tr.raise_on_status()
    stage_ms = ({name: float(np.mean([ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(K)]))
                 for i, name in enumerate(STAGES)} if B == 1 and not graphs else None)
    # per-step device time (first to last stage event of each step)
    step_ms = ([ev[s][0].elapsed_time(ev[s][len(STAGES)]) for s in range(K)] if stage_ms is not None else None)
    value = whole_job_rate(ws, K, ms)

    # ---------------------------------------------------------------- e2e leg
    e2e = None
    if not args.no_e2e:
        graphs.clear()  # they read the device-resident targets freed below
        tr.params.copy_(snap[0])
        tr.m.copy_(snap[1])
        tr.v.copy_(snap[2])
        tr.t = snap[3]
        del snap
        host_t = torch.empty_like(targets, device="cpu").pin_memory()
        host_t.copy_(targets)
        del targets
        torch.cuda.empty_cache()
        staged = gs.HostTargets((3, H, W), dev, slots=2 * B)
        loss_host = torch.empty((K, max(2, B)), dtype=torch.float32).pin_memory()

        def timed_e2e():
            # each step's target is uploaded from pinned host memory on a copy stream
            # while the previous step computes; every upload and read-back lies
            # between the two events
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            staged.stream.wait_event(a)
            slots = [staged.put(host_t[v]) for v in views_of(args.warmup)]
            for s in range(K):
                vs = views_of(args.warmup + s)
                if B == 1:
                    tr.step_staged(cams[vs[0]], staged, slots[0])
                    # the next target's upload starts as soon as its slot is free (the step
                    # before this one has released it), so it has a whole step to land
                    nxt = ([staged.put(host_t[v]) for v in views_of(args.warmup + s + 1)]
                           if s + 1 < K else None)
                    loss_host[s, 0:1].copy_(tr.loss, non_blocking=True)
                    if args.dssim > 0:
                        loss_host[s, 1:2].copy_(tr.ssim_val, non_blocking=True)
                else:
                    nxt = [staged.put(host_t[v]) for v in views_of(args.warmup + s + 1)] if s + 1 < K else None
                    tr.step_batch([cams[v] for v in vs], [staged.get(sl) for sl in slots])
                    for sl in slots:
                        staged.release(sl)
                    loss_host[s, :B].copy_(tr.batch_losses, non_blocking=True)
                slots = nxt
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        ms_e2e = time_replicas(dist, timed_e2e, torch.cuda.synchronize, dev)
        e2e = {"value": whole_job_rate(ws, K, ms_e2e), "unit": "steps/s", "h2d_bytes_per_step": B * 3 * H * W * 4,
               "d2h_bytes_per_step": 4 * B if B > 1 else (8 if args.dssim > 0 else 4), "ms_per_step": ms_e2e / K}
        del host_t

    if rank != 0:
        return

    # ---------------------------------------------------------------- roofline
    views = [v for s in range(K) for v in views_of(args.warmup + s)]
    Kmean = float(np.mean([Ks[v] for v in views]))
    Vmean = float(np.mean([Vs[v] for v in views]))
    Emean = float(np.mean([E[v] for v in views]))
    Eused = float(np.mean([E_used[v] for v in views]))
    Pix = W * H
    byt = stage_bytes(n, n_pad, Vmean, Kmean, Pix, passes, dssim=args.dssim > 0, E=Emean)
    peak_bw = _peak("hbm_gbs", 6800.0)
    sm_mhz = clk.get("sm_max_mhz") or 2070.0
    sms = gs.sm_count()
    sms_torch = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_fp32 = fp32_peak_tflops(sm_mhz, sms)
    flops = {"render_fwd": FLOP_FWD_PAIR * Emean, "render_bwd": FLOP_BWD_PAIR * Emean, "ssim": FLOP_SSIM_PIX * Pix}
    # the same rule charging a skipped pair (iterated, not composited) only its
    # evaluation up to the 1/255 test
    flops_comp = {"render_fwd": composited_flops(FLOP_FWD_PAIR, Emean, Eused),
                  "render_bwd": composited_flops(FLOP_BWD_PAIR, Emean, Eused), "ssim": FLOP_SSIM_PIX * Pix}
    per_stage = {}
    t_star = 0.0
    row_t = {}
    rows_all = STAGE_ROWS["project_bwd_adam"] + ["project", "bin_sort", "render_fwd", "render_bwd"]
    if args.dssim > 0:
        rows_all.append("ssim")
    for row in rows_all:
        row_t[row] = max(byt[row] / (peak_bw * 1e9), flops.get(row, 0.0) / (peak_fp32 * 1e12))
    t_star = sum(row_t.values())
    # the same sum with the fused projection backward + Adam charged the bytes it moves
    t_star_fused = (t_star - row_t["project_bwd"] - row_t["adam"]
                    + fused_bytes(n, n_pad, Vmean) / (peak_bw * 1e9)) if not args.separate else None
    if B > 1:
        # a batch step: every row but Adam once per view, Adam once
        t_star = B * sum(t for r, t in row_t.items() if r != "adam") + row_t["adam"]
    for name in (STAGES if stage_ms is not None else []):
        rows = STAGE_ROWS[name]
        t_meas = stage_ms[name] / 1e3
        t_rows = sum(row_t[r] for r in rows)
        moved = fused_bytes(n, n_pad, Vmean) if name == "project_bwd_adam" else sum(byt[r] for r in rows)
        fl = sum(flops.get(r, 0.0) for r in rows)
        bound = "alu" if fl / (peak_fp32 * 1e12) > moved / (peak_bw * 1e9) else "hbm"
        t_own = max(moved / (peak_bw * 1e9), fl / (peak_fp32 * 1e12))
        per_stage[name] = {"ms": stage_ms[name], "bound": bound, "rows": rows,
                           "gbs": moved / t_meas / 1e9, "tflops": fl / t_meas / 1e12, "frac": t_own / t_meas}
        fl_c = sum(flops_comp.get(r, 0.0) for r in rows)
        if fl_c:
            per_stage[name]["tflops_composited"] = fl_c / t_meas / 1e12
            per_stage[name]["frac_composited"] = max(moved / (peak_bw * 1e9), fl_c / (peak_fp32 * 1e12)) / t_meas
        if len(rows) > 1:
            # the fused stage against the rows it replaces (their gradient planes
            # included), as the step roofline charges it
            per_stage[name]["frac_rows"] = t_rows / t_meas
    roof = None  # batch and graph steps have no per-stage events
    if stage_ms is not None:
        dom = max(STAGES, key=lambda s: stage_ms[s])
        d = per_stage[dom]
        traffic = measured_traffic({"render_fwd": "k_render_fwd", "render_bwd": "k_render_bwd"}.get(dom, ""))
        if d["bound"] == "hbm":
            roof = {"kernel": dom, "bound": "hbm", "achieved": d["gbs"], "peak": peak_bw, "unit": "GB/s",
                    "frac": d["gbs"] / peak_bw, "traffic": traffic, "peak_source": _peak_src("hbm_gbs")}
        else:
            roof = {"kernel": dom, "bound": "alu", "achieved": d["tflops"], "peak": peak_fp32, "unit": "TFLOP/s",
                    "frac": d["tflops"] / peak_fp32, "traffic": traffic,
                    "peak_source": f"{sms} SMs (queried) x 128 FP32 lanes x 2 x {sm_mhz:.0f} MHz (max SM clock "
                                   f"sampled during the timed region); MEASURED_PEAKS.json has no FP32 entry",
                    "flop_per_pair": FLOP_FWD_PAIR if dom == "render_fwd" else FLOP_BWD_PAIR,
                    "achieved_composited": d.get("tflops_composited"),
                    "frac_composited": (d.get("tflops_composited") or 0.0) / peak_fp32,
                    "flop_model_composited": f"{FLOP_SKIP_PAIR} FLOP per iterated pair that does not composite, "
                                             f"the full count per composited pair"}

    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        try:
            cpu = cpu_baseline(cfg, P, cams[0], W, H, args.seed)
        except Exception as exc:  # the baseline is reported, never required
            cpu = {"value": None, "unit": "steps/s", "kind": "oracle", "error": repr(exc)}

    # project 1; binning 12 + p (prep, 3 scans, compact, 4 depth passes, sorted sums, emit,
    # p tile passes, gather); forward 1; backward 2 (clear + raster); fused 1
    per_view = 1 + (12 + passes) + 1 + 2 + 1 + (3 if args.dssim > 0 else 0) + (1 if args.graph else 0)
    launches_per_step = B * per_view + (1 if args.separate else 0)
    line = {
        "metric": METRIC if B == 1 else METRIC_BATCH.format(B=B), "value": value, "unit": "steps/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(_config_dict(cfg), parallelism=f"replicas{ws}", capacity_K=capacity,
                       objective=(f"{1 - args.dssim:g} L1 + {args.dssim:g} (1 - SSIM)" if args.dssim > 0 else "L1"),
                       K_mean=Kmean, visible_mean=Vmean, pairs_bwd_mean=Emean, pairs_composited_mean=Eused,
                       entries_per_pixel=Emean / float(W * H), composited_per_pixel=Eused / float(W * H),
                       visible_frac_all_views={"min": min(Vs) / n, "mean": float(np.mean(Vs)) / n,
                                               "views": V_views},
                       batch=B, storage_order=args.order, seed=args.seed,
                       gpu=torch.cuda.get_device_name(dev), sm_count=sms, sm_count_torch=sms_torch,
                       cuda_graph=bool(graphs)),
        "views_per_s": value * B,
        "roofline": roof,
        "step_roofline_frac": t_star / (ms / K / 1e3),
        "step_roofline_frac_fused_bytes": (t_star_fused / (ms / K / 1e3)) if (t_star_fused and B == 1) else None,
        "step_ms_median": float(np.median(step_ms)) if step_ms else None,
        "step_ms_p90": float(np.percentile(step_ms, 90)) if step_ms else None,
        "stages_ms": stage_ms, "stages": per_stage,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * K,
        "clocks": clk, "setup_s": setup_s,
    }
    print(json.dumps(line), flush=True)


def measured_traffic(kernel: str):
    """DRAM bytes per launch of ``kernel`` from profiles/dram_traffic.md, or None if the
    kernel's sources changed since that capture (fingerprint mismatch) or it has none."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) != 6 or cells[0] != kernel:
            continue
        h = hashlib.sha256()
        try:
            for f in cells[1].split():
                h.update(open(os.path.join(ROOT, "gaussian_splatting_differentiable_project_gb300", "csrc", f),
                              "rb").read())
        except OSError:
            return None
        return int(cells[5]) if h.hexdigest()[:16] == cells[2] else None
    return None


def _peak(key, fallback):
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))[key])
    except (OSError, KeyError, ValueError):
        return fallback


def _peak_src(key):
    return "of measured" if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else "of fallback"


def cpu_baseline(cfg, P, cam, W, H, seed):
    """One whole oracle step of view 0 on this host's cores (unsampled)."""
    ost = OracleStep(P, cfg.n, W, H, seed=seed)
    sec = ost.seconds(cam, ost.target(0))
    return {"value": 1.0 / sec, "unit": "steps/s", "cores": ost.oracle.threads(), "kind": "oracle",
            "sample": ost.desc("one step of orbit view 0"), "seconds_per_step": sec, "extrapolated": False}


def main():
    args = parse()
    ws, rank, local = dist_env()
    cfg = gi.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    run_gb300(args, cfg, ws, rank, local)


if __name__ == "__main__":
    main()
