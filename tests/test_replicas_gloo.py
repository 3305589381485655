"""Several GPUs run the step as independent replicas (each rank trains its own copy
on its own views; there is no exchange on the data path).  What the multi-rank
bench adds is host logic: a barrier and a device synchronise around the timed
region, the slowest rank's time, and the whole-job rate over all ranks.  These
tests run that logic on world size 2 with the gloo backend on the CPU, and check
that the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys
import time

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_env() == (ws, rank, rank)
    d = bench.dist_init(ws, backend="gloo")
    try:
        # exact reduction: each rank reports a fixed duration
        fixed = bench.time_replicas(d, lambda: [3.0, 7.5][rank], lambda: None)
        # the barrier before the body: rank 1 arrives late, rank 0 must wait for it
        if rank == 1:
            time.sleep(0.3)
        t0 = time.perf_counter()
        slept = bench.time_replicas(d, lambda: (time.sleep(0.05 * (rank + 1)), 50.0 * (rank + 1))[1],
                                    lambda: None)
        waited = time.perf_counter() - t0
        rate = bench.whole_job_rate(ws, 10, slept)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"fixed": fixed, "slept": slept, "waited": waited, "rate": rate}, f)
    finally:
        d.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank_world_size_2(tmp_path):
    ws = 2
    mp.start_processes(_worker, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(ws)]
    for k in range(ws):
        assert r[k]["fixed"] == 7.5
        assert r[k]["slept"] == 100.0
        assert r[k]["rate"] == pytest.approx(ws * 10 / 0.1)
    # rank 0 entered first and left only after rank 1's 100 ms body: the barrier after
    # the body holds it (the barrier before it covers the late start)
    assert r[0]["waited"] >= 0.09


def test_whole_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(1, 100, 1000.0) == pytest.approx(100.0)
    assert bench.whole_job_rate(4, 100, 1000.0) == pytest.approx(400.0)
    assert bench.max_over_ranks(None, 2.5) == 2.5


def _bench(args, rank, ws):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env, capture_output=True,
                          text=True, timeout=300, cwd=ROOT)


def test_reference_arm_runs_on_rank_0_only():
    """Under a multi-rank launch the oracle arm prints one line from rank 0; every
    other rank exits 0 without work or output."""
    args = ["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1", "--gpus", "2"]
    p1 = _bench(args, rank=1, ws=2)
    assert p1.returncode == 0, p1.stderr
    assert p1.stdout.strip() == ""
    p0 = _bench(args, rank=0, ws=2)
    assert p0.returncode == 0, p0.stderr
    lines = [ln for ln in p0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
