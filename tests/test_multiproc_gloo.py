"""The multi-replica host logic of bench.py on CPU: two gloo ranks, each its own replica
(no data-path collective; only the timing is reduced).  The job's time is the slowest
rank's, and throughput counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r+1) * 10 ms: the job takes the slowest rank's time
        t = bench.max_over_ranks(10.0 * (rank + 1), torch.device("cpu"))
        out[rank] = t
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_throughput():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 20.0, 1: 20.0}
    import bench
    # 2 replicas x 1 GB per step in 0.5 s -> 4 GB/s for the whole job
    assert bench.job_throughput(1e9, 2, 0.5) == pytest.approx(4.0)
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5  # single process


def test_reference_arm_prints_one_oracle_line():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cpu_model"]
    assert d["cpu_baseline"]["single_thread"]["cores"] == 1
    # what ran: steps x ms_per_step is the measured total, not an extrapolation
    assert d["steps"] * d["ms_per_step"] <= 1.5 * d["ms_per_step_total"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"].startswith("invariant GEMM")
