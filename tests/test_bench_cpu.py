"""bench.py's multi-rank aggregation on CPU (gloo, 2 ranks) and its argument handling."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(float(rank + 1) * 1.5, world, torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 3.0, 1: 3.0}


def test_single_rank_helpers():
    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.barrier(1)
    r, w, l = bench.dist_env()
    assert w >= 1


def test_peaks_and_traffic_records():
    peak, src = bench.read_peaks()
    assert peak > 1000
    # the committed traffic record matches the current kernel sources or is dropped
    t = bench.read_traffic("decode_batch")
    assert bench.read_traffic("decode_batch", "9:9") is None  # another plan: no record
    assert t is None or t > 5e6


def test_gpus_flag_spawns_the_ranks_itself():
    """`bench.py --gpus 2` without a launcher starts two ranks (gloo here, no GPU) and rank 0
    reports the aggregate over both."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry-run", "--steps", "3"],
                         capture_output=True, text=True, timeout=300, env=env, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["dry_run"] and line["scaling"] == "weak"
