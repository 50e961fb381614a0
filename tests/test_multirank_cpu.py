"""The multi-rank benchmark logic on CPU with gloo, world size 2: barrier, max-over-ranks
timing and the weak-scaling aggregate (each rank scans its own copy; no data collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    bench.barrier(ws)
    t = bench.max_over_ranks(1.0 + rank, ws)       # rank 1 is the slow one
    v = bench.weak_scaling_value(100.0, ws, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_ranks_max_timing_and_weak_value():
    if not dist.is_gloo_available():
        pytest.skip("gloo not available")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, v in res:
        assert t == 2.0                      # max over ranks
        assert v == 2 * 100.0 / 2.0          # all ranks' units over the slowest rank


def test_gpus_flag_spawns_ranks_without_a_launcher():
    """`bench.py --gpus 2` run directly (no torchrun, WORLD_SIZE unset) starts two ranks
    itself; only rank 0 prints its line (the reference arm runs on the host cores, so this
    runs without a GPU)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, cwd=root, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
    assert lines[0]["n_gpus"] == 2
