"""The N>1 path of bench.py on CPU with gloo (world size 2): ranks are
independent replicas (requests are independent, Flide Prop. 3.1); the only
collectives are the timing barrier and the max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    total_ms = [120.0, 150.0][rank]              # each replica's own timed region
    bench.barrier(ws)
    mx = bench.reduce_max(torch, total_ms, ws)
    env = bench.dist_env()
    q.put((rank, mx, env))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, mx, env in out:
        assert mx == 150.0                        # every rank sees the slowest rank's time
        assert env == (2, rank, rank)
    import bench
    # whole-job throughput: all ranks' units over the slowest rank's time
    assert bench.aggregate([0.12, 0.15], [100, 100]) == pytest.approx(200 / 0.15)


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference launched with two ranks: rank 0 alone times
    the oracle and prints one JSON line; the other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
