"""Multi-GPU runs are independent replicas: no collective on the data path,
only the benchmark's barrier and max/sum-over-ranks timing reductions.
Checked here with two gloo ranks on the CPU."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, 1.0 + rank)          # slowest rank sets the time
        total = bench.sum_over_ranks(dist, 100.0)            # every rank's units count
        bench.barrier(dist)
        q.put((rank, ms, total))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2.0, 200.0), (1, 2.0, 200.0)]


def test_reference_arm_under_two_ranks_prints_once():
    env = dict(os.environ, WORLD_SIZE="2")
    outs = []
    for rank in (0, 1):
        env.update(RANK=str(rank), LOCAL_RANK=str(rank))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--steps", "1", "--warmup", "1", "--layers", "1"],
                           env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        outs.append(r.stdout.strip())
    assert outs[0].startswith("{") and '"impl": "reference"' in outs[0]
    assert outs[1] == ""
