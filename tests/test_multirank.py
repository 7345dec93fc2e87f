"""The N > 1 host path of bench.py on CPU (gloo, world size 2).

Requests shard across ranks as independent replicas: there is no data-path
collective, only the host-side merge of the timed seconds (max over ranks) and
of the units processed (sum over ranks), and rank 0 alone prints the line.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _merge_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    t, units = bench.merge_ranks(1.5 + rank, [100.0 * (rank + 1), 7.0], world)
    bench.barrier(world)
    q.put((rank, t, units))
    dist.destroy_process_group()


def test_merge_ranks_gloo_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_merge_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, units in got:
        assert t == 2.5                       # the slowest rank's time
        assert units == [300.0, 14.0]         # units of every rank


def test_merge_ranks_single():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.merge_ranks(3.0, [5, 6], 1) == (3.0, [5, 6])


def test_reference_arm_under_torchrun_world2():
    """`--impl reference` launched like the driver's N = 2 run: rank 0 prints
    one JSON line, the other rank exits 0 without work."""
    pytest.importorskip("torch.distributed.run")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "tiny_chain", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle"
    assert out["e2e"]["h2d_bytes_per_step"] == 0
