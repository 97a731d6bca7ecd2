"""bench.py's multi-process logic on the CPU (gloo, world size 2; no GPU).

`bench.py --gpus N` runs N independent replicas (the path does not shard), one process per GPU
under torchrun: the ranks meet at barriers around the timed region, the step time reported is
the maximum over the ranks, and rank 0 alone prints the JSON line. The reference arm (the oracle
on the host cores) runs on rank 0 only, over gloo, and the other ranks exit 0 without work.
"""

from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks_child(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    ws, r, local = bench.dist_env()
    torch.distributed.init_process_group("gloo", rank=r, world_size=ws)
    try:
        bench.barrier(ws)
        slowest = bench.allreduce_max(ws, 1.5 + 2.0 * r, "cpu")  # rank r "measured" 1.5 + 2r ms
        bench.barrier(ws)
        out.put((r, ws, local, slowest))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ranks_child, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 2, 0, 3.5), (1, 2, 1, 3.5)]  # every rank reports the slowest rank's time


def test_reference_arm_under_torchrun_prints_one_line():
    """The driver's launch line for N > 1, on the reference arm: one JSON line (rank 0), exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "1", "--ref-rows", "8"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["higher_is_better"] is True
    assert rec["value"] > 0 and rec["unit"] == "TB/s" and rec["dtype"] == "f64"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"] == {"value": rec["value"], "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert rec["config"]["workload"]


def test_single_process_environment():
    sys.path.insert(0, ROOT)
    import bench

    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_env() == (1, 0, 0)
        assert bench.allreduce_max(1, 2.5, "cpu") == 2.5  # one process: no collective
        bench.barrier(1)
    finally:
        os.environ.update(env)
