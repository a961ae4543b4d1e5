"""The multi-rank host logic on CPU (gloo, two processes): every rank agrees
on the slowest rank's time, the whole-job value counts every rank's copy of the
workload, and under torchrun the reference arm prints one line from rank 0
while the other rank exits without work."""
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


def _rank_main(rank, world, port, local_ms, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out.put((rank, bench.max_over_ranks(local_ms[rank], world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local = [1.5, 4.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 4.0, 1: 4.0}


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_value(1e12, 1, 2.0)
    assert one == pytest.approx(500.0)
    assert bench.whole_job_value(1e12, 4, 2.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
