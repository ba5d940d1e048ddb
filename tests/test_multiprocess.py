"""The bench's multi-process path on CPU (gloo, two ranks): the timed region's reduction takes
the slowest rank, the whole-job rate counts every rank's replica, and the reference arm prints
one line from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [3.0, 7.5][rank]  # the second rank is slower
    got = bench.max_over_ranks(local_ms, world)
    rate = bench.whole_job_rate(1000.0, world, got / 1e3)
    out[rank] = (got, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_with_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        got, rate = res[rank]
        assert got == 7.5  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 / 7.5e-3)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_prints_once_under_torchrun(tmp_path):
    """`bench.py --impl reference` launched as two ranks: rank 0 prints one JSON line, rank 1
    exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
