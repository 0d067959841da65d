"""Host logic of the benchmark's multi-rank (weak scaling) path, on CPU with
two gloo ranks: the job time is the slowest rank's and the job's work is the
sum over ranks; the reference arm prints from rank 0 only."""

import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [2.0, 5.0][rank]
    units_local = 1.0e12
    ms, rate = bench.job_throughput(ms_local, units_local)
    out[rank] = (ms, rate)
    dist.destroy_process_group()


def test_job_throughput_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, rate = out[r]
        assert ms == 5.0                                  # slowest rank
        assert abs(rate - 2.0e12 / 5e-3) < 1e3            # both ranks' work over that time


def test_job_throughput_single_process():
    sys.path.insert(0, ROOT)
    import bench
    ms, rate = bench.job_throughput(4.0, 8.0e9)
    assert ms == 4.0 and rate == pytest.approx(2.0e12)


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    port = 29600 + os.getpid() % 1000
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1 and '"impl": "reference"' in lines[0]
