"""CPU, two processes (gloo): the benchmark's replica logic.  The path has no exchange step
("replicas only"), so what needs checking across processes is the host side: the timed
region is the slowest rank's, the job's value counts every rank's units over that time, and
the reference arm prints one line from rank 0 while the other ranks leave without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        w = bench.WORKLOADS["mxfp4_mlp_12288x4096"]
        units = 321.4e6  # algorithmic bytes one rank streams per step
        value = bench.job_rate(w, units, world, slowest * 1e-3)
        q.put((rank, slowest, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world, port = 2, _free_port()
    times = [0.104, 0.131]  # ms per step on each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in out:
        assert slowest == pytest.approx(max(times))
        # GB/s of the whole job: both ranks' bytes over the slowest rank's step
        assert value == pytest.approx(2 * 321.4e6 / (max(times) * 1e-3) / 1e9)


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "nvfp4_gemm_2048x1024", "--steps", "1",
           "--warmup", "3", "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
