"""The replica bookkeeping of bench.py on CPU: two gloo ranks, the slowest
rank's time sets the whole-job figure, and the reference arm prints only on
rank 0."""

import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks([1.0 + rank, 10.0 * (2 - rank), 3.0], dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world_2():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 20.0, 3.0]


def test_job_tflops_counts_every_replica():
    import bench
    assert bench.job_tflops(1, 2e12, 1.0) == pytest.approx(2000.0)
    assert bench.job_tflops(4, 2e12, 2.0) == pytest.approx(4000.0)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_reference_arm_prints_only_on_rank_0(repo_root):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(repo_root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--gpus", "2"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
