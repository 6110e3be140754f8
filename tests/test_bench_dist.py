"""The replica path of bench.py on CPU: world size 2 over gloo.

bench.py --gpus N runs N independent replicas (the path is not partitioned
across GPUs); the timed region is bracketed by barriers, the time is the
maximum over ranks and the value counts every rank's work. These tests run
that logic with two gloo ranks on the host, and check that the reference
arm's extra ranks exit without work.
"""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        # rank r "took" 1 + r milliseconds per step; the job time is the max
        t = bench.reduce_max(torch, 1e-3 * (1 + r), w)
        rate = bench.aggregate_rate(w, 1e9, t)
        bench.barrier(w)
        q.put((r, w, local, t, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    out = sorted(q.get(timeout=5) for _ in range(world))
    for rank, (r, w, local, t, rate) in enumerate(out):
        assert (r, w, local) == (rank, world, rank)
        assert t == pytest.approx(2e-3)               # the slower rank's time on both
        assert rate == pytest.approx(2 * 1e9 / 2e-3)  # both ranks' units over that time


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(torch, 0.5, 1) == 0.5
    bench.barrier(1)
    assert bench.aggregate_rate(1, 10.0, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        config, dtype, steps, warmup = 1, "f32", 1, 1
    # rank 1 returns before touching CUDA or the library
    assert bench.run_reference(Args()) == 0
