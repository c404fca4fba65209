"""Replica (N > 1) host logic of bench.py on CPU: two gloo ranks.

The mixer block's work is independent per decode row and per prefill
sequence, so N GPUs run N full replicas with no exchange on the data path;
the only cross-rank steps are the barrier around the timed region and the
max-over-ranks step time.  These tests run that logic with world_size 2 on the
gloo backend, and the reference arm's rank-0-only rule."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = [0.75, 1.25][rank]                 # the second replica is slower
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.job_throughput(bench.TOKENS_PER_STEP, ms, world)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_replicas_take_the_slowest_step_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    sys.path.insert(0, ROOT)
    import bench
    for rank, ms, value in got:
        assert ms == 1.25                                 # max over ranks, on every rank
        assert value == pytest.approx(2 * bench.TOKENS_PER_STEP / 1.25e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5) == 0.5
    assert bench.job_throughput(1000, 2.0, 1) == pytest.approx(5e5)


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the oracle arm runs on rank 0 alone; other ranks exit 0
    without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
