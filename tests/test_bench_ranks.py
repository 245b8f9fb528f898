"""Multi-process host logic of bench.py on CPU (gloo, two ranks).

Every rank runs its own replica of the step, so the only cross-rank logic is
host-side: the step time is the maximum over ranks, the reported rate is the
whole job's (world x per-rank work over that time), and the reference arm runs
on rank 0 alone while the other ranks exit without work or output.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method="env://")
    try:
        w, r, local = bench.rank_env()
        ms = 2.0 + 3.0 * r            # the higher rank is the slower one
        m = bench.rank_max(ms, w, torch.device("cpu"))
        q.put((r, w, local, m, bench.job_rate(100.0, w, m)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_step_time_is_max_over_ranks_and_rate_is_whole_job():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, m, rate in out:
        assert w == world and local == r
        assert m == 5.0                                     # the slow rank's time, on every rank
        assert rate == pytest.approx(world * 100.0 / 5e-3)  # both ranks' work over that time


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench

    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.rank_env() == (1, 0, 0)
        assert bench.rank_max(3.5, 1, None) == 3.5
        assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
    finally:
        os.environ.update(env)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
