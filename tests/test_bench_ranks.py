"""The multi-rank path of bench.py on the CPU (gloo, world size 2).

Under torchrun each rank runs an independent replica of the step (the path
shards by independent problems, so there is no collective on the data path);
the job's time is the slowest rank's, and its value counts the bytes of every
rank.  The reference arm runs on rank 0 only; other ranks exit at once.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [10.0, 12.5][rank]  # this rank's timed region
    slowest = bench.max_over_ranks(ms, "cpu", world)
    value = bench.whole_job_gbs(1_000_000_000, 4, slowest, world)
    q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_bytes():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, slowest, value in res:
        assert slowest == 12.5
        # 2 ranks x 4 steps x 1 GB in 12.5 ms
        assert value == pytest.approx(2 * 4 * 1.0 / 12.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, "cpu", 1) == 3.0
    assert bench.whole_job_gbs(2_000_000_000, 5, 10.0, 1) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
