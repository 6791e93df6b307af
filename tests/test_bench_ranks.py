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


def test_roofline_entries():
    """The bench line's roofline object: HBM for streams and decode calls, the
    FMA pipe for verify with R >= 2 (R + 1 lane-ops per weight)."""
    import argparse

    sys.path.insert(0, ROOT)
    import bench

    a = argparse.Namespace(config="cfg2", rows=6, steps=10)
    r = bench.roofline(a, "stream_plan_q8_0", 1, 5000.0, 6778.0, "measured", 123, "x", 1.0)
    assert r["bound"] == "hbm" and r["frac"] == round(5000.0 / 6778.0, 4)
    a = argparse.Namespace(config="cfg5", rows=6, steps=10)
    r = bench.roofline(a, "verify", 14, 500.0, 6778.0, "measured", None, None, 100.0)
    weights = bench.CFG5_COPIES * (17408 * 5120 + 5120 * 17408)
    assert r["bound"] == "alu" and r["ops_per_weight"] == 7
    assert r["achieved"] == pytest.approx(weights * 7 * 10 / 0.1 / 1e9, abs=0.05)
    assert r["hbm"]["bound"] == "hbm"
    assert bench.step_bytes_static(argparse.Namespace(config="cfg2", layers=0, qkv="separate")) \
        == 604_714_496


@pytest.mark.parametrize("config,rows,want", [
    # one Q8_0 GEMV 3072x1024: 3,342,336 packed + 4 (M + K) = 3,358,720 B, 96 rotated copies
    ("cfg1", 6, 96 * 3_358_720),
    # Qwen3-0.6B-shaped Q8_0 token, gate and up fused (169 ops)
    ("cfg2", 6, 604_714_496),
    # 7B-shaped Q4_0 token, gate and up fused: 3,977,035,776 weight + activation bytes
    ("cfg3", 6, 3_985_629_184),
    # the same 7B-shaped token in Q4_K super-blocks (144 B per 256 weights = 18 per 32)
    ("cfg3k", 6, 3_985_629_184),
    # RMSNorm + gate/up + SiLU 3072x1024: 6,705,152 B per call, 28 rotated pairs
    ("cfg4", 6, 28 * 6_705_152),
    # Q4_0 verify 17408x5120 and its transpose: 50,135,040 packed + R * 4 (M + K) B per matrix, 7 copies
    ("cfg5", 1, 7 * 2 * (50_135_040 + 1 * 90_112)),
    ("cfg5", 6, 7 * 2 * (50_135_040 + 6 * 90_112)),
    # fp16 LM head 151936x1024: 2 B per weight + 4 (M + K)
    ("f16", 6, 2 * 151936 * 1024 + 4 * (151936 + 1024)),
])
def test_step_bytes_of_every_configuration(config, rows, want):
    """The algorithmic bytes behind every GB/s figure and roofline fraction,
    against per-unit figures derived from the shapes and block sizes."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench

    a = argparse.Namespace(config=config, layers=0, qkv="separate", rows=rows)
    assert bench.step_bytes_static(a) == want


def test_hold_load_replays_in_synced_batches_for_the_given_time():
    import time
    sys.path.insert(0, ROOT)
    import bench

    calls = []
    t0 = time.perf_counter()
    n = bench.hold_load(lambda: calls.append("r"), lambda: calls.append("s"), 0.05, batch=4)
    assert time.perf_counter() - t0 >= 0.05
    assert n == calls.count("r") and n % 4 == 0 and n >= 4
    assert calls.count("s") == n // 4
    assert calls[:5] == ["r"] * 4 + ["s"] and calls[-1] == "s"
