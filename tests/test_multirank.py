"""The multi-rank path of bench.py on the CPU: world size 2 over gloo at 127.0.0.1.

The step does not shard (every request is independent; one GPU per box), so several GPUs run
replicas: each rank times its own steps, the ranks meet at barriers, the job's time is the
slowest rank's, rank 0 alone prints, and the reference arm runs on rank 0 only."""
import argparse
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(dist)
        slowest = bench.rank_max(dist, 0.040 + 0.0035 * rank, device="cpu")  # ms per step on this rank
        bench.rank_barrier(dist)
        q.put((rank, slowest, bench.job_us_per_step(slowest, world)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [r for r, _, _ in got] == [0, 1]
    for _, slowest, us in got:
        assert slowest == pytest.approx(0.0435)        # both ranks hold the slower rank's time
        assert us == pytest.approx(0.0435 * 1e3 / 2)   # the job's µs per layer-step (two replicas)


def test_single_rank_needs_no_process_group():
    import bench
    bench.rank_barrier(None)
    assert bench.rank_max(None, 1.25) == 1.25
    assert bench.job_us_per_step(0.05, 1) == pytest.approx(50.0)


def test_reference_arm_is_rank_zero_only(capsys):
    import bench
    bench.run_reference(argparse.Namespace(gpus=2, steps=1, warmup=0), rank=1)
    assert capsys.readouterr().out == ""  # other ranks exit without work or output
