"""Multi-process logic of bench.py on the CPU (gloo, world size 2): the timed
region's max over ranks, the whole-job value, and the reference arm running on
rank 0 only. The GPU path runs one replica per GPU with no data-path
collective; these are the only cross-rank steps."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.max_over_ranks(1.0 + 2.5 * rank, torch.device("cpu"))
        args = type("A", (), {"workload": "tiny", "steps": 1, "warmup": 3})()
        ref = bench.run_reference(args, rank, world) if rank != 0 else "rank0"
        out.put((rank, ms, ref))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_reference_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_worker, args=(world, port, q), nprocs=world, join=True, start_method="spawn")
    got = sorted(q.get(timeout=60) for _ in range(world))
    assert [g[1] for g in got] == [3.5, 3.5]          # both ranks see the slowest rank's time
    assert got[1][2] is None                           # the reference arm does no work off rank 0


def test_job_value_is_the_sum_over_replicas():
    import bench

    assert bench.job_value(2_000_000_000, 1, 1.0) == pytest.approx(2.0)
    assert bench.job_value(2_000_000_000, 4, 0.5) == pytest.approx(16.0)
