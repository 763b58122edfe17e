"""The multi-GPU form of the benchmark is replicas only: each rank decodes
its own batch-1 stream, and the only cross-rank step is the timing reduction
(max over ranks) that turns per-rank times into the whole job's throughput.
These tests run that reduction on two CPU processes over gloo."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took 2 + r seconds for 100 tokens
        rate, slowest = bench.whole_job_rate(100, 2.0 + rank)
        per_sched = bench.max_over_ranks([1.0 + rank, 5.0 - 3 * rank])
        q.put((rank, rate, slowest, per_sched))
    finally:
        dist.destroy_process_group()


def test_two_replicas_aggregate_over_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, slowest, per_sched in out:
        assert slowest == 3.0                       # the max over ranks, on every rank
        assert rate == pytest.approx(200 / 3.0)     # both ranks' tokens over that time
        assert per_sched == [2.0, 5.0]              # element-wise max, same on each rank


def test_single_process_is_unchanged():
    import bench
    assert not dist.is_initialized()
    assert bench.whole_job_rate(64, 2.0) == (32.0, 2.0)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
