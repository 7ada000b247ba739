"""bench.py on several GPUs runs one full replica of the workload per rank (the units
shard with no exchange step, so there is no collective on the data path): a step's
time is the slowest rank's and the throughput counts every rank's rows.  Checked here
with two gloo ranks on the CPU (127.0.0.1 rendezvous)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        own = [0.180, 0.210][rank]          # rank 1 is the slow one
        ms = bench.slowest(own, world, "cpu")
        q.put((rank, ms, bench.job_rows_per_s(world, 1, 8, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [0.210, 0.210]
    assert all(g[2] == pytest.approx(2 * 8 / 0.210e-3) for g in got)


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.slowest(0.25, 1) == 0.25
    assert bench.job_rows_per_s(1, 32, 15, 0.5) == pytest.approx(32 * 15 / 0.5e-3)
