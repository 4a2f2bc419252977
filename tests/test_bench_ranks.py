"""Host logic of a multi-GPU benchmark run (replicas), on CPU: two gloo ranks agree on the
slowest rank's timings, and the whole-job rate counts every rank's tokens."""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank 0 is slower on the device, rank 1 on the host path
    got = bench.max_over_ranks([100.0 + 50.0 * (rank == 0), 2.0 + 3.0 * (rank == 1)], world)
    q.put((rank, got, bench.whole_job_rate(1024, got[0] * 1e-3, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_count_all_tokens():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [150.0, 5.0]
        assert rate == pytest.approx(2 * 1024 / 0.150)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_rate(512, 0.5, 1) == 1024.0
