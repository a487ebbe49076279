"""The N > 1 bench path on the CPU: two gloo ranks, each an independent
replica (the decode path has no exchange step). The job's step time is the
slowest rank's, and its throughput counts every rank's bytes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.aggregate_over_ranks(1.0 + rank, 1_000_000)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in results:
        assert ms == pytest.approx(2.0)                     # slowest rank: 2 ms
        assert value == pytest.approx(2 * 1e6 / 2e-3 / 1e9)  # both ranks' bytes


def test_single_process_is_the_one_gpu_case():
    import bench
    ms, value = bench.aggregate_over_ranks(4.0, 8_000_000)
    assert ms == 4.0 and value == pytest.approx(8e6 / 4e-3 / 1e9)
