"""The multi-process path of bench.py on CPU: two gloo ranks, each timing a
different amount, agree on the slowest rank's time; ranks never exchange
attention data (the work partitions by sequence)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(values[rank])
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


@pytest.mark.parametrize("values", [(3.5, 7.25), (9.0, 1.0)])
def test_max_over_ranks_with_two_gloo_ranks(values):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=10) for _ in range(2))
    assert results[0] == results[1] == max(values)


def test_max_over_ranks_without_a_process_group():
    import bench
    assert bench.max_over_ranks(4.5) == 4.5
