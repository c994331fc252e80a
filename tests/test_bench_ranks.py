"""The multi-rank aggregation of bench.py on CPU: two gloo ranks, each with its
own replica's timings and KV-token count. Times take the max over ranks and
work units are summed; one rank gets its inputs back unchanged."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    times = [10.0 + rank, 5.0 - rank, 20.0 * (rank + 1)]
    out = bench.aggregate_over_ranks(times, 1000 * (rank + 1))
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        times, units = res[r]
        assert times == [11.0, 5.0, 40.0]
        assert units == 3000.0


def test_single_rank_is_identity():
    import bench

    assert bench.aggregate_over_ranks([1.0, 2.0], 7) == ([1.0, 2.0], 7.0)
