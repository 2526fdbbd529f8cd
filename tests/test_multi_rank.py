"""The multi-replica aggregation of bench.py on two CPU ranks (gloo): the whole-job time is
the slowest rank's and the verified tokens are summed over ranks. The verify path itself
runs one replica per GPU with no collective (sequences are independent)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = bench.aggregate(10.0 * (rank + 1), 20.0 + rank, 7 * (rank + 1), 3 + rank, torch.device("cpu"))
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r] == (20.0, 21.0, 21, 7)


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(1.5, 2.5, 3, 4, torch.device("cpu")) == (1.5, 2.5, 3, 4)
