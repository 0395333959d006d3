"""The benchmark's replica aggregation across ranks (torch.distributed, gloo, 2 ranks on the
CPU): the timed region is the max over ranks and the value counts every rank's tokens."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [100.0, 250.0][rank]
    t, value = bench.aggregate_over_ranks(local_ms, 15 * 10, dist, "cpu")
    out[rank] = (t, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        t, value = out[r]
        assert t == 250.0                       # slowest rank
        assert abs(value - 2 * 150 / 0.25) < 1e-9  # both ranks' tokens over the max time


def test_single_rank_aggregation():
    t, value = __import__("bench").aggregate_over_ranks(50.0, 30, None)
    assert t == 50.0 and abs(value - 600.0) < 1e-9
