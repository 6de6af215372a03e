"""The multi-replica path of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs an independent replica, so the only cross-rank step is the
aggregation after the timed region: work is summed over ranks and each time
is the maximum over ranks (the slowest replica bounds the job).
"""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, _ = bench.dist_info()
    assert (ws, r) == (world, rank)
    res = bench.aggregate_over_ranks({"decode_bytes": 100.0 * (rank + 1), "extend_flops": 7.0},
                                     {"total_ms": 1.0 + rank, "decode_ms": 0.5 * (2 - rank)}, ws)
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            res = out[r]
            assert res["decode_bytes"] == 300.0 and res["extend_flops"] == 14.0
            assert res["total_ms"] == 2.0 and res["decode_ms"] == 1.0


def test_single_rank_is_identity():
    import bench
    res = bench.aggregate_over_ranks({"decode_bytes": 5}, {"total_ms": 3.0}, 1)
    assert res == {"decode_bytes": 5, "total_ms": 3.0}
