"""The replicated (N > 1) path of bench.py on CPU ranks over gloo.

The step shards by batch row with no exchange; the only cross-rank steps are
the barrier around the timed region and the reduction of the timed figures:
the slowest rank's time and the sum of the rows every rank processed.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_env() == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms, units = bench.reduce_over_ranks(dist, [3.0, 5.5, 4.0][rank], [100, 250, 7][rank],
                                            torch.device("cpu"))
        out.put((rank, ms, units))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_reduce_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    want_ms = max([3.0, 5.5, 4.0][:world])
    want_units = sum([100, 250, 7][:world])
    assert [g[0] for g in got] == list(range(world))
    for _, ms, units in got:
        assert ms == want_ms and units == want_units


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(None, 2.5, 11, torch.device("cpu")) == (2.5, 11)
