"""Multi-rank host logic on CPU with the gloo backend (world size 2 and 3):
rows are split disjointly and completely, and the timed region's max-over-ranks
and unit sums agree with a single-process computation."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from sparse_top_kv_fathom_gb300 import shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, total, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    a, b = shard.partition(total, world, rank)
    elapsed = 1.0 + rank * 0.25  # this rank's timed region
    mx = shard.reduce_scalar(elapsed, "max")
    units = shard.reduce_scalar(b - a, "sum")
    shard.barrier()
    q.put((rank, a, b, mx, units))
    torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_partition_and_reductions_over_gloo(world):
    total = 288
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, total, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    spans = [(a, b) for _, a, b, _, _ in res]
    assert spans[0][0] == 0 and spans[-1][1] == total
    for (a0, b0), (a1, b1) in zip(spans, spans[1:]):
        assert b0 == a1
    for _, _, _, mx, units in res:
        assert mx == 1.0 + (world - 1) * 0.25
        assert units == total


def test_partition_single_process():
    assert shard.partition(10, 1, 0) == (0, 10)
    assert [shard.partition(10, 4, r) for r in range(4)] == [(0, 3), (3, 6), (6, 8), (8, 10)]
    with pytest.raises(ValueError):
        shard.partition(10, 2, 2)
    assert shard.reduce_scalar(3.5) == 3.5
