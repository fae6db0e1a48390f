"""The bench's multi-rank logic (one replica per rank, weak scaling) on CPU with gloo.

Each rank times its own replica; the job's time is the max over ranks and the
throughput counts every rank's queries.  No data-path collective exists: the
only collectives are the timing barrier and the max.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier()
        local_seconds = 0.5 + rank          # rank r pretends its K steps took 0.5 + r seconds
        total = bench.max_over_ranks(local_seconds)
        out[rank] = total
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_barrier_with_gloo(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert dict(out) == {r: 0.5 + (world - 1) for r in range(world)}


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.dist_env()[1] >= 1
