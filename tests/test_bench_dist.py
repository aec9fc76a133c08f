"""The bench's multi-rank logic on CPU: two gloo ranks, max-over-ranks timing
and whole-job throughput (each rank runs its own replica: no data exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier(world)
        mine = 0.5 + rank  # rank 1 is the slow one
        slowest = bench.reduce_max_seconds(mine, world)
        gbs = bench.aggregate_gbs(1_000_000, 10, world, slowest)
        q.put((rank, slowest, gbs))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, gbs in got:
        assert slowest == 1.5
        assert gbs == pytest.approx(2 * 1_000_000 * 10 / 1.5 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_seconds(0.25, 1) == 0.25
    assert bench.aggregate_gbs(2e9, 3, 1, 1.0) == 6.0
