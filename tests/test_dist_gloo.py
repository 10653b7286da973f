"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the
decode path shards by sequence with no data-path collective, so the only
cross-rank steps are the barrier and the max-over-ranks timing."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(world)
    elapsed = [120.0, 180.0][rank]
    mx = bench.max_over_ranks(elapsed, world)
    gbs = bench.aggregate_throughput(1_000_000_000, 10, mx / 1e3, world)
    q.put((rank, mx, gbs))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_timing_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, mx, gbs in res:
        assert mx == 180.0
        # 2 ranks x 10 steps x 1 GB in 0.18 s
        assert abs(gbs - 2 * 10 / 0.18) < 1e-9
