"""The N > 1 bench path on CPU: two gloo ranks (no GPU). Each rank runs its own
replica of the workload (weak scaling, no data-path collective); only the timings
are reduced, by a max over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports step times (1 + r, 10 - r): the max over ranks is (world, 10)
        out[rank] = bench.reduce_max([1.0 + rank, 10.0 - rank], world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        assert out[r] == [float(world), 10.0]


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max([3.5, 1.25], 1) == [3.5, 1.25]
