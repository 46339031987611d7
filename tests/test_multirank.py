"""Host side of the multi-GPU benchmark path (replicas), as two gloo ranks on CPU:
the timing barrier, the max-over-ranks reduction and the whole-job rate."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    r, w, local = bench.dist_setup(world)
    bench.barrier(w)
    ms = bench.max_over_ranks(10.0 * (rank + 1), w, "cpu")
    q.put((r, w, ms, bench.whole_job_rate(w, 64, 5, ms)))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_aggregation(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, ms, rate) in enumerate(res):
        assert rank == r and w == world
        assert ms == 20.0  # slowest rank
        assert rate == world * 64 * 5 / 0.020
