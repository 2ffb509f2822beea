"""The N-GPU benchmark runs independent replicas: no data-path collective, only the
timing aggregation (barrier, slowest rank's time, total work).  That host logic is
exercised here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), world)      # per-rank elapsed ms
    tokens = bench.sum_over_ranks(1000.0 * (rank + 1), world)     # per-rank tokens
    q.put((rank, slowest, tokens))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_benchmark():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, tokens in got:
        assert slowest == 20.0 and tokens == 3000.0
    # weak scaling: value = total work / slowest time
    assert got[0][2] / (got[0][1] / 1e3) == 3000.0 / 0.02
