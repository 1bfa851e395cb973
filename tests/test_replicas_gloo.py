"""The multi-GPU form of the benchmark is independent replicas (the layer has
no exchange step in decode).  Its host-side aggregation -- every rank's tokens
over the slowest rank's time -- is checked here with two gloo ranks on CPU."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 * (rank + 1)          # rank 1 is the slow one
    value, max_ms, tokens = bench.aggregate_replicas(local_ms, 50 * (rank + 1))
    q.put((rank, value, max_ms, tokens))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_slowest_rank():
    world, port = 2, 29531
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, max_ms, tokens in res:
        assert max_ms == 200.0
        assert tokens == 150
        assert value == pytest.approx(150 / 0.2)


def test_single_process_is_a_noop():
    import bench
    assert bench.aggregate_replicas(250.0, 10) == (40.0, 250.0, 10)
