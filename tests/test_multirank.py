"""The benchmark's multi-rank path on CPU: two gloo ranks, each with its own
(independent) batch, report the slowest rank's time and the sum of bytes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.0][rank]                   # rank 1 is the slower one
    kv = [1_000_000, 3_000_000][rank]       # bytes per step of each rank's batch
    results[rank] = bench.aggregate_ranks(ms, kv)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_sums_bytes():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        ms, gbs = results[r]
        assert ms == 3.0
        assert gbs == pytest.approx(4_000_000 / 3e-3 / 1e9)


def test_single_rank_aggregation_is_identity():
    import bench
    ms, gbs = bench.aggregate_ranks(2.0, 4_000_000)
    assert ms == 2.0 and gbs == pytest.approx(4_000_000 / 2e-3 / 1e9)
