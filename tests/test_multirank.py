"""The multi-rank path on CPU (gloo): the data-parallel split of one global batch
by sequence (every sequence owned by exactly one rank, ranks balanced by token
count), the benchmark's aggregation (the slowest rank's time, the sum of all
ranks' bytes), and the key-range and head splits with their one exchange each
(the oracle standing in for each rank's GPU work)."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_cache_215_gb300 import dp
from paged_kv_cache_215_gb300 import workloads as wl


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


def _check_partition(lens, world):
    parts = dp.partition(lens, world)
    assert len(parts) == world
    assert parts[0][0] == 0 and parts[-1][1] == len(lens)
    for (a0, a1), (b0, b1) in zip(parts, parts[1:]):
        assert a0 <= a1 == b0 <= b1                       # contiguous, disjoint
    lens = np.asarray(lens, dtype=np.int64)
    total, mx = int(lens.sum()), int(lens.max()) if len(lens) else 0
    for lo, hi in parts:                                  # within one sequence of the mean
        assert abs(int(lens[lo:hi].sum()) - total / world) <= mx + 1e-9
    return parts


def test_partition_covers_every_sequence_once():
    rng = np.random.default_rng(0)
    for world in (1, 2, 3, 4, 8):
        for B in (1, 2, 7, 64, 200):
            for kind in ("uniform", "loguniform", "one_long", "zeros"):
                if kind == "uniform":
                    lens = rng.integers(4096, 12289, B)
                elif kind == "loguniform":
                    lens = np.round(np.exp(rng.uniform(np.log(512), np.log(131072), B)))
                elif kind == "one_long":
                    lens = np.full(B, 100)
                    lens[B // 2] = 1 << 20
                else:
                    lens = np.zeros(B, dtype=np.int64)
                _check_partition(lens.astype(np.int64), world)
    # a world larger than the batch leaves some ranks empty, never a sequence twice
    parts = _check_partition([5, 6], 4)
    assert sum(hi - lo for lo, hi in parts) == 2


def test_weak_scaling_global_batch_is_world_times_the_workload():
    for name in ("llama8b_b32_8k", "long_128k", "fp8_b8_32k", "llama70b_prefix_bs16"):
        one = wl.FULL[name]()
        for world in (2, 4):
            glob = wl.FULL[name](world)
            assert glob.batch == world * one.batch
            got = sorted(int(n) for r in range(world)
                         for n in dp.rank_case(name, r, world).seq_lens)
            assert got == sorted(int(n) for n in glob.seq_lens)
    assert dp.rank_case("long_128k", 0, 1).name == wl.FULL["long_128k"]().name


def _shard_worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = dp.rank_case("llama8b_b32_8k", rank, world)
    lo, hi = dp.partition(wl.FULL["llama8b_b32_8k"](world).seq_lens, world)[rank]
    mine = (lo, hi, [int(n) for n in case.seq_lens], int(case.num_blocks))
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    results[rank] = gathered
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_own_disjoint_shards_of_one_global_batch():
    """Each gloo rank builds its own share of the 8K x 32 workload's two-GPU global
    batch (64 sequences); gathered, the shares are disjoint, contiguous, cover the
    global batch once with its lengths, and each rank's pool holds its own blocks."""
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    glob = wl.FULL["llama8b_b32_8k"](2)
    for r in range(2):
        g = results[r]
        assert g[0][0] == 0 and g[0][1] == g[1][0] and g[1][1] == glob.batch
        lens = g[0][2] + g[1][2]
        assert lens == [int(n) for n in glob.seq_lens]
        for lo, hi, ls, nb in g:
            need = sum((n + 15) // 16 for n in ls)
            assert nb >= need                              # its own pool covers its blocks


def test_key_ranges_cover_a_sequence_once_on_block_boundaries():
    for n in (0, 1, 15, 16, 17, 1000, 131072):
        for world in (1, 2, 3, 8):
            rs = dp.key_ranges(n, world, 16)
            assert rs[0][0] == 0 and rs[-1][1] == n and len(rs) == world
            for (a0, a1), (b0, b1) in zip(rs, rs[1:]):
                assert a1 == b0 and a0 <= a1 and b0 <= b1
            assert all(lo % 16 == 0 for lo, _ in rs)
    with pytest.raises(ValueError):
        dp.key_ranges(10, 0, 16)


def _seqpar_worker(rank, world, port, results):
    """Rank r attends over its key range of every sequence (the oracle stands in
    for the GPU kernel here), then the gather-and-merge exchange over gloo."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    import oracle
    from tests.helpers import np_raw, oracle_pool
    case = wl.make_case("seqpar", [300, 77, 5], 8, 2, 32, 16, "f32", "f32", "f32", seed=61)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    ranges = [dp.key_ranges(int(n), world, 16)[rank] for n in case.seq_lens]
    lo = np.array([r[0] for r in ranges], np.int32)
    hi = np.array([r[1] for r in ranges], np.int32)
    o, lse, _ = oracle.decode(np_raw(tens.q), "f32", pool, "f32", case.geometry, 0, case.tables,
                              case.seq_lens, case.scale, tok_begin=lo, tok_end=hi)

    def merge(out, part_o, part_lse):
        B, H, S, D = part_o.shape
        m, _ = oracle.merge(part_o.numpy().reshape(B * H, S, D), part_lse.numpy().reshape(B * H, S))
        out.copy_(torch.from_numpy(m.reshape(B, H, D)))
        return out
    out = torch.empty(case.batch, 8, 32, dtype=torch.float64)
    dp.gather_and_merge(torch.from_numpy(o), torch.from_numpy(lse), merge, out)
    full, _, _ = oracle.decode(np_raw(tens.q), "f32", pool, "f32", case.geometry, 0, case.tables,
                               case.seq_lens, case.scale)
    results[rank] = float(np.abs(out.numpy() - full).max())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_key_range_split_gathers_and_merges_to_the_whole_attention(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_seqpar_worker, args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    for r in range(world):
        assert results[r] < 1e-12


def test_head_ranges_split_kv_heads_evenly():
    assert dp.head_ranges(8, 1) == [(0, 8)]
    assert dp.head_ranges(8, 4) == [(0, 2), (2, 4), (4, 6), (6, 8)]
    with pytest.raises(ValueError):
        dp.head_ranges(8, 3)


def _heads_worker(rank, world, port, results):
    """Rank r attends with the query heads of its KV heads only (the oracle's rows
    of those heads stand in for the GPU kernel on a pool of those heads), then the
    all-gather that concatenates the heads."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    import oracle
    from tests.helpers import np_raw, oracle_pool
    case = wl.make_case("heads", [300, 77, 5], 8, 4, 32, 16, "f32", "f32", "f32", seed=62)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    G = case.num_q_heads // case.num_kv_heads
    lo, hi = dp.head_ranges(case.num_kv_heads, world)[rank]
    rows = np.array([s * case.num_q_heads + h for s in range(case.batch)
                     for h in range(lo * G, hi * G)], np.int32)
    o, _, _ = oracle.decode(np_raw(tens.q), "f32", pool, "f32", case.geometry, 0, case.tables,
                            case.seq_lens, case.scale, rows=rows)
    mine = torch.from_numpy(np.ascontiguousarray(o[:, lo * G:hi * G]))
    out = torch.empty(case.batch, case.num_q_heads, 32, dtype=torch.float64)
    dp.gather_heads(mine, out)
    full, _, _ = oracle.decode(np_raw(tens.q), "f32", pool, "f32", case.geometry, 0, case.tables,
                               case.seq_lens, case.scale)
    results[rank] = float(np.abs(out.numpy() - full).max())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_head_split_gathers_to_the_whole_attention(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_heads_worker, args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    for r in range(world):
        assert results[r] == 0.0
