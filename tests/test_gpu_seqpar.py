"""Key-range and head splits of decode across GPUs, emulated on one GPU (needs a GPU).

"Sequence-parallel engineering for long-context LLM inference" splits a long
sequence's keys across devices; each attends over its own range and the
partial results are combined by the log-sum-exp correction.  Here rank r of N
holds the block-aligned range dp.key_ranges(n, N, bs)[r] of every sequence in a
pool of its own (local positions 0 .. hi - lo); paged_decode_attention_partial
gives its fp32 partial output and natural log-sum-exp per row; the partials of
the N ranks, stacked, go through merge_partials.  The ranks run one after the
other on the one GPU (no kernel waits for another).  Checked against the fp64
oracle: each rank's partial output and log-sum-exp against the oracle over the
same key range, and the merged output against the whole attention, within
2e-3 x max|V| (bf16) or 5e-3 x max|V| (E4M3).  The head split gives each rank
the blocks of a range of KV heads (dp.head_ranges) and concatenates the ranks'
outputs along the heads.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_215_gb300 import dp
from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import TOL, oracle_side, vmax_per_seq
from tests.helpers import fp8_scales, np_raw

pytestmark = pytest.mark.gpu


def _full_kv(case, tens):
    """Every sequence's K and V rows in position order (the new token last)."""
    ks, vs = [], []
    seq, pos = tens.tok_seq.numpy(), tens.tok_pos.numpy()
    for s in range(case.batch):
        n = int(case.seq_lens[s])
        k = torch.zeros(n, case.num_kv_heads, case.head_dim, dtype=tens.k_tokens.dtype)
        v = torch.zeros_like(k)
        m = seq == s
        k[pos[m]] = tens.k_tokens[torch.from_numpy(m)]
        v[pos[m]] = tens.v_tokens[torch.from_numpy(m)]
        if n:
            k[n - 1] = tens.k_new[s]
            v[n - 1] = tens.v_new[s]
        ks.append(k)
        vs.append(v)
    return ks, vs


def _rank_partial(case, ks, vs, ranges, q, k_scale, v_scale):
    """One rank: a pool holding range (lo, hi) of each sequence at local positions."""
    from paged_kv_cache_215_gb300 import pkv
    bs = case.block_size
    lens = [hi - lo for lo, hi in ranges]
    nbs = [(n + bs - 1) // bs for n in lens]
    nb = max(sum(nbs), 1) + 3
    geom = pkv.geometry(1, case.num_q_heads, case.num_kv_heads, case.head_dim, bs, nb,
                        case.kv_dtype)
    pool = pkv.KVPool(geom)
    pool.storage.fill_(0xFF)                     # unwritten slots: NaN patterns
    mb = max(max(nbs), 1)
    tables = np.full((case.batch, mb), -1, np.int32)
    pool.prepare_append(np.zeros(case.batch, np.int32), tables, new_tokens=lens)
    k = torch.cat([ks[s][lo:hi] for s, (lo, hi) in enumerate(ranges)])
    v = torch.cat([vs[s][lo:hi] for s, (lo, hi) in enumerate(ranges)])
    seq = torch.cat([torch.full((hi - lo,), s, dtype=torch.int32)
                     for s, (lo, hi) in enumerate(ranges)])
    pos = torch.cat([torch.arange(hi - lo, dtype=torch.int32) for lo, hi in ranges])
    td = torch.from_numpy(tables).cuda()
    if k.shape[0]:
        pool.append_tokens(0, k.cuda(), v.cuda(), td, seq.cuda(), pos.cuda(), k_scale, v_scale)
    out = torch.full((case.batch, case.num_q_heads, case.head_dim), float("nan"), device="cuda")
    lse = torch.full((case.batch, case.num_q_heads), float("nan"), device="cuda")
    pkv.paged_decode_attention_partial(out, lse, q.cuda(), pool, 0, td,
                                       torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                       max(max(lens), 0), case.scale, k_scale, v_scale)
    torch.cuda.synchronize()
    assert pool.check_status() == 0
    return out, lse


@pytest.mark.parametrize("world", [2, 3, 5])
@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_key_range_split_partials_merge_to_the_whole_attention(kv, world):
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    # a long sequence, a short one (empty ranges on some ranks) and one of 1 token
    case = wl.make_case(f"seqpar_{kv}", [6000, 40, 1], 32, 8, 128, 16, kv, "bf16", "bf16",
                        seed=70, spike_frac=0.01)
    tens = wl.make_tensors(case)
    ks_, vs_ = (1.0, 1.0) if kv != "e4m3" else fp8_scales(tens)
    pool, ref, seqs = oracle_side(case, tens, None, ks_, vs_)
    vm = vmax_per_seq(case, pool, seqs, vs_)
    kall, vall = _full_kv(case, tens)
    tol = TOL[kv]
    outs, lses = [], []
    for r in range(world):
        ranges = [dp.key_ranges(int(n), world, 16)[r] for n in case.seq_lens]
        o, l = _rank_partial(case, kall, vall, ranges, tens.q, ks_, vs_)
        lo = np.array([a for a, _ in ranges], np.int32)
        hi = np.array([b for _, b in ranges], np.int32)
        ro, rl, _ = oracle.decode(np_raw(tens.q), "bf16", pool, kv, case.geometry, 0,
                                  case.tables, case.seq_lens, case.scale, ks_, vs_,
                                  tok_begin=lo, tok_end=hi)
        go, gl = o.double().cpu().numpy(), l.double().cpu().numpy()
        for s in seqs:
            if hi[s] == lo[s]:
                assert np.all(go[s] == 0) and np.all(np.isneginf(gl[s])), (r, s)
                continue
            assert np.abs(go[s] - ro[s]).max() <= tol * vm[s], (r, s)
            assert np.abs(gl[s] - rl[s]).max() <= 1e-3 + 1e-5 * np.abs(rl[s]).max(), (r, s)
        outs.append(o)
        lses.append(l)
    part_o = torch.stack(outs, dim=2).contiguous()
    part_lse = torch.stack(lses, dim=2).contiguous()
    out = torch.full((case.batch, 32, 128), float("nan"), device="cuda")
    pkv.merge_partials(out, part_o, part_lse)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    for s in seqs:
        assert np.abs(got[s] - ref[s]).max() <= tol * vm[s], s


@pytest.mark.parametrize("world", [2, 4, 8])
@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_head_split_outputs_concatenate_to_the_whole_attention(kv, world):
    """Rank r of N holds every sequence's blocks for KV heads dp.head_ranges(8, N)[r]
    only, in a pool of its own, and attends with their query heads; the ranks'
    outputs, concatenated along the heads, must match the oracle's whole
    attention (E4M3: the per-tensor scales of the whole tensors, as one pool would
    use)."""
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    case = wl.make_case(f"heads_{kv}", [3000, 40, 1], 32, 8, 128, 16, kv, "bf16", "bf16",
                        seed=71, spike_frac=0.01)
    tens = wl.make_tensors(case)
    ks_, vs_ = (1.0, 1.0) if kv != "e4m3" else fp8_scales(tens)
    pool_o, ref, seqs = oracle_side(case, tens, None, ks_, vs_)
    vm = vmax_per_seq(case, pool_o, seqs, vs_)
    kall, vall = _full_kv(case, tens)
    G, bs = 4, 16
    lens = [int(n) for n in case.seq_lens]
    outs = []
    for lo, hi in dp.head_ranges(8, world):
        nbs = [(n + bs - 1) // bs for n in lens]
        geom = pkv.geometry(1, (hi - lo) * G, hi - lo, 128, bs, sum(nbs) + 3, kv)
        pool = pkv.KVPool(geom)
        pool.storage.fill_(0xFF)
        tables = np.full((case.batch, max(nbs)), -1, np.int32)
        pool.prepare_append(np.zeros(case.batch, np.int32), tables, new_tokens=lens)
        k = torch.cat([kall[s][:, lo:hi] for s in range(case.batch)]).contiguous()
        v = torch.cat([vall[s][:, lo:hi] for s in range(case.batch)]).contiguous()
        seq = torch.cat([torch.full((n,), s, dtype=torch.int32) for s, n in enumerate(lens)])
        pos = torch.cat([torch.arange(n, dtype=torch.int32) for n in lens])
        td = torch.from_numpy(tables).cuda()
        pool.append_tokens(0, k.cuda(), v.cuda(), td, seq.cuda(), pos.cuda(), ks_, vs_)
        q = tens.q[:, lo * G:hi * G].contiguous().cuda()
        out = torch.full((case.batch, (hi - lo) * G, 128), float("nan"), device="cuda")
        pkv.paged_decode_attention(out, q, pool, 0, td,
                                   torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                   max(lens), case.scale, ks_, vs_)
        torch.cuda.synchronize()
        assert pool.check_status() == 0
        outs.append(out)
    got = torch.cat(outs, dim=1).double().cpu().numpy()
    for s in seqs:
        assert np.abs(got[s] - ref[s]).max() <= TOL[kv] * vm[s], s
