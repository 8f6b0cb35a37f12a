"""The seeded input recipe (no GPU): the full-size workloads have the shapes,
length mixes, block-id layout and value structure the measurements are quoted
on, and every draw is reproducible from its seed."""
import numpy as np
import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl


def _blocks(case, s):
    n = int(case.seq_lens[s])
    return case.tables[s, :(n + case.block_size - 1) // case.block_size]


def test_8b_batch_lengths_and_private_block_ids():
    c = wl.FULL["llama8b_b32_8k"]()
    assert (c.batch, c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size) == (32, 32, 8, 128, 16)
    assert c.seq_lens.min() >= 4096 and c.seq_lens.max() <= 12288
    ids = np.concatenate([_blocks(c, s) for s in range(c.batch)])
    assert ids.min() >= 0 and ids.max() < c.num_blocks
    assert len(np.unique(ids)) == len(ids)                       # no block used twice
    need = sum((int(n) + 15) // 16 for n in c.seq_lens)
    assert c.num_blocks == int(np.ceil(need * 1.1))              # +10% pool slack
    assert not np.array_equal(np.sort(ids), ids)                 # a permutation, not in order


def test_long_context_spikes_one_percent_of_k_rows():
    c = wl.make_case("spikes", [3000], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=1002,
                     spike_frac=0.01)
    t = wl.make_tensors(c)
    plain = wl.make_tensors(wl.make_case("nospikes", [3000], 32, 8, 128, 16, "bf16", "bf16",
                                         "bf16", seed=1002))
    k = torch.cat([t.k_tokens, t.k_new]).float()
    k0 = torch.cat([plain.k_tokens, plain.k_new]).float()
    ratio = (k / torch.where(k0 == 0, torch.ones_like(k0), k0))
    spiked = ((ratio - 4.0).abs() < 0.05).all(dim=(1, 2))        # every head and channel x4
    assert int(spiked.sum()) == 30                               # floor(0.01 * 3000)
    assert torch.equal(t.v_tokens, plain.v_tokens)               # V untouched


def test_70b_lengths_log_uniform_and_prefix_blocks_shared():
    c = wl.FULL["llama70b_prefix_bs16"]()
    assert (c.batch, c.num_q_heads, c.num_kv_heads) == (64, 64, 8)
    assert c.seq_lens.min() >= 512 and c.seq_lens.max() <= 131072
    logs = np.log(c.seq_lens)
    assert np.log(2048) < np.median(logs) < np.log(32768)        # log-uniform, not uniform
    pb = 4096 // 16
    for s in range(c.batch):
        n = int(c.seq_lens[s])
        k = min(n, 4096) // 16                                   # full blocks inside the prefix
        assert np.array_equal(_blocks(c, s)[:k], c.shared_blocks[:k])
    ids = np.concatenate([_blocks(c, s)[min(int(n), 4096) // 16:]
                          for s, n in enumerate(c.seq_lens)])
    assert len(np.unique(ids)) == len(ids)                       # private blocks never shared
    assert not np.intersect1d(ids, c.shared_blocks[:pb]).size


def test_shared_prefix_tokens_carry_the_same_values():
    c = wl.make_case("shared", [100, 70, 33], 4, 2, 64, 16, "bf16", "bf16", "bf16", seed=5,
                     shared_prefix_tokens=64)
    t = wl.make_tensors(c)
    k = {}
    for i in range(t.tok_seq.numel()):
        s, p = int(t.tok_seq[i]), int(t.tok_pos[i])
        k[(s, p)] = t.k_tokens[i]
    for p in range(32):                                          # inside every sequence's prefix
        assert torch.equal(k[(0, p)], k[(1, p)]) and torch.equal(k[(0, p)], k[(2, p)])
    assert not torch.equal(k[(0, 70 - 2)], k[(1, 70 - 2)])       # past the prefix: private


def test_prefix_args_round_to_whole_blocks():
    c = wl.make_case("pa", [100, 70, 33], 4, 2, 64, 16, "bf16", "bf16", "bf16", seed=5,
                     shared_prefix_tokens=64)
    table, used, lens = wl.prefix_args(c)
    assert used == 64 and len(table) == 4
    assert list(lens) == [64, 64, 32]
    table, used, lens = wl.prefix_args(c, 40)
    assert used == 32 and list(lens) == [32, 32, 32]


@pytest.mark.parametrize("name", ["tiny", "fp8_b8_32k", "long_128k_bs64", "shared_prefix_64k_b32"])
def test_cases_and_tensors_are_reproducible(name):
    a, b = wl.FULL[name](), wl.FULL[name]()
    assert np.array_equal(a.seq_lens, b.seq_lens) and np.array_equal(a.tables, b.tables)
    if name in ("tiny",):
        ta, tb = wl.make_tensors(a), wl.make_tensors(b)
        for f in ("k_tokens", "v_tokens", "q", "k_new", "v_new", "tok_seq", "tok_pos"):
            assert torch.equal(getattr(ta, f), getattr(tb, f)), f


def test_tensors_place_every_token_once():
    c = wl.FULL["tiny"]()
    t = wl.make_tensors(c)
    pairs = set(zip(t.tok_seq.tolist(), t.tok_pos.tolist()))
    assert len(pairs) == t.tok_seq.numel()
    for s, n in enumerate(c.seq_lens):
        assert {(s, p) for p in range(int(n) - 1)} <= pairs      # all but the appended token
        assert (s, int(n) - 1) not in pairs
    assert t.new_pos.tolist() == [int(n) - 1 for n in c.seq_lens]


def test_block_waste_is_internal_fragmentation():
    c = wl.make_case("w", [16, 17, 31], 4, 2, 64, 16, "bf16", "bf16", "bf16", seed=1)
    slots = 16 * (1 + 2 + 2)
    assert wl.block_waste(c) == pytest.approx((slots - (16 + 17 + 31)) / slots)
