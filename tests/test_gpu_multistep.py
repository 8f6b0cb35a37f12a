"""Many consecutive decode steps through the library's own block management
(needs a GPU).

Each step calls kv_pool_prepare_append (a fresh block when a sequence's next
token starts one, "The engineering truth of long-context inference 2026"
section 2.2; copy-on-write of a shared tail block, "Unlocking long context"
section 3.1), uploads the tables, and runs paged_decode_step, which stores the
new token and attends over every token.  Three sequences: two share a 40-token
prefix whose last block is only partly filled (so the first step must copy it
for one of them), the third is private.  After every one of 48 steps the
output must match the fp64 oracle, which keeps each sequence's tokens in its
own contiguous layout (no sharing, no copies), within 2e-3 x max|V|.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import np_raw

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128
STEPS = 48


def _oracle_step(seq_k, seq_v, q, bs, scale):
    """The oracle's own pool: sequence s in blocks [s*MB, s*MB + ceil(n/bs))."""
    B = len(seq_k)
    lens = np.array([len(k) for k in seq_k], np.int32)
    MB = int((lens.max() + bs - 1) // bs)
    geom = dict(num_layers=1, num_q_heads=HQ, num_kv_heads=HKV, head_dim=D, block_size=bs,
                num_blocks=B * MB)
    tables = np.arange(B * MB, dtype=np.int32).reshape(B, MB)
    pool = np.zeros(oracle.kv_bytes(1, HKV, D, B * MB * bs, 2), np.uint8)
    k = torch.cat([torch.stack(x) for x in seq_k])
    v = torch.cat([torch.stack(x) for x in seq_v])
    seq = np.concatenate([np.full(n, s, np.int32) for s, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lens])
    oracle.append_tokens(pool, "bf16", geom, 0, np_raw(k), np_raw(v), "bf16", tables, seq, pos)
    out, _, _ = oracle.decode(np_raw(q), "bf16", pool, "bf16", geom, 0, tables, lens, scale)
    vmax = [float(torch.stack(x).float().abs().max()) for x in seq_v]
    return out, vmax


@pytest.mark.parametrize("route", ["fused", "simt"])
@pytest.mark.parametrize("bs", [16, 32])
def test_decode_steps_grow_tables_and_copy_shared_tails(bs, route):
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    g = torch.Generator().manual_seed(1000 + bs)
    rnd = lambda *shape: torch.randn(*shape, generator=g).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    nb, max_blocks = 48, 16
    geom = pkv.geometry(1, HQ, HKV, D, bs, nb, "bf16")
    pool = pkv.KVPool(geom)
    pool.storage.fill_(0xFF)                      # unwritten slots hold bf16 NaN patterns
    tables = np.full((3, max_blocks), -1, np.int32)
    lens = np.zeros(3, np.int32)
    # sequence 0: a 40-token prompt; sequence 2: 23 tokens of its own
    first = pool.prepare_append(lens, tables, new_tokens=[40, 0, 23])
    assert list(first) == [0, -1, 0]
    seq_k = [[rnd(HKV, D) for _ in range(40)], [], [rnd(HKV, D) for _ in range(23)]]
    seq_v = [[rnd(HKV, D) for _ in range(40)], [], [rnd(HKV, D) for _ in range(23)]]
    k0 = torch.stack(seq_k[0] + seq_k[2]).cuda()
    v0 = torch.stack(seq_v[0] + seq_v[2]).cuda()
    tok_seq = torch.tensor([0] * 40 + [2] * 23, dtype=torch.int32, device="cuda")
    tok_pos = torch.tensor(list(range(40)) + list(range(23)), dtype=torch.int32, device="cuda")
    pool.append_tokens(0, k0, v0, torch.from_numpy(tables).cuda(), tok_seq, tok_pos)
    lens[:] = [40, 0, 23]
    # sequence 1 forks from sequence 0: the same blocks, one more reference each
    shared = tables[0, :(40 + bs - 1) // bs].copy()
    tables[1, :shared.size] = shared
    pool.share(shared.tolist())
    lens[1] = 40
    seq_k[1], seq_v[1] = list(seq_k[0]), list(seq_v[0])
    tail = 40 // bs                               # the partly filled shared block's entry
    copies = 0
    for step in range(STEPS):
        free_before = pool.num_free()
        first = pool.prepare_append(lens, tables)
        starts = [int(n) % bs == 0 for n in lens]
        if step == 0:
            # sequence 0 writes into the shared tail: it gets a copy; sequence 1,
            # now the tail's only owner, writes in place
            assert first[0] == tail and first[1] == (tail if starts[1] else -1)
            assert tables[0, tail] != tables[1, tail]
            assert pool.refcount(int(tables[1, tail])) == 1
            copies += 1
        for s in range(3):
            if step > 0:
                assert first[s] == (lens[s] // bs if starts[s] else -1)
        assert free_before - pool.num_free() == sum(starts) + (1 if step == 0 else 0)
        q = rnd(3, HQ, D)
        kn, vn = rnd(3, HKV, D), rnd(3, HKV, D)
        out = torch.full((3, HQ, D), float("nan"), device="cuda")
        after = torch.from_numpy(lens + 1).cuda()
        opts = pkv.launch_opts(kernel=1) if route == "simt" else None
        pkv.paged_decode_step(out, q.cuda(), kn.cuda(), vn.cuda(), pool, 0,
                              torch.from_numpy(tables).cuda(), after, int(lens.max()) + 1,
                              scale, opts=opts)
        for s in range(3):
            seq_k[s].append(kn[s])
            seq_v[s].append(vn[s])
        lens += 1
        torch.cuda.synchronize()
        assert pool.check_status() == 0, f"step {step}"
        ref, vmax = _oracle_step(seq_k, seq_v, q, bs, scale)
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"step {step}"
        for s in range(3):
            err = float(np.abs(got[s] - ref[s]).max())
            assert err <= 2e-3 * vmax[s], f"bs {bs} step {step} seq {s}: {err}"
    # the prompt's full blocks are still shared, the sequences diverged after them
    for j in range(tail):
        assert tables[0, j] == tables[1, j] and pool.refcount(int(tables[0, j])) == 2
    assert copies == 1 and lens.tolist() == [40 + STEPS, 40 + STEPS, 23 + STEPS]
