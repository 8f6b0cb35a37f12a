"""Decode steps chained with programmatic dependent launch (needs a GPU).

With launch_opts(pdl=1) a decode step's attention kernel may start while the
previous step's attention and merge are still running; it must wait for them
before it loads the blocks holding the previous step's new token (and before it
writes anything).  Here 40 steps run back to back on one stream with no copy or
host call between them (tables, lengths and every step's q and new token are
on the device beforehand), so each step's kernels follow the previous step's
directly; every step attends over the token the step before it stored.  Each
step's output must match the fp64 oracle over that step's tokens within
2e-3 x max|V| ("Unlocking long context", section 4.1 attention over the paged
cache of "The engineering truth of long-context inference 2026", section 2.2).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import np_raw

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128
STEPS = 40


@pytest.mark.parametrize("lens0", [[37, 300, 16], [4000, 1, 95, 2048]], ids=["short", "mixed"])
def test_chained_steps_see_the_previous_token(lens0):
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    bs = 16
    B = len(lens0)
    g = torch.Generator().manual_seed(4242 + B)
    rnd = lambda *shape: torch.randn(*shape, generator=g).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    nb = sum((n + STEPS + bs - 1) // bs for n in lens0) + 4
    geom = pkv.geometry(1, HQ, HKV, D, bs, nb, "bf16")
    pool = pkv.KVPool(geom)
    pool.storage.fill_(0xFF)                       # unwritten slots hold bf16 NaN patterns
    max_blocks = max((n + STEPS + bs - 1) // bs for n in lens0)
    tables = np.full((B, max_blocks), -1, np.int32)
    lens = np.zeros(B, np.int32)
    # every block the prompt and all steps need, taken before the first step
    pool.prepare_append(lens, tables, new_tokens=[n + STEPS for n in lens0])
    keys = [[rnd(HKV, D) for _ in range(n)] for n in lens0]
    vals = [[rnd(HKV, D) for _ in range(n)] for n in lens0]
    k0 = torch.stack([x for ks in keys for x in ks]).cuda()
    v0 = torch.stack([x for vs in vals for x in vs]).cuda()
    tok_seq = torch.tensor([s for s, n in enumerate(lens0) for _ in range(n)], dtype=torch.int32)
    tok_pos = torch.tensor([p for n in lens0 for p in range(n)], dtype=torch.int32)
    td = torch.from_numpy(tables).cuda()
    pool.append_tokens(0, k0, v0, td, tok_seq.cuda(), tok_pos.cuda())
    q = rnd(STEPS, B, HQ, D)
    kn, vn = rnd(STEPS, B, HKV, D), rnd(STEPS, B, HKV, D)
    qd, knd, vnd = q.cuda(), kn.cuda(), vn.cuda()
    lens_d = torch.tensor([[n + i + 1 for n in lens0] for i in range(STEPS)], dtype=torch.int32,
                          device="cuda")
    out = torch.full((STEPS, B, HQ, D), float("nan"), device="cuda")
    ws = torch.empty(pkv.workspace_bytes(geom, B, max(lens0) + STEPS, 0), dtype=torch.uint8,
                     device="cuda")
    opts = pkv.launch_opts(pdl=1)
    torch.cuda.synchronize()
    for i in range(STEPS):
        pkv.paged_decode_step(out[i], qd[i], knd[i], vnd[i], pool, 0, td, lens_d[i],
                              max(lens0) + i + 1, scale, workspace=ws, opts=opts)
    torch.cuda.synchronize()
    assert pool.check_status() == 0
    got = out.double().cpu().numpy()
    for i in range(STEPS):
        for s in range(B):
            keys[s].append(kn[i, s])
            vals[s].append(vn[i, s])
        n = np.array([len(k) for k in keys], np.int32)
        MB = int((n.max() + bs - 1) // bs)
        geo = dict(num_layers=1, num_q_heads=HQ, num_kv_heads=HKV, head_dim=D, block_size=bs,
                   num_blocks=B * MB)
        otab = np.arange(B * MB, dtype=np.int32).reshape(B, MB)
        opool = np.zeros(oracle.kv_bytes(1, HKV, D, B * MB * bs, 2), np.uint8)
        seq = np.concatenate([np.full(m, s, np.int32) for s, m in enumerate(n)])
        pos = np.concatenate([np.arange(m, dtype=np.int32) for m in n])
        kk = torch.stack([x for ks in keys for x in ks])
        vv = torch.stack([x for vs in vals for x in vs])
        oracle.append_tokens(opool, "bf16", geo, 0, np_raw(kk), np_raw(vv), "bf16", otab, seq, pos)
        ref, _, _ = oracle.decode(np_raw(q[i]), "bf16", opool, "bf16", geo, 0, otab, n, scale)
        for s in range(B):
            vmax = float(torch.stack(vals[s]).float().abs().max())
            err = float(np.abs(got[i, s] - ref[s]).max())
            assert np.isfinite(got[i, s]).all(), (i, s)
            assert err <= 2e-3 * vmax, f"step {i} seq {s}: {err}"
