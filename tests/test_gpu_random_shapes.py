"""Decode attention on seeded random shapes against the fp64 oracle (needs a GPU).

Forty configurations drawn from a fixed seed, each a small batch through the
public entry points: KV heads 1-8, GQA groups 1-8 (the mhpn.cn long-context
article, section 3.2: query head h reads KV head h / G), head_dim 64 / 128,
block sizes 16 / 32 / 64 ("The engineering truth of long-context inference
2026", section 2.3), bf16 / f16 / E4M3 pools ("Unlocking long context",
section 3.2), f32 / bf16 outputs, the
automatic split or a fixed one of three partitions, and sequence lengths mixed
from the edges (0, 1, a block minus one, a block, a block plus one) and random
lengths up to 3000.  One step appends each sequence's new token, then attends;
every output must be within 2e-3 x max|V| (16-bit pools) or 5e-3 x max|V|
(E4M3) of the oracle (plus half an output ulp for bf16 output).  A third of
the configurations also run a 2- or 3-token causal decode through
paged_decode_attention_mq against the oracle's multi-token attention.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, TOL, assert_parity, oracle_side, vmax_per_seq
from tests.helpers import np_raw

pytestmark = pytest.mark.gpu

N_CONFIGS = 40


def _config(i):
    r = np.random.RandomState(9100 + i)
    hkv = int(r.choice([1, 2, 4, 8]))
    g = int(r.choice([1, 2, 4, 8]))
    d = int(r.choice([128, 128, 64]))
    bs = int(r.choice([16, 32, 64]))
    kv = str(r.choice(["bf16", "f16", "e4m3"]))
    q = "bf16" if kv in ("bf16", "e4m3") else "f16"
    out = str(r.choice(["f32", "bf16"]))
    b = int(r.randint(1, 7))
    edges = [0, 1, bs - 1, bs, bs + 1]
    lens = [int(r.choice(edges)) if r.rand() < 0.4 else int(r.randint(2, 3001)) for _ in range(b)]
    lens = [max(n, 1) for n in lens]           # every sequence holds at least its new token
    if r.rand() < 0.2:
        lens[0] = 0                            # ... except an empty one, now and then
    splits = int(r.choice([0, 0, 3]))
    q_len = int(r.choice([2, 3])) if i % 3 == 0 else 1
    return dict(hkv=hkv, g=g, d=d, bs=bs, kv=kv, q=q, out=out, lens=lens, splits=splits,
                q_len=q_len)


@pytest.mark.parametrize("i", range(N_CONFIGS))
def test_random_shape_matches_oracle(i):
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    c = _config(i)
    case = wl.make_case(f"rand{i}", c["lens"], c["hkv"] * c["g"], c["hkv"], c["d"], c["bs"],
                        c["kv"], c["q"], c["out"], seed=9300 + i)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    try:
        out = gc.step(out_dtype=c["out"], num_splits=c["splits"])
    except pkv.PkvError as e:
        if e.code == pkv.PKV_EUNSUPPORTED:
            pytest.skip(f"no kernel for {c}")
        raise
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"rand{i} {c}", out_dtype=c["out"])
    if c["q_len"] == 1:
        return
    # multi-token decode: the last q_len tokens of each sequence attend causally
    q_len = c["q_len"]
    g = torch.Generator().manual_seed(9500 + i)
    qm = torch.randn(case.batch, q_len, case.num_q_heads, case.head_dim, generator=g)
    qm = qm.to(torch.bfloat16 if c["q"] == "bf16" else torch.float16)
    refm, _ = oracle.decode_mq(np_raw(qm), c["q"], pool, c["kv"], case.geometry, case.layer,
                               case.tables, case.seq_lens, q_len, case.scale, gc.k_scale,
                               gc.v_scale)
    outm = torch.full((case.batch, q_len, case.num_q_heads, case.head_dim), float("nan"),
                      device="cuda")
    try:
        pkv.paged_decode_attention_mq(outm, qm.cuda(), gc.pool, case.layer, gc.tables,
                                      gc.seq_lens, gc.max_seq_len, case.scale, gc.k_scale,
                                      gc.v_scale, num_splits=c["splits"])
    except pkv.PkvError as e:
        if e.code == pkv.PKV_EUNSUPPORTED:
            return
        raise
    torch.cuda.synchronize()
    assert gc.status() == 0
    vm = vmax_per_seq(case, pool, seqs, gc.v_scale)
    got = outm.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    for s in seqs:
        err = float(np.abs(got[s] - refm[s]).max())
        assert err <= TOL[c["kv"]] * vm[s], f"rand{i} mq seq {s}: {err} {c}"
