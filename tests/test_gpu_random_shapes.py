"""Seeded random shapes against the fp64 oracle (needs a GPU): decode, chunked
prefill on the tcgen05 kernel, and shared-prefix decode.

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


N_PREFILL = 16


def _prefill_config(i):
    r = np.random.RandomState(9700 + i)
    hkv = int(r.choice([1, 2, 4, 8]))
    g = int(r.choice([1, 2, 4, 8, 16]))
    bs = int(r.choice([16, 32, 64]))
    kv = str(r.choice(["bf16", "f16", "e4m3"]))
    q = kv if kv != "e4m3" else str(r.choice(["bf16", "f16"]))
    b = int(r.randint(1, 5))
    q_len = int(r.randint(max(17, 16 // g + 1), 301))
    lens = [int(r.choice([r.randint(1, q_len + 1), r.randint(q_len, 3001), bs * r.randint(1, 40)]))
            for _ in range(b)]
    kernel = int(r.choice([0, 3]))
    return dict(hkv=hkv, g=g, bs=bs, kv=kv, q=q, lens=lens, q_len=q_len, kernel=kernel)


@pytest.mark.parametrize("i", range(N_PREFILL))
def test_random_chunked_prefill_matches_oracle(i):
    """Chunked prefill (q_len 17-300, more than 16 query rows per KV head, so the
    automatic route and kernel = 3 both take the tcgen05 kernel) over random head
    counts, GQA groups up to 16, block sizes, pool and query dtypes and lengths
    (some shorter than the chunk), against the oracle's causal multi-token
    attention ("Unlocking long context", section 5.2)."""
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    c = _prefill_config(i)
    case = wl.make_case(f"rand_pf{i}", c["lens"], c["hkv"] * c["g"], c["hkv"], 128, c["bs"],
                        c["kv"], c["q"], c["q"], seed=9800 + i)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos, gc.k_scale, gc.v_scale)
    pool, _, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    g = torch.Generator().manual_seed(9900 + i)
    q = torch.randn(case.batch, c["q_len"], case.num_q_heads, 128, generator=g).to(
        wl.TORCH_DT[c["q"]])
    ref, _ = oracle.decode_mq(np_raw(q), c["q"], pool, c["kv"], case.geometry, case.layer,
                              case.tables, case.seq_lens, c["q_len"], case.scale, gc.k_scale,
                              gc.v_scale)
    out = torch.full((case.batch, c["q_len"], case.num_q_heads, 128), float("nan"), device="cuda")
    pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, case.layer, gc.tables, gc.seq_lens,
                                  gc.max_seq_len, case.scale, gc.k_scale, gc.v_scale,
                                  opts=pkv.launch_opts(kernel=c["kernel"]))
    torch.cuda.synchronize()
    assert gc.status() == 0
    vm = vmax_per_seq(case, pool, seqs, gc.v_scale)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got)), c
    for s in seqs:
        err = float(np.abs(got[s] - ref[s]).max())
        assert err <= TOL[c["kv"]] * vm[s], f"rand_pf{i} seq {s}: {err} {c}"


N_CASCADE = 12


def _cascade_config(i):
    r = np.random.RandomState(10100 + i)
    hkv = int(r.choice([2, 4, 8]))
    g = int(r.choice([1, 2, 4, 8]))
    bs = int(r.choice([16, 32, 64]))
    kv = str(r.choice(["bf16", "f16", "e4m3"]))
    q = "f16" if kv == "f16" else "bf16"
    prefix = bs * int(r.randint(1, 2049 // bs + 1))
    b = int(r.randint(2, 9))
    # inside the prefix, exactly the prefix, or the prefix and a private suffix
    lens = [int(r.choice([r.randint(1, prefix + 1), prefix, prefix + r.randint(1, 2001)]))
            for _ in range(b)]
    used = int(r.choice([prefix, bs * r.randint(1, prefix // bs + 1)]))
    route = int(r.choice([0, 3]))
    return dict(hkv=hkv, g=g, bs=bs, kv=kv, q=q, prefix=prefix, lens=lens, used=used, route=route)


@pytest.mark.parametrize("i", range(N_CASCADE))
def test_random_shared_prefix_matches_oracle(i):
    """paged_decode_attention_cascade over random shared prefixes (one block to
    2,048 tokens, all or part of it declared shared), sequences inside, equal to
    or beyond the prefix, GQA groups 1-8, block sizes and pool dtypes, by the
    forced prefix pass or the automatic route: each sequence's output against the
    oracle's attention over its whole table ("Unlocking long context", section 3.1
    shared blocks)."""
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    c = _cascade_config(i)
    case = wl.make_case(f"rand_casc{i}", c["lens"], c["hkv"] * c["g"], c["hkv"], 128, c["bs"],
                        c["kv"], c["q"], c["q"], seed=10200 + i,
                        shared_prefix_tokens=c["prefix"])
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos, gc.k_scale, gc.v_scale)
    table, P, plens = wl.prefix_args(case, c["used"])
    out = torch.full((case.batch, case.num_q_heads, 128), float("nan"),
                     dtype=wl.TORCH_DT[c["q"]], device="cuda")
    pkv.paged_decode_attention_cascade(out, gc.q, gc.pool, case.layer,
                                       torch.from_numpy(table).cuda(), P,
                                       torch.from_numpy(plens).cuda(), gc.tables, gc.seq_lens,
                                       gc.max_seq_len, case.scale, gc.k_scale, gc.v_scale,
                                       opts=pkv.launch_opts(kernel=c["route"]))
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"rand_casc{i} {c}", out_dtype=c["q"])
