"""Shared-prefix decode (needs a GPU): paged_decode_attention_cascade reads the
blocks shared by many sequences once (tcgen05 prefix pass) and their private
suffixes through the decode kernel, then merges; a prefix small enough to stay in
L2 goes through the plain decode instead.  Every route must equal the fp64
oracle's attention over each sequence's whole table, within the decode bound
max |err| <= 2e-3 x max|V| per sequence (5e-3 for E4M3 pools)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, assert_parity, oracle_side

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_215_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def _cases():
    return [
        # 64 query / 8 KV heads, lengths 512 .. 20000, first 4096 tokens' full blocks shared
        (wl.llama70b_prefix(batch=6, lo=512, hi=20000, block_size=16, seed=16), [4096, 1024]),
        (wl.llama70b_prefix(batch=6, lo=512, hi=20000, block_size=32, seed=17), [4096]),
        # 32 / 8 heads; sequences wholly inside the prefix (256, 32), one shorter than it
        (wl.make_case("casc_g4", [256, 100, 4096 + 17, 32, 1000], 32, 8, 128, 16, "bf16", "bf16",
                      "bf16", seed=90, shared_prefix_tokens=256), [256, 128]),
        (wl.make_case("casc_f16_bs64", [700, 129, 2000], 32, 8, 128, 64, "f16", "f16", "f16",
                      seed=91, shared_prefix_tokens=640), [640]),
        # E4M3 pool, per-tensor scales (the prefix pass converts each tile to f16)
        (wl.make_case("casc_fp8", [300, 40, 2000, 777], 32, 8, 128, 16, "e4m3", "bf16", "bf16",
                      seed=92, shared_prefix_tokens=256), [256, 128]),
        # 16 query heads per KV head (two n-tiles in the decode kernel), block size 32
        (wl.make_case("casc_g16_bs32", [700, 300, 2000], 128, 8, 128, 32, "bf16", "bf16", "bf16",
                      seed=93, shared_prefix_tokens=256), [256]),
        (wl.make_case("casc_g16_bs16", [900, 200, 1700], 128, 8, 128, 16, "bf16", "bf16", "bf16",
                      seed=94, shared_prefix_tokens=512), [512, 256]),
        (wl.make_case("casc_g16_fp8_bs16", [900, 200, 1700], 64, 4, 128, 16, "e4m3", "bf16",
                      "bf16", seed=95, shared_prefix_tokens=512), [512]),
    ]


CASES = _cases()
_SIDE = {}


def _sides(case):
    if case.name not in _SIDE:
        tens = wl.make_tensors(case)
        gc = GpuCase(case, tens)
        pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
        gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos, gc.k_scale,
                       gc.v_scale)
        _SIDE[case.name] = (gc, pool, ref, seqs)
    return _SIDE[case.name]


def _prefix(case, used):
    table, used, lens = wl.prefix_args(case, used)
    return torch.from_numpy(table).cuda(), used, torch.from_numpy(lens).cuda()


@pytest.mark.parametrize("route", [3, 0, 2], ids=["prefix_pass", "auto", "plain"])
@pytest.mark.parametrize("case,prefixes", CASES, ids=lambda c: getattr(c, "name", ""))
def test_cascade_matches_oracle_and_plain_decode(case, prefixes, route):
    from paged_kv_cache_215_gb300 import pkv
    gc, pool, ref, seqs = _sides(case)
    plain = gc.step(append=False)
    for used in prefixes + [0]:
        table, P, lens = _prefix(case, used)
        out = torch.full_like(plain, float("nan"))
        for _ in range(2):                                  # twice: reused workspace state
            pkv.paged_decode_attention_cascade(out, gc.q, gc.pool, case.layer, table, P, lens,
                                               gc.tables, gc.seq_lens, gc.max_seq_len,
                                               case.scale, gc.k_scale, gc.v_scale,
                                               opts=pkv.launch_opts(kernel=route))
        torch.cuda.synchronize()
        assert gc.status() == 0
        assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} prefix {P}")
        tol = 5e-3 if case.kv_dtype == "e4m3" else 2e-3
        assert (out - plain).abs().max().item() <= tol * float(plain.abs().max())
        if route != 3:                                      # these prefixes all fit in L2
            assert torch.equal(out, plain)


@pytest.mark.parametrize("route", [3, 0])
def test_cascade_reports_a_prefix_that_is_not_shared(route):
    from paged_kv_cache_215_gb300 import pkv
    case = CASES[2][0]
    gc, _, _, _ = _sides(case)
    table, P, lens = _prefix(case, 256)
    bad = table.clone()
    bad[3] = (bad[3] + 1) % case.num_blocks                 # no longer the sequences' block
    out = torch.empty(case.batch, case.num_q_heads, case.head_dim, device="cuda")
    o = pkv.launch_opts(kernel=route)
    pkv.paged_decode_attention_cascade(out, gc.q, gc.pool, case.layer, bad, P, lens, gc.tables,
                                       gc.seq_lens, gc.max_seq_len, case.scale, opts=o)
    assert gc.status() == pkv.PKV_EINVAL
    odd = lens.clone()
    odd[1] = 8                                              # not a multiple of the block size
    pkv.paged_decode_attention_cascade(out, gc.q, gc.pool, case.layer, table, P, odd, gc.tables,
                                       gc.seq_lens, gc.max_seq_len, case.scale, opts=o)
    assert gc.status() == pkv.PKV_EINVAL


def test_cascade_rejects_bad_arguments():
    from paged_kv_cache_215_gb300 import pkv
    c8 = CASES[4][0]
    g8, _, _, _ = _sides(c8)
    table, P, lens = _prefix(c8, 256)
    out = torch.empty(c8.batch, c8.num_q_heads, c8.head_dim, device="cuda")
    with pytest.raises(pkv.PkvError) as e:                  # an E4M3 pool needs its scales
        pkv.paged_decode_attention_cascade(out, g8.q, g8.pool, c8.layer, table, P, lens,
                                           g8.tables, g8.seq_lens, g8.max_seq_len, c8.scale,
                                           0.0, g8.v_scale)
    assert e.value.code == pkv.PKV_EINVAL
    c16 = CASES[2][0]
    g16, _, _, _ = _sides(c16)
    table, P, lens = _prefix(c16, 256)
    out = torch.empty(c16.batch, c16.num_q_heads, c16.head_dim, device="cuda")
    with pytest.raises(pkv.PkvError) as e:                  # not a route of this entry
        pkv.paged_decode_attention_cascade(out, g16.q, g16.pool, c16.layer, table, P, lens,
                                           g16.tables, g16.seq_lens, g16.max_seq_len, c16.scale,
                                           opts=pkv.launch_opts(kernel=1))
    assert e.value.code == pkv.PKV_EINVAL
