"""Multi-token decode (needs a GPU): the last q_len tokens of every sequence
attend causally over the paged pool.  CUDA path vs the fp64 oracle, same bounds
as the single-token tests: max |err| <= 2e-3 x max|V| (bf16/f16 KV),
5e-3 x max|V| (E4M3 KV)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import TOL, GpuCase, oracle_side, vmax_per_seq
from tests.helpers import np_raw

pytestmark = pytest.mark.gpu


def _q(case, q_len, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(case.batch, q_len, case.num_q_heads, case.head_dim, generator=g).to(
        wl.TORCH_DT[case.q_dtype])


CASES = [
    (wl.make_case("mq_g4_bs16", [1, 2, 17, 500, 1033], 32, 8, 128, 16, "bf16", "bf16", "bf16",
                  seed=60), [1, 2, 3, 4]),
    (wl.make_case("mq_g8_bs32", [3, 64, 777], 64, 8, 128, 32, "bf16", "bf16", "bf16",
                  seed=61), [1, 2]),
    (wl.make_case("mq_fp8_g4", [5, 300, 2100], 32, 8, 128, 16, "e4m3", "bf16", "bf16",
                  seed=62), [2, 4]),
    (wl.make_case("mq_f16_g4", [40, 999], 32, 8, 128, 16, "f16", "f16", "f16", seed=63), [4]),
    (wl.make_case("mq_bs64_g4", [70, 640], 32, 8, 128, 64, "bf16", "bf16", "bf16", seed=64), [2]),
    (wl.make_case("mq_g2_empty", [0, 1, 9], 4, 2, 128, 16, "bf16", "bf16", "bf16", seed=65),
     [3, 8]),
]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("case,q_lens", CASES, ids=lambda c: getattr(c, "name", ""))
def test_multi_token_decode_parity(case, q_lens, splits):
    from paged_kv_cache_215_gb300 import pkv
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos, gc.k_scale,
                   gc.v_scale)
    pool, _, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(gc.pool.storage.cpu().numpy(), pool)
    vm = vmax_per_seq(case, pool, seqs, gc.v_scale)
    for q_len in q_lens:
        q = _q(case, q_len, seed=q_len)
        ref, _ = oracle.decode_mq(np_raw(q), case.q_dtype, pool, case.kv_dtype, case.geometry,
                                  case.layer, case.tables, case.seq_lens, q_len, case.scale,
                                  gc.k_scale, gc.v_scale)
        out = torch.full((case.batch, q_len, case.num_q_heads, case.head_dim), float("nan"),
                         device="cuda")
        pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, case.layer, gc.tables, gc.seq_lens,
                                      gc.max_seq_len, case.scale, gc.k_scale, gc.v_scale,
                                      num_splits=splits)
        torch.cuda.synchronize()
        assert gc.status() == 0
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        for s in seqs:
            err = np.abs(got[s] - ref[s]).max()
            assert err <= TOL[case.kv_dtype] * vm[s], f"{case.name} q_len {q_len} seq {s}: {err}"


def test_multi_token_decode_with_one_token_equals_decode():
    from paged_kv_cache_215_gb300 import pkv
    case = wl.llama8b_batch(batch=4, lo=100, hi=900, seed=66)
    gc = GpuCase(case)
    single = gc.step()
    out = torch.empty(case.batch, 1, 32, 128, device="cuda")
    pkv.paged_decode_attention_mq(out, gc.q.view(case.batch, 1, 32, 128), gc.pool, 0, gc.tables,
                                  gc.seq_lens, gc.max_seq_len, case.scale)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], single)


def test_large_chunks_route_to_tcgen05():
    """More than 16 query rows per KV head run on the tcgen05 kernel, bf16 and
    E4M3 pools alike (checked against the oracle)."""
    from paged_kv_cache_215_gb300 import pkv
    case = wl.llama8b_batch(batch=2, lo=100, hi=200, seed=67)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos)
    pool, _, seqs = oracle_side(case, tens, None)
    q = _q(case, 5, seed=5)                                      # 5 x 4 = 20 rows
    ref, _ = oracle.decode_mq(np_raw(q), "bf16", pool, "bf16", case.geometry, 0, case.tables,
                              case.seq_lens, 5, case.scale)
    out = torch.empty(2, 5, 32, 128, device="cuda")
    pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, 0, gc.tables, gc.seq_lens,
                                  gc.max_seq_len, case.scale)
    torch.cuda.synchronize()
    vm = vmax_per_seq(case, pool, seqs, 1.0)
    got = out.double().cpu().numpy()
    for s_ in seqs:
        assert np.abs(got[s_] - ref[s_]).max() <= TOL["bf16"] * vm[s_]
    c8 = wl.make_case("mq_fp8_big", [300], 32, 8, 128, 16, "e4m3", "bf16", "bf16", seed=68)
    t8 = wl.make_tensors(c8)
    g8 = GpuCase(c8, t8)
    g8.pool.append(0, g8.k_new, g8.v_new, g8.tables, g8.new_pos, g8.k_scale, g8.v_scale)
    pool8, _, seqs8 = oracle_side(c8, t8, None, g8.k_scale, g8.v_scale)
    q8 = _q(c8, 5, seed=6)
    ref8, _ = oracle.decode_mq(np_raw(q8), "bf16", pool8, "e4m3", c8.geometry, 0, c8.tables,
                               c8.seq_lens, 5, c8.scale, g8.k_scale, g8.v_scale)
    out8 = torch.empty(1, 5, 32, 128, device="cuda")
    pkv.paged_decode_attention_mq(out8, q8.cuda(), g8.pool, 0, g8.tables, g8.seq_lens,
                                  g8.max_seq_len, c8.scale, g8.k_scale, g8.v_scale)
    torch.cuda.synchronize()
    assert g8.status() == 0
    vm8 = vmax_per_seq(c8, pool8, seqs8, g8.v_scale)
    assert np.abs(out8.double().cpu().numpy()[0] - ref8[0]).max() <= TOL["e4m3"] * vm8[0]
