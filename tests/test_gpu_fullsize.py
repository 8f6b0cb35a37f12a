"""Parity at the full workload sizes the benchmark times (needs a GPU).

The GPU runs the whole batch in the benchmark's launch configuration
(automatic split, bf16 and fp32 output); the oracle builds its own pool for a
sample of sequences (through its own append) and computes every query head of
those sequences in fp64.  Bounds as in test_gpu_parity: max |err| <= 2e-3 x
max|V| (bf16 KV), 5e-3 x max|V| (E4M3 KV), plus half an output ulp for bf16
output; the sampled part of the pool must equal the oracle's byte for byte.
"""
import gc as _gc

import numpy as np
import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, assert_parity, oracle_side

pytestmark = pytest.mark.gpu


def _extremes(case, k=3):
    order = np.argsort(case.seq_lens)
    return sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})[:k]


SAMPLES = {
    "llama8b_b32_8k": lambda c: [0, 13, 31],
    "long_128k": lambda c: [0],
    "long_1m": lambda c: [0],
    "fp8_b8_32k": lambda c: [0, 7],
    "llama70b_prefix_bs16": _extremes,
    "llama70b_prefix_bs32": _extremes,
}


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_sampled_parity(name):
    case = wl.FULL[name]()
    tens = wl.make_tensors(case, device="cuda")
    g = GpuCase(case, tens)
    out_lo = g.step(out_dtype=case.out_dtype)          # the benchmark's output dtype
    out_32 = g.step(out_dtype="f32", append=False)
    torch.cuda.synchronize()
    assert g.status() == 0
    seqs = SAMPLES[name](case)
    pool, ref, seqs = oracle_side(case, tens, seqs, g.k_scale, g.v_scale)
    # the sampled sequences' blocks hold exactly the oracle's bytes
    gpu_pool = g.pool.view().cpu()
    ora_pool = torch.from_numpy(pool).view(gpu_pool.dtype).view(gpu_pool.shape)
    for s in seqs:
        n = int(case.seq_lens[s])
        blocks = torch.from_numpy(case.tables[s, :(n + case.block_size - 1) // case.block_size]
                                  .astype(np.int64))
        a, b = gpu_pool[blocks], ora_pool[blocks]          # [nb, 2, L, Hkv, bs, D]
        # token order is (block, slot): only the n slots the sequence uses are compared
        a = a.permute(0, 4, 1, 2, 3, 5).reshape(-1, *a.shape[1:4], a.shape[5])[:n].contiguous()
        b = b.permute(0, 4, 1, 2, 3, 5).reshape(-1, *b.shape[1:4], b.shape[5])[:n].contiguous()
        if a.element_size() == 2:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"pool bytes of sequence {s} differ"
    assert_parity(case, out_32, ref, pool, seqs, g.v_scale, name)
    assert_parity(case, out_lo, ref, pool, seqs, g.v_scale, name, out_dtype=case.out_dtype)
    del g, tens, pool
    _gc.collect()
    torch.cuda.empty_cache()


def test_full_size_shared_prefix_decode_sampled_parity():
    """The shared-prefix (cascade) decode on the 64K-token shared-document
    workload, whole batch on the GPU, sampled sequences against the oracle."""
    from paged_kv_cache_215_gb300 import pkv
    case = wl.FULL["shared_prefix_64k_b32"]()
    tens = wl.make_tensors(case, device="cuda")
    g = GpuCase(case, tens)
    g.pool.append(case.layer, g.k_new, g.v_new, g.tables, g.new_pos)
    table, P, lens = wl.prefix_args(case)
    out = torch.full((case.batch, case.num_q_heads, case.head_dim), float("nan"), device="cuda")
    pkv.paged_decode_attention_cascade(out, g.q, g.pool, case.layer, torch.from_numpy(table).cuda(),
                                       P, torch.from_numpy(lens).cuda(), g.tables, g.seq_lens,
                                       g.max_seq_len, case.scale)
    torch.cuda.synchronize()
    assert g.status() == 0
    seqs = _extremes(case)
    pool, ref, seqs = oracle_side(case, tens, seqs, g.k_scale, g.v_scale)
    assert_parity(case, out, ref, pool, seqs, g.v_scale, case.name)
    del g, tens, pool
    _gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_full_size_chunked_prefill_sampled_parity(kv):
    """The chunked-prefill workload the benchmark times (4 sequences x 16,384
    tokens whose last 2,048 are new, 32/8 heads, D 128, bs 16; bf16 or E4M3
    pool) on the tcgen05 kernel, whole batch on the GPU.  The oracle computes
    the first and the last 16 query tokens of two sequences: the last ones as
    the last 16 tokens of the sequence, the first ones as the last 16 tokens of
    the sequence cut right after them (the same causal key range)."""
    import oracle
    from paged_kv_cache_215_gb300 import pkv
    from tests.gpu_harness import TOL, vmax_per_seq
    from tests.helpers import np_raw
    B, ctx, chunk, m = 4, 16384, 2048, 16
    case = wl.make_case(f"fullsize_prefill_{kv}", [ctx] * B, 32, 8, 128, 16, kv, "bf16", "bf16",
                        seed=1007)
    tens = wl.make_tensors(case, device="cuda")
    g = GpuCase(case, tens)
    g.pool.append(case.layer, g.k_new, g.v_new, g.tables, g.new_pos, g.k_scale, g.v_scale)
    q = torch.randn(B, chunk, 32, 128, generator=torch.Generator().manual_seed(78)).bfloat16()
    out = torch.full((B, chunk, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.paged_decode_attention_mq(out, q.cuda(), g.pool, case.layer, g.tables, g.seq_lens,
                                  g.max_seq_len, case.scale, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    assert g.status() == 0
    pool, _, seqs = oracle_side(case, tens, [0, 3], g.k_scale, g.v_scale)
    vm = vmax_per_seq(case, pool, seqs, g.v_scale)
    got = out.double().cpu().numpy()
    for s in seqs:
        for first, n in ((0, ctx - chunk + m), (chunk - m, ctx)):
            ref, _ = oracle.decode_mq(np_raw(q[s:s + 1, first:first + m]), "bf16", pool, kv,
                                      case.geometry, case.layer, case.tables[s:s + 1],
                                      np.array([n], dtype=np.int32), m, case.scale, g.k_scale,
                                      g.v_scale)
            err = np.abs(got[s, first:first + m] - ref[0])
            bound = TOL[kv] * vm[s] + 2.0 ** -8 * np.abs(ref[0])   # + half a bf16 ulp
            assert np.all(err <= bound), f"{kv} seq {s} tokens {first}+: {err.max():.3e}"
    del g, tens, pool
    _gc.collect()
    torch.cuda.empty_cache()
