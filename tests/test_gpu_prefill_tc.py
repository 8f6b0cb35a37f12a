"""Chunked prefill on the tcgen05 kernel (needs a GPU): the last q_len tokens of
every sequence attend causally over the paged pool, many query rows per KV
head (UMMA tiles of 128 rows).  CUDA path vs the fp64 oracle's causal decode:
max |err| <= 2e-3 x max|V| per sequence (5e-3 for E4M3 pools, the oracle
dequantising the same bytes)."""
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
    (wl.make_case("tc_g4_bs16", [300, 1000, 40], 32, 8, 128, 16, "bf16", "bf16", "bf16",
                  seed=80), [17, 64, 100]),
    (wl.make_case("tc_g8_bs32", [500, 2000], 64, 8, 128, 32, "bf16", "bf16", "bf16", seed=81),
     [48]),
    (wl.make_case("tc_f16_bs64", [700, 129], 32, 8, 128, 64, "f16", "f16", "f16", seed=82),
     [130]),
    (wl.make_case("tc_mha_bs16", [260, 77], 4, 4, 128, 16, "bf16", "bf16", "bf16", seed=83),
     [128, 200]),
    # E4M3 pools: each tile converted to f16 with the per-tensor scales
    (wl.make_case("tc_fp8_g4_bs16", [300, 1000, 40], 32, 8, 128, 16, "e4m3", "bf16", "bf16",
                  seed=86, spike_frac=0.01), [17, 100]),
    (wl.make_case("tc_fp8_g8_bs32_f16q", [500, 2000], 64, 8, 128, 32, "e4m3", "f16", "f16",
                  seed=87), [48]),
    (wl.make_case("tc_fp8_bs64", [700, 129], 32, 8, 128, 64, "e4m3", "bf16", "bf16", seed=88),
     [130]),
]


def _check(case, q_lens, kernel, scale=None):
    from paged_kv_cache_215_gb300 import pkv
    scale = case.scale if scale is None else scale
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos, gc.k_scale, gc.v_scale)
    pool, _, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    vm = vmax_per_seq(case, pool, seqs, gc.v_scale)
    worst = 0.0
    for q_len in q_lens:
        q = _q(case, q_len, seed=q_len)
        ref, _ = oracle.decode_mq(np_raw(q), case.q_dtype, pool, case.kv_dtype, case.geometry,
                                  case.layer, case.tables, case.seq_lens, q_len, scale,
                                  gc.k_scale, gc.v_scale)
        out = torch.full((case.batch, q_len, case.num_q_heads, case.head_dim), float("nan"),
                         device="cuda")
        pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, case.layer, gc.tables,
                                      gc.seq_lens, gc.max_seq_len, scale, gc.k_scale, gc.v_scale,
                                      opts=pkv.launch_opts(kernel=kernel) if kernel else None)
        torch.cuda.synchronize()
        assert gc.status() == 0
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        for s in seqs:
            err = np.abs(got[s] - ref[s]).max()
            bound = TOL[case.kv_dtype] * vm[s]
            worst = max(worst, err / bound)
            assert err <= bound, f"{case.name} q_len {q_len} seq {s}: {err} > {bound}"
    return worst


@pytest.mark.parametrize("case,q_lens", CASES, ids=lambda c: getattr(c, "name", ""))
def test_chunked_prefill_tcgen05_parity(case, q_lens):
    _check(case, q_lens, kernel=0)


def test_tcgen05_e4m3_every_code():
    """A pool whose bytes are drawn from all 254 finite E4M3 codes (subnormals,
    both zeros, +-448): the tcgen05 kernel's E4M3 -> f16 tiles against the
    oracle's decoding of the same bytes."""
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("tc_fp8_codes", [200, 70], 32, 8, 128, 16, "e4m3", "bf16", "bf16", seed=89)
    gc = GpuCase(case)
    rng = np.random.default_rng(89)
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    pool = rng.choice(codes, size=gc.pool.storage.numel()).astype(np.uint8)
    gc.pool.storage.copy_(torch.from_numpy(pool))
    ks, vs = 0.02, 0.03
    seqs = list(range(case.batch))
    vm = vmax_per_seq(case, pool, seqs, vs)
    for q_len in (40, 70):
        q = _q(case, q_len, seed=q_len)
        ref, _ = oracle.decode_mq(np_raw(q), "bf16", pool, "e4m3", case.geometry, case.layer,
                                  case.tables, case.seq_lens, q_len, case.scale, ks, vs)
        out = torch.full((case.batch, q_len, 32, 128), float("nan"), device="cuda")
        pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, case.layer, gc.tables, gc.seq_lens,
                                      gc.max_seq_len, case.scale, ks, vs)
        torch.cuda.synchronize()
        assert gc.status() == 0
        got = out.double().cpu().numpy()
        for s_ in seqs:
            err = np.abs(got[s_] - ref[s_]).max()
            assert err <= TOL["e4m3"] * vm[s_], f"q_len {q_len} seq {s_}: {err}"


def test_tcgen05_kernel_forced_on_short_chunks():
    case = wl.make_case("tc_forced", [90, 33, 5], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=84)
    _check(case, [1, 2, 7], kernel=3)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("scale", [-0.125, 0.3])
def test_tcgen05_softmax_scale_sign_and_size(scale, kv):
    """A negative scale (carried on Q by the kernel) and a large one (frequent
    rescales of O) against the oracle at the same scale; on E4M3 pools the scale
    also carries k_scale."""
    case = wl.make_case(f"tc_scale_{kv}", [400, 129], 32, 8, 128, 16, kv, "bf16", "bf16",
                        seed=85)
    _check(case, [64, 100], kernel=0, scale=scale)
