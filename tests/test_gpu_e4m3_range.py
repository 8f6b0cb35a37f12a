"""E4M3 paths across the whole input range (needs a GPU).

The E4M3 kernels run f16 tensor-core operands, so a legal bf16 q larger than
f16's range (or much smaller than 1), a per-block scale far from 1, or a long
tail of tiny softmax weights could leave f16's range.  These cases check every
route against the fp64 oracle (dequantising the same bytes) within
5e-3 x max|V| for E4M3 pools and 2e-3 x max|V| for f16 pools, and that no
output is NaN:
  - q scaled by 2^-20, 2^12 and 2^17 ("Unlocking long context" section 3.2
    pairs bf16 queries with the E4M3 cache): decode (balanced and fixed split),
    the mma.sync multi-token kernel and the tcgen05 chunked-prefill kernel;
  - per-block scales of blocks whose amax is far above 65504 or far below 1,
    and a pool mixing both, on every decode route and the tcgen05 kernel;
  - f32 q on an E4M3 pool (run in fp32 on the CUDA-core kernel);
  - one dominant key and 300K keys each 2^-26 as likely: the tail carries
    0.5% of the weight, which f16 P would round to zero.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import TOL, GpuCase, oracle_side, vmax_per_seq
from tests.helpers import np_raw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_215_gb300 import build
    build.build()


def _bf16(x):
    return x.float().to(torch.bfloat16)


def _assert_close(got, ref, seqs, vm, tol, what):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else got
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    for s in seqs:
        err = float(np.abs(got[s] - ref[s]).max())
        assert err <= tol * vm[s], f"{what} seq {s}: {err:.3e} > {tol} x {vm[s]:.3e}"


# ------------------------------------------------------------------ per-tensor scales, scaled q
QSCALES = [2.0 ** -20, 2.0 ** 12, 2.0 ** 17]


@pytest.mark.parametrize("qscale", QSCALES, ids=lambda x: f"q2^{int(np.log2(x))}")
@pytest.mark.parametrize("mode", ["auto", "split3", "simt", "fused"])
def test_e4m3_decode_with_scaled_q(qscale, mode):
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("e4m3_qrange", [3000, 777, 1, 64], 32, 8, 128, 16, "e4m3", "bf16",
                        "bf16", seed=300)
    tens = wl.make_tensors(case)
    tens.q = _bf16(tens.q * qscale)
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    if mode == "fused":
        out = gc.fused_step()
    else:
        opts = pkv.launch_opts(kernel=1) if mode == "simt" else None
        out = gc.step(num_splits=3 if mode == "split3" else 0, opts=opts)
    torch.cuda.synchronize()
    assert gc.status() == 0
    vm = vmax_per_seq(case, pool, seqs, gc.v_scale)
    _assert_close(out, ref, seqs, vm, TOL["e4m3"], f"{mode} q x {qscale}")


@pytest.mark.parametrize("qscale", QSCALES, ids=lambda x: f"q2^{int(np.log2(x))}")
@pytest.mark.parametrize("q_len", [3, 48])
def test_e4m3_multi_token_with_scaled_q(qscale, q_len):
    """q_len 3 (12 rows per KV head): the mma.sync kernel; q_len 48: tcgen05."""
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("e4m3_qrange_mq", [900, 300], 32, 8, 128, 16, "e4m3", "bf16", "bf16",
                        seed=301)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos, gc.k_scale, gc.v_scale)
    pool, _, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    g = torch.Generator().manual_seed(q_len)
    q = _bf16(torch.randn(case.batch, q_len, 32, 128, generator=g) * qscale)
    # one query row far smaller than the rest of its warp / tile
    q[0, 0, 0] = _bf16(q[0, 0, 0].float() * 2.0 ** -30)
    ref, _ = oracle.decode_mq(np_raw(q), "bf16", pool, "e4m3", case.geometry, case.layer,
                              case.tables, case.seq_lens, q_len, case.scale, gc.k_scale,
                              gc.v_scale)
    out = torch.full((case.batch, q_len, 32, 128), float("nan"), device="cuda")
    pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, case.layer, gc.tables, gc.seq_lens,
                                  gc.max_seq_len, case.scale, gc.k_scale, gc.v_scale)
    torch.cuda.synchronize()
    assert gc.status() == 0
    vm = vmax_per_seq(case, pool, seqs, gc.v_scale)
    _assert_close(out, ref, seqs, vm, TOL["e4m3"], f"mq{q_len} q x {qscale}")


def test_e4m3_decode_with_f32_q():
    """f32 q on an E4M3 pool keeps its 24 bits: the automatic route runs it on the
    CUDA cores in fp32 (f16 tensor-core operands would round it)."""
    case = wl.make_case("e4m3_q32", [2000, 100], 32, 8, 128, 16, "e4m3", "f32", "f32", seed=302)
    tens = wl.make_tensors(case)
    g = torch.Generator().manual_seed(5)
    tens.q = torch.randn(case.batch, 32, 128, generator=g) * 4096.0 + 0.1234567
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    out = gc.step()
    torch.cuda.synchronize()
    assert gc.status() == 0
    _assert_close(out, ref, seqs, vmax_per_seq(case, pool, seqs, gc.v_scale), TOL["e4m3"],
                  "f32 q")


# ------------------------------------------------------------------ per-block scales far from 1
def _block_pool(case, tens):
    """Library pool with per-block scales (kv_block_scales over every token), and the
    oracle's scales and pool built the same way on the CPU."""
    from paged_kv_cache_215_gb300 import pkv
    dev = "cuda"
    g = pkv.geometry(case.num_layers, case.num_q_heads, case.num_kv_heads, case.head_dim,
                     case.block_size, case.num_blocks, "e4m3")
    pool = pkv.KVPool(g)
    pool.storage.zero_()
    ids = case.tables[case.tables >= 0]
    uniq, counts = np.unique(ids, return_counts=True)
    pool.reserve(uniq.tolist())
    if (counts > 1).any():
        pool.share(np.repeat(uniq, counts - 1).tolist())
    scales = torch.ones((case.num_blocks, 2, case.num_layers, case.num_kv_heads),
                        dtype=torch.float32, device=dev)
    pool.set_block_scales(scales)
    tables = torch.from_numpy(case.tables).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    seq = torch.cat([tens.tok_seq, torch.arange(case.batch, dtype=torch.int32)])
    pos = torch.cat([tens.tok_pos, tens.new_pos])
    k_all = torch.cat([tens.k_tokens, tens.k_new])
    v_all = torch.cat([tens.v_tokens, tens.v_new])
    keep = pos >= 0
    seq, pos, k_all, v_all = seq[keep], pos[keep], k_all[keep], v_all[keep]
    pool.compute_block_scales(case.layer, k_all.to(dev), v_all.to(dev), tables, seq.to(dev),
                              pos.to(dev))
    pool.append_tokens(case.layer, k_all.to(dev), v_all.to(dev), tables, seq.to(dev),
                       pos.to(dev))
    osc = np.ones(tuple(scales.shape), np.float32)
    oracle.block_scales(osc, case.geometry, case.layer, np_raw(k_all), np_raw(v_all), "bf16",
                        case.tables, np_raw(seq), np_raw(pos))
    opool = np.zeros(pool.nbytes, np.uint8)
    oracle.append_tokens(opool, "e4m3", case.geometry, case.layer, np_raw(k_all), np_raw(v_all),
                         "bf16", case.tables, np_raw(seq), np_raw(pos), block_scales=osc)
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(pool.storage.cpu().numpy(), opool)
    return pool, tables, lens, osc, opool


def _vmax_blocks(case, opool, osc):
    dec = torch.from_numpy(opool).view(torch.float8_e4m3fn).double().numpy().reshape(
        case.num_blocks, 2, case.num_layers, case.num_kv_heads, case.block_size,
        case.head_dim) * osc[:, :, :, :, None, None].astype(np.float64)
    vm = {}
    for s in range(case.batch):
        n = int(case.seq_lens[s])
        blocks = case.tables[s, :(n + case.block_size - 1) // case.block_size]
        vm[s] = float(np.abs(dec[blocks, 1, case.layer]).max()) if n else 0.0
    return vm


def _magnify(tens, case, kind):
    """Scale the cached K/V: 'huge' (x 2^20, block amax ~ 4e6 > 65504), 'tiny'
    (x 2^-24), or 'mixed' (sequence 0's first 64 tokens x 2^20, the rest x 2^-10,
    so a CTA meets blocks 2^30 apart)."""
    def f(x, seqs, pos):
        x = x.float()
        if kind == "huge":
            x = x * 2.0 ** 20
        elif kind == "tiny":
            x = x * 2.0 ** -24
        else:
            big = (seqs == 0) & (pos < 64)
            x = torch.where(big[:, None, None], x * 2.0 ** 20, x * 2.0 ** -10)
        return x.to(torch.bfloat16)
    B = case.batch
    new_pos = tens.new_pos.cpu()
    tens.k_tokens = f(tens.k_tokens, tens.tok_seq.cpu(), tens.tok_pos.cpu())
    tens.v_tokens = f(tens.v_tokens, tens.tok_seq.cpu(), tens.tok_pos.cpu())
    tens.k_new = f(tens.k_new, torch.arange(B), new_pos)
    tens.v_new = f(tens.v_new, torch.arange(B), new_pos)
    return tens


@pytest.mark.parametrize("kind", ["huge", "tiny", "mixed"])
@pytest.mark.parametrize("mode", ["auto", "split3", "simt", "mq3", "mq48", "cascade"])
def test_block_scales_far_from_one(kind, mode):
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case(f"bs_range_{kind}", [1500, 333, 64], 32, 8, 128, 16, "e4m3", "bf16",
                        "bf16", seed=310)
    tens = _magnify(wl.make_tensors(case), case, kind)
    pool, tables, lens, osc, opool = _block_pool(case, tens)
    q = tens.q.cuda()
    maxlen = int(case.seq_lens.max())
    vm = _vmax_blocks(case, opool, osc)
    seqs = list(range(case.batch))
    if mode in ("mq3", "mq48"):
        ql = 3 if mode == "mq3" else 48
        g = torch.Generator().manual_seed(ql)
        q2 = torch.randn(case.batch, ql, 32, 128, generator=g).bfloat16()
        ref, _ = oracle.decode_mq(np_raw(q2), "bf16", opool, "e4m3", case.geometry, case.layer,
                                  case.tables, case.seq_lens, ql, case.scale, block_scales=osc)
        out = torch.full((case.batch, ql, 32, 128), float("nan"), device="cuda")
        pkv.paged_decode_attention_mq(out, q2.cuda(), pool, case.layer, tables, lens, maxlen,
                                      case.scale)
    else:
        ref, _, _ = oracle.decode(np_raw(tens.q), "bf16", opool, "e4m3", case.geometry,
                                  case.layer, case.tables, case.seq_lens, case.scale,
                                  block_scales=osc)
        out = torch.full((case.batch, 32, 128), float("nan"), device="cuda")
        if mode == "cascade":
            kb = int(case.seq_lens[1]) // case.block_size
            ptab = torch.from_numpy(case.tables[1, :kb].copy()).cuda()
            plens = torch.zeros(case.batch, dtype=torch.int32, device="cuda")
            plens[1] = kb * case.block_size
            pkv.paged_decode_attention_cascade(out, q, pool, case.layer, ptab,
                                               kb * case.block_size, plens, tables, lens, maxlen,
                                               case.scale, opts=pkv.launch_opts(kernel=3))
        else:
            opts = pkv.launch_opts(kernel=1) if mode == "simt" else None
            pkv.paged_decode_attention(out, q, pool, case.layer, tables, lens, maxlen,
                                       case.scale, num_splits=3 if mode == "split3" else 0,
                                       opts=opts)
    torch.cuda.synchronize()
    assert pool.check_status() == 0
    _assert_close(out, ref, seqs, vm, TOL["e4m3"], f"{kind} {mode}")


# ------------------------------------------------------------------ a long tail of tiny weights
def _tail_case(q_len):
    """One sequence of 300,001 tokens, 4 query heads on 1 KV head, f16 pool, scale 1:
    q = e_0 for every query; key 0 has k[0] = 18 (weight 1), every other key
    k[0] = 0 (weight e^-18 ~ 2^-26 each, 0.46% of the total); V = e_0 except
    key 0's V = 0, so the output's first element is the tail's share."""
    n = 300_001
    case = wl.make_case("f16_tail", [n], 4, 1, 128, 16, "f16", "f16", "f16", seed=320)
    T = n - 1
    k = torch.zeros(T, 1, 128, dtype=torch.float16)
    v = torch.zeros(T, 1, 128, dtype=torch.float16)
    v[1:, 0, 0] = 1.0
    k[0, 0, 0] = 18.0
    k_new = torch.zeros(1, 1, 128, dtype=torch.float16)
    v_new = torch.zeros(1, 1, 128, dtype=torch.float16)
    v_new[0, 0, 0] = 1.0
    tens = wl.Tensors(k_tokens=k, v_tokens=v, tok_seq=torch.zeros(T, dtype=torch.int32),
                      tok_pos=torch.arange(T, dtype=torch.int32),
                      q=torch.zeros(1, 4, 128, dtype=torch.float16), k_new=k_new, v_new=v_new,
                      new_pos=torch.tensor([n - 1], dtype=torch.int32))
    tens.q[0, :, 0] = 1.0
    return case, tens


@pytest.mark.parametrize("q_len", [1, 32])
def test_long_tail_of_small_weights_is_kept(q_len):
    """q_len 1: the mma.sync decode kernel; q_len 32 (128 rows): tcgen05."""
    from paged_kv_cache_215_gb300 import pkv
    case, tens = _tail_case(q_len)
    gc = GpuCase(case, tens)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos)
    pool, _, seqs = oracle_side(case, tens, None)
    q = torch.zeros(1, q_len, 4, 128, dtype=torch.float16)
    q[..., 0] = 1.0
    ref, _ = oracle.decode_mq(np_raw(q), "f16", pool, "f16", case.geometry, case.layer,
                              case.tables, case.seq_lens, q_len, 1.0)
    assert ref[0, -1, 0, 0] > 4e-3                # the tail's share, well above the bound
    out = torch.full((1, q_len, 4, 128), float("nan"), device="cuda")
    pkv.paged_decode_attention_mq(out, q.cuda(), gc.pool, case.layer, gc.tables, gc.seq_lens,
                                  gc.max_seq_len, 1.0)
    torch.cuda.synchronize()
    assert gc.status() == 0
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert float(np.abs(got - ref).max()) <= TOL["f16"] * 1.0
