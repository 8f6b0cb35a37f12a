"""Block-wise E4M3 scales (needs a GPU): one fp32 scale per scale group of a
sequence's positions, K/V, layer and KV head, stored in each of the group's
blocks -- one block, or the pages' 64 and 128 tokens ("Unlocking long context"
section 3.2).  Scales and pool bytes are bit-exact with the oracle; decode
results match the oracle (dequantising the same bytes with the same scales)
within 5e-3 x max|V|."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import TOL, vmax_per_seq
from tests.helpers import np_raw

pytestmark = pytest.mark.gpu


def _setup(case, group=0):
    from paged_kv_cache_215_gb300 import pkv
    tens = wl.make_tensors(case)
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
    scales = torch.full((case.num_blocks, 2, case.num_layers, case.num_kv_heads), 7.0,
                        dtype=torch.float32, device=dev)
    pool.set_block_scales(scales)
    tables = torch.from_numpy(case.tables).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    seq = torch.cat([tens.tok_seq, torch.arange(case.batch, dtype=torch.int32)]).to(dev)
    pos = torch.cat([tens.tok_pos, tens.new_pos]).to(dev)
    k_all = torch.cat([tens.k_tokens, tens.k_new]).to(dev)
    v_all = torch.cat([tens.v_tokens, tens.v_new]).to(dev)
    pool.compute_block_scales(case.layer, k_all, v_all, tables, seq, pos, group_tokens=group)
    pool.append_tokens(case.layer, tens.k_tokens.to(dev), tens.v_tokens.to(dev), tables,
                       tens.tok_seq.to(dev), tens.tok_pos.to(dev))
    # oracle side
    osc = np.full(tuple(scales.shape), 7.0, np.float32)
    oracle.block_scales(osc, case.geometry, case.layer, np_raw(k_all), np_raw(v_all), "bf16",
                        case.tables, np_raw(seq), np_raw(pos), group)
    opool = np.zeros(pool.nbytes, np.uint8)
    oracle.append_tokens(opool, "e4m3", case.geometry, case.layer, np_raw(k_all), np_raw(v_all),
                         "bf16", case.tables, np_raw(seq), np_raw(pos), block_scales=osc)
    return tens, pool, scales, tables, lens, osc, opool


CASES = [
    wl.make_case("bs64_blockscale", [700, 130, 2000, 1], 32, 8, 128, 64, "e4m3", "bf16", "bf16",
                 seed=90, spike_frac=0.01),
    wl.make_case("bs16_blockscale_g8", [333, 64, 17], 64, 8, 128, 16, "e4m3", "bf16", "bf16",
                 seed=91),
    wl.make_case("bs32_blockscale_layers2", [90, 600], 32, 8, 128, 32, "e4m3", "bf16", "bf16",
                 seed=92, num_layers=2, layer=1),
]


GROUPS = [0, 64, 128]


@pytest.mark.parametrize("group", GROUPS, ids=lambda g: f"group{g}")
@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_block_scales_and_pool_bit_exact(case, group):
    tens, pool, scales, tables, lens, osc, opool = _setup(case, group)
    pool.append(case.layer, tens.k_new.cuda(), tens.v_new.cuda(), tables, tens.new_pos.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(pool.storage.cpu().numpy(), opool)
    assert pool.check_status() == 0


@pytest.mark.parametrize("group", GROUPS, ids=lambda g: f"group{g}")
@pytest.mark.parametrize("mode", ["auto", "simt", "split3", "fused", "mq2", "mq40", "cascade"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_block_scaled_decode_parity(case, mode, group):
    from paged_kv_cache_215_gb300 import pkv
    tens, pool, scales, tables, lens, osc, opool = _setup(case, group)
    q = tens.q.cuda()
    maxlen = int(case.seq_lens.max())
    if mode in ("mq2", "mq40"):
        # 2 tokens: the mma.sync kernel; 40 tokens (160+ rows per KV head): the
        # tcgen05 kernel, converting each E4M3 tile with its block's scale
        ql = 2 if mode == "mq2" else 40
        pool.append(case.layer, tens.k_new.cuda(), tens.v_new.cuda(), tables, tens.new_pos.cuda())
        g = torch.Generator().manual_seed(3)
        q2 = torch.randn(case.batch, ql, case.num_q_heads, case.head_dim, generator=g).bfloat16()
        ref, _ = oracle.decode_mq(np_raw(q2), "bf16", opool, "e4m3", case.geometry, case.layer,
                                  case.tables, case.seq_lens, ql, case.scale, block_scales=osc)
        out = torch.full((case.batch, ql, case.num_q_heads, case.head_dim), float("nan"),
                         device="cuda")
        pkv.paged_decode_attention_mq(out, q2.cuda(), pool, case.layer, tables, lens, maxlen,
                                      case.scale)
    else:
        ref, _, _ = oracle.decode(np_raw(tens.q), "bf16", opool, "e4m3", case.geometry,
                                  case.layer, case.tables, case.seq_lens, case.scale,
                                  block_scales=osc)
        out = torch.full((case.batch, case.num_q_heads, case.head_dim), float("nan"),
                         device="cuda")
        if mode == "fused":
            pkv.paged_decode_step(out, q, tens.k_new.cuda(), tens.v_new.cuda(), pool, case.layer,
                                  tables, lens, maxlen, case.scale)
        elif mode == "cascade":
            # sequence 0's full blocks as a "shared" prefix that only it uses, on the
            # forced prefix pass (tcgen05, each tile scaled by its block's scales)
            pool.append(case.layer, tens.k_new.cuda(), tens.v_new.cuda(), tables,
                        tens.new_pos.cuda())
            kb = int(case.seq_lens[0]) // case.block_size
            ptab = torch.from_numpy(case.tables[0, :max(kb, 1)].copy()).cuda()
            plens = torch.zeros(case.batch, dtype=torch.int32, device="cuda")
            plens[0] = kb * case.block_size
            pkv.paged_decode_attention_cascade(out, q, pool, case.layer, ptab,
                                               kb * case.block_size, plens, tables, lens, maxlen,
                                               case.scale, opts=pkv.launch_opts(kernel=3))
        else:
            pool.append(case.layer, tens.k_new.cuda(), tens.v_new.cuda(), tables,
                        tens.new_pos.cuda())
            opts = pkv.launch_opts(kernel=1) if mode == "simt" else None
            pkv.paged_decode_attention(out, q, pool, case.layer, tables, lens, maxlen,
                                       case.scale, num_splits=3 if mode == "split3" else 0,
                                       opts=opts)
    torch.cuda.synchronize()
    assert pool.check_status() == 0
    assert np.array_equal(pool.storage.cpu().numpy(), opool)      # the new tokens too
    vm = vmax_per_seq(case, opool, list(range(case.batch)), 1.0) if False else None
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    dec = torch.from_numpy(opool).view(torch.float8_e4m3fn).double().numpy().reshape(
        case.num_blocks, 2, case.num_layers, case.num_kv_heads, case.block_size,
        case.head_dim) * osc[:, :, :, :, None, None]
    for s in range(case.batch):
        n = int(case.seq_lens[s])
        blocks = case.tables[s, :(n + case.block_size - 1) // case.block_size]
        vmax = np.abs(dec[blocks, 1, case.layer]).max()
        err = np.abs(got[s] - ref[s]).max()
        assert err <= TOL["e4m3"] * vmax, f"{case.name} {mode} seq {s}: {err}"


@pytest.mark.parametrize("group", [64, 128])
def test_every_block_of_a_group_holds_its_scale(group):
    """A 64- or 128-token group at block size 16 spans 4 or 8 scattered blocks:
    every one of them holds the group's scale (read back from the device)."""
    case = CASES[1]                                          # block size 16
    tens, pool, scales, tables, lens, osc, opool = _setup(case, group)
    got = scales.cpu().numpy()
    per = group // case.block_size
    for s in range(case.batch):
        nb = (int(case.seq_lens[s]) + case.block_size - 1) // case.block_size
        for e0 in range(0, nb, per):
            blocks = case.tables[s, e0:min(e0 + per, nb)]
            assert np.all(got[blocks] == got[blocks[0]]), (s, e0)
