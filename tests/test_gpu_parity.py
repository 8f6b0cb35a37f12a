"""Parity of the CUDA path with the fp64 oracle (needs a GPU).

Every comparison runs the library through its C ABI (the ctypes binding) and
the oracle on the CPU on the same seeded inputs.  Bounds, written here:
  append / slot indexing / E4M3 encoding / amax: bit-exact
  attention: max |gpu - oracle| <= 2e-3 * max|V| (f32, f16, bf16 KV)
             max |gpu - oracle| <= 5e-3 * max|V| (E4M3 KV, oracle dequantising the same bytes)
  (plus half an ulp of the exact value when the output dtype is bf16 or f16)
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, assert_parity, oracle_side
from tests.helpers import fp8_scales, np_raw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_215_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def small_cases():
    return [
        wl.tiny_gqa2_d64_f32(),
        wl.llama8b_batch(batch=5, lo=100, hi=1500, seed=11),
        wl.make_case("llama8b_f16_b3", [700, 33, 1601], 32, 8, 128, 16, "f16", "f16", "f16",
                     seed=12),
        wl.long_context(tokens=20000, seed=13),
        wl.make_case("fp8_b3_h32-8_d128", [3000, 777, 1], 32, 8, 128, 16, "e4m3", "bf16",
                     "bf16", seed=14),
        wl.make_case("fp8_b2_h4-2_d64", [300, 123], 4, 2, 64, 16, "e4m3", "bf16", "bf16",
                     seed=15),
        wl.llama70b_prefix(batch=6, lo=512, hi=20000, block_size=16, seed=16),
        wl.llama70b_prefix(batch=6, lo=512, hi=20000, block_size=32, seed=17),
        wl.make_case("ragged_edges_bf16", [1, 16, 17, 31, 32, 33, 0, 2], 32, 8, 128, 16, "bf16",
                     "bf16", "bf16", seed=18),
        wl.make_case("ragged_edges_bs32_g8", [1, 32, 33, 64, 0, 95], 64, 8, 128, 32, "bf16",
                     "bf16", "bf16", seed=19),
        wl.make_case("bs64_bf16", [1, 63, 64, 65, 700, 2049], 32, 8, 128, 64, "bf16", "bf16",
                     "bf16", seed=40),
        wl.make_case("bs64_fp8", [64, 129, 1500], 32, 8, 128, 64, "e4m3", "bf16", "bf16",
                     seed=41),
        wl.make_case("fp8_bs32_g8", [31, 33, 900], 64, 8, 128, 32, "e4m3", "bf16", "bf16",
                     seed=42),
        wl.make_case("layers3_layer2_bf16", [40, 333, 1000], 32, 8, 128, 16, "bf16", "bf16",
                     "bf16", seed=43, num_layers=3, layer=2),
        wl.make_case("layers2_layer0_fp8_bs32", [77, 600], 32, 8, 128, 32, "e4m3", "bf16",
                     "bf16", seed=44, num_layers=2, layer=0),
    ]


CASES = small_cases()
_SIDE = {}


def _sides(case):
    """GPU case plus the oracle's pool and result, computed once per case."""
    if case.name not in _SIDE:
        tens = wl.make_tensors(case)                           # CPU draw, shared by both sides
        gc = GpuCase(case, tens)
        pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
        _SIDE[case.name] = (gc, pool, ref, seqs)
    return _SIDE[case.name]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_append_is_bit_exact(case):
    gc, pool, _, _ = _sides(case)
    gc.step()                                                  # appends every last token
    torch.cuda.synchronize()
    got = gc.pool.storage.cpu().numpy()
    assert np.array_equal(got, pool), "pool bytes differ from the oracle's"
    assert gc.status() == 0


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fp8_scales_match_oracle(case):
    """The library's per-tensor scales (kv_absmax of the cached and the new tokens,
    then kv_fp8_scale) equal the oracle's absmax and scale rule bit for bit."""
    if case.kv_dtype != "e4m3":
        pytest.skip("per-tensor scales exist only for E4M3 pools")
    gc, _, _, _ = _sides(case)
    ks, vs = fp8_scales(gc.tens)
    assert (gc.k_scale, gc.v_scale) == (ks, vs)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_fp8_scale_matches_oracle_on_awkward_tensors(dt):
    """kv_absmax + kv_fp8_scale against oracle.absmax + oracle.fp8_scale, bit for
    bit, on tensors held in three pieces with NaN, +-Inf, -0, subnormals and a
    negative maximum planted, on magnitudes from 2^-20 to 2^20, and on all-zero
    and all-non-finite tensors (scale 1)."""
    from paged_kv_cache_215_gb300 import pkv
    name = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dt]
    g = torch.Generator().manual_seed(7)
    exps = [-20, -3, 0, 9, 20] if dt != torch.float16 else [-10, -3, 0, 4, 9]
    for e in exps:
        parts = [(torch.randn(n, generator=g) * 2.0 ** e).to(dt) for n in (4097, 1, 333)]
        parts[0][5] = float("nan")
        parts[0][6] = float("inf")
        parts[2][7] = float("-inf")
        parts[2][8] = -0.0
        parts[2][9] = torch.finfo(dt).tiny / 4
        parts[1][0] = -float(parts[0].float().nan_to_num(0, 0, 0).abs().max()) * 1.5
        amax = torch.zeros(3, dtype=torch.float32, device="cuda")
        for i, x in enumerate(parts):
            pkv.kv_absmax(x.cuda(), amax[i:i + 1])
        sc = torch.zeros(1, dtype=torch.float32, device="cuda")
        pkv.kv_fp8_scale(amax, sc)
        want_amax = max(oracle.absmax(np_raw(x), name) for x in parts)
        assert amax.cpu().tolist() == [oracle.absmax(np_raw(x), name) for x in parts]
        assert float(sc.item()) == oracle.fp8_scale(want_amax), (e, float(sc.item()))
    for x in (torch.zeros(100, dtype=dt),
              torch.tensor([float("nan"), float("inf"), -float("inf")] * 10).to(dt)):
        amax = torch.zeros(1, dtype=torch.float32, device="cuda")
        pkv.kv_absmax(x.cuda(), amax)
        sc = torch.zeros(1, dtype=torch.float32, device="cuda")
        pkv.kv_fp8_scale(amax, sc)
        assert float(amax.item()) == 0.0 and float(sc.item()) == 1.0


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("kernel", [0, 1, 2])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_decode_parity(case, kernel, splits):
    from paged_kv_cache_215_gb300 import pkv
    gc, pool, ref, seqs = _sides(case)
    opts = pkv.launch_opts(kernel=kernel) if kernel else None
    try:
        out = gc.step(num_splits=splits, opts=opts)
    except pkv.PkvError as e:
        if e.code == pkv.PKV_EUNSUPPORTED:
            pytest.skip("kernel does not take this shape")
        raise
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} k{kernel} s{splits}")


# (KV heads per CTA, CTAs per SM) away from the default plan: the widest CTA
# (8 consumer warps), one head per CTA, and shapes that change the stage count
# and the balanced partition's run lengths.
LAUNCH_SHAPES = [(8, 1), (1, 6), (2, 4), (4, 1), (2, 2)]


@pytest.mark.parametrize("shape", LAUNCH_SHAPES, ids=lambda s: f"hg{s[0]}c{s[1]}")
@pytest.mark.parametrize("case", [c for c in CASES if c.kv_dtype != "f32"], ids=lambda c: c.name)
def test_decode_parity_launch_shapes(case, shape):
    from paged_kv_cache_215_gb300 import pkv
    gc, pool, ref, seqs = _sides(case)
    hg, ctas = shape
    if case.num_kv_heads % hg:
        pytest.skip("head group does not divide the KV heads")
    opts = pkv.launch_opts(kernel=2, kv_heads_per_cta=hg, ctas_per_sm=ctas)
    try:
        out = gc.step(opts=opts)
    except pkv.PkvError as e:
        if e.code == pkv.PKV_EUNSUPPORTED:
            pytest.skip("kernel does not take this shape")
        raise
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} hg{hg} c{ctas}")
    assert torch.equal(out, gc.step(opts=opts))                 # deterministic


@pytest.mark.parametrize("case", [c for c in CASES if c.kv_dtype != "f32"], ids=lambda c: c.name)
def test_decode_parity_low_precision_out(case):
    gc, pool, ref, seqs = _sides(case)
    out = gc.step(out_dtype=case.out_dtype)
    torch.cuda.synchronize()
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, case.name, out_dtype=case.out_dtype)


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fused_decode_step_matches_append_then_attend(case, kernel, splits):
    """paged_decode_step stores the new tokens itself; its pool must equal the
    oracle's and its output must match the oracle like the two-call path."""
    from paged_kv_cache_215_gb300 import pkv
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)                                    # new tokens not yet stored
    _, pool, ref, seqs = _sides(case)
    opts = pkv.launch_opts(kernel=kernel) if kernel else None
    try:
        out = gc.fused_step(num_splits=splits, opts=opts)
    except pkv.PkvError as e:
        if e.code == pkv.PKV_EUNSUPPORTED:
            pytest.skip("kernel does not take this shape")
        raise
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert np.array_equal(gc.pool.storage.cpu().numpy(), pool), "pool bytes differ"
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} fused k{kernel} s{splits}")
    two_call = gc.step(num_splits=splits, opts=opts)             # same pool, same inputs
    assert torch.equal(out, two_call)


def test_programmatic_dependent_launch_keeps_results():
    from paged_kv_cache_215_gb300 import pkv
    case = wl.llama8b_batch(batch=5, lo=100, hi=1500, seed=11)
    gc, pool, ref, seqs = _sides(case)
    plain = gc.fused_step()
    outs = [gc.fused_step(opts=pkv.launch_opts(pdl=1)) for _ in range(3)]   # back to back
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, plain)


def test_zero_length_sequence_gives_zero_and_single_token_gives_v():
    case = [c for c in CASES if c.name == "ragged_edges_bf16"][0]
    gc, pool, ref, seqs = _sides(case)
    out = gc.step().double().cpu()
    s0 = list(case.seq_lens).index(0)
    assert torch.all(out[s0] == 0)
    s1 = list(case.seq_lens).index(1)
    v = gc.v_new.double().cpu()[s1]                            # the only token
    G = case.num_q_heads // case.num_kv_heads
    for h in range(case.num_q_heads):
        assert torch.equal(out[s1, h], v[h // G])


def test_results_do_not_depend_on_physical_block_ids():
    base = wl.llama8b_batch(batch=4, lo=200, hi=900, seed=21)
    tens = wl.make_tensors(base)
    outs = []
    for seed in (1, 2):
        c = wl.llama8b_batch(batch=4, lo=200, hi=900, seed=21)
        perm = np.random.default_rng(seed).permutation(c.num_blocks).astype(np.int32)
        c.tables, _, _ = wl._build_tables(c.seq_lens, 16, c.num_blocks, perm)
        outs.append(GpuCase(c, tens).step().cpu())
    assert torch.equal(outs[0], outs[1])


def test_garbage_in_unused_slots_is_ignored():
    case = wl.make_case("nan_fill", [37, 100, 5], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=22)
    tens = wl.make_tensors(case)
    clean = GpuCase(case, tens, fill_byte=0).step()
    dirty = GpuCase(case, tens, fill_byte=0xFF).step()          # 0xFFFF is a bf16 NaN
    assert torch.equal(clean, dirty)
    case8 = wl.make_case("nan_fill8", [37, 100], 32, 8, 128, 16, "e4m3", "bf16", "bf16", seed=23)
    tens8 = wl.make_tensors(case8)
    assert torch.equal(GpuCase(case8, tens8, fill_byte=0).step(),
                       GpuCase(case8, tens8, fill_byte=0xFF).step())   # 0xFF is an E4M3 NaN


def test_out_of_range_block_id_is_reported_not_faulted():
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("bad_id", [40, 20], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=24)
    gc = GpuCase(case)
    bad = gc.tables.clone()
    bad[0, 1] = case.num_blocks + 7
    out = torch.empty(2, 32, 128, dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention(out, gc.q, gc.pool, 0, bad, gc.seq_lens, 40, case.scale)
    assert gc.status() == pkv.PKV_EBOUNDS
    assert gc.status() == 0                                     # cleared by the read
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("scale", [1.0, 4.75 / 448, 0.02, 3.0])
def test_fp8_encode_exhaustive_over_bf16(scale):
    from paged_kv_cache_215_gb300 import pkv
    # every bf16 bit pattern as one element of a token's k and v
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16).reshape(-1, 1, 128)        # 512 tokens x 1 head x 128
    n = vals.shape[0]
    case = wl.make_case("enc", [n + 1], 1, 1, 128, 16, "e4m3", "bf16", "bf16", seed=25)
    g = pkv.geometry(1, 1, 1, 128, 16, case.num_blocks, "e4m3")
    pool = pkv.KVPool(g)
    pool.storage.zero_()
    pool.reserve(sorted(set(case.tables[0][case.tables[0] >= 0].tolist())))
    tab = torch.from_numpy(case.tables).cuda()
    seq = torch.zeros(n, dtype=torch.int32, device="cuda")
    pos = torch.arange(n, dtype=torch.int32, device="cuda")
    k = vals.cuda().contiguous()
    pool.append_tokens(0, k, k, tab, seq, pos, scale, scale)
    torch.cuda.synchronize()
    want = np.zeros(pool.nbytes, np.uint8)
    oracle.append_tokens(want, "e4m3", case.geometry, 0, np_raw(vals), np_raw(vals), "bf16",
                         case.tables, np.zeros(n, np.int32), np.arange(n, dtype=np.int32),
                         scale, scale)
    assert np.array_equal(pool.storage.cpu().numpy(), want)


def test_fp8_encode_special_f32_inputs():
    from paged_kv_cache_215_gb300 import pkv
    specials = [0.0, -0.0, float("inf"), float("-inf"), float("nan"), 448.0, 464.0, 465.0,
                -1e30, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875, 1e-45, -1e-40]
    x = torch.tensor((specials * 8)[:128], dtype=torch.float32).reshape(1, 1, 128)
    case = wl.make_case("enc32", [2], 1, 1, 128, 16, "e4m3", "f32", "f32", seed=26)
    g = pkv.geometry(1, 1, 1, 128, 16, case.num_blocks, "e4m3")
    pool = pkv.KVPool(g)
    pool.storage.zero_()
    pool.reserve([int(case.tables[0, 0])])
    tab = torch.from_numpy(case.tables).cuda()
    pool.append(0, x.cuda(), x.cuda(), tab, torch.zeros(1, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    want = np.zeros(pool.nbytes, np.uint8)
    oracle.append(want, "e4m3", case.geometry, 0, x.numpy(), x.numpy(), "f32", case.tables,
                  np.zeros(1, np.int32))
    assert np.array_equal(pool.storage.cpu().numpy(), want)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_absmax_matches_oracle(dt):
    from paged_kv_cache_215_gb300 import pkv
    x = (torch.randn(1 << 20, generator=torch.Generator().manual_seed(3)) * 7).to(dt)
    x[12345] = float("nan")
    x[2345] = float("inf")
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    pkv.kv_absmax(x.cuda(), out)
    name = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dt]
    assert float(out.item()) == oracle.absmax(np_raw(x), name)


@pytest.mark.parametrize("S", [1, 2, 7, 40])
def test_merge_partials_matches_oracle(S):
    from paged_kv_cache_215_gb300 import pkv
    B, H, D = 3, 8, 128
    g = torch.Generator().manual_seed(S)
    po = torch.randn(B, H, S, D, generator=g)
    pl = torch.randn(B, H, S, generator=g) * 5
    pl[0, 0, 0] = -math.inf                                     # an empty partition
    pl[1, 2, :] = -math.inf                                     # a row with no tokens
    out = torch.empty(B, H, D, device="cuda")
    pkv.merge_partials(out, po.cuda(), pl.cuda())
    ref, _ = oracle.merge(po.double().numpy().reshape(B * H, S, D),
                          pl.double().numpy().reshape(B * H, S))
    got = out.double().cpu().numpy().reshape(B * H, D)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)
    assert np.all(got[1 * H + 2] == 0)


def test_copy_on_write_keeps_other_sequence_unchanged():
    """Two sequences share their first block; appending into it for one of them
    copies the block first (the pages' copy-on-write prefix sharing)."""
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("cow", [10, 10], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=27)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    gc.step()                                                   # every token in place
    # make sequence 1 share sequence 0's (partial) first block
    shared = int(case.tables[0, 0])
    old1 = int(case.tables[1, 0])
    gc.pool.free([old1])
    gc.pool.share([shared])
    gc.tables[1, 0] = shared
    case.tables[1, 0] = shared
    assert gc.pool.refcount(shared) == 2
    before = gc.step(append=False).clone()                      # both read the same block
    new = gc.pool.cow(shared)
    assert new != shared and gc.pool.refcount(shared) == 1 and gc.pool.refcount(new) == 1
    v = gc.pool.view()
    torch.cuda.synchronize()
    assert torch.equal(v[new], v[shared])                       # copied bytes
    gc.tables[1, 0] = new
    # overwrite the last token of sequence 1 with new values: sequence 0 must not change
    gc.k_new[1] = torch.randn_like(gc.k_new[1].float()).to(gc.k_new.dtype)
    out = gc.step()
    assert torch.equal(out[0], before[0])
    assert not torch.equal(out[1], before[1])


def test_launch_counter_counts_kernels():
    from paged_kv_cache_215_gb300 import pkv
    gc, _, _, _ = _sides(CASES[1])
    n0 = pkv.launch_count()
    gc.step()
    torch.cuda.synchronize()
    assert pkv.launch_count() - n0 == 3                         # append, attention, merge


@pytest.mark.parametrize("kv,bs", [("bf16", 16), ("f16", 32), ("e4m3", 16), ("bf16", 32)])
def test_decode_sixteen_query_heads_per_kv_head(kv, bs):
    """Single-token decode with G = 16 (128 query / 8 KV heads, and 16 / 1): the
    tensor-core kernel holds the 16 query rows of a KV head as two n-tiles
    (the mhpn.cn long-context article, section 3.2 grouping), against the oracle."""
    from paged_kv_cache_215_gb300 import pkv
    for hq, hkv, lens in ((128, 8, [1, 17, 700, 2100]), (16, 1, [33, 1500])):
        q = "f16" if kv == "f16" else "bf16"
        case = wl.make_case(f"g16_{kv}_bs{bs}_{hq}", lens, hq, hkv, 128, bs, kv, q, "f32",
                            seed=150 + bs + hq, spike_frac=0.01)
        tens = wl.make_tensors(case)
        gc = GpuCase(case, tens)
        pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
        for splits in (0, 3):
            out = gc.step(num_splits=splits, opts=pkv.launch_opts(kernel=2))
            torch.cuda.synchronize()
            assert gc.status() == 0
            assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} splits {splits}")
        # the decode step with the new token's store fused into the attention launch
        out = gc.fused_step()
        torch.cuda.synchronize()
        assert gc.status() == 0
        assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} fused step")


@pytest.mark.parametrize("stages", [2, 3, 5])
@pytest.mark.parametrize("name", ["llama8b_f16_b3", "fp8_b3_h32-8_d128", "ragged_edges_bf16"])
def test_decode_parity_ring_depths(name, stages):
    """An explicit ring depth (opts.stages) on the tensor-core decode kernel: the
    producer/consumer barrier phases wrap at every depth; a depth the shared
    memory cannot hold is refused with PKV_EUNSUPPORTED."""
    from paged_kv_cache_215_gb300 import pkv
    case = next(c for c in CASES if c.name == name)
    gc, pool, ref, seqs = _sides(case)
    opts = pkv.launch_opts(kernel=2, stages=stages)
    try:
        out = gc.step(opts=opts)
    except pkv.PkvError as e:
        if e.code == pkv.PKV_EUNSUPPORTED:
            pytest.skip("the ring does not fit at this depth")
        raise
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} stages {stages}")
