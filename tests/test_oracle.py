"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: values the
pages print, the OCP FP8 definition and a library decoder, closed forms and
special cases of softmax attention, a library (numpy/scipy) naive attention on
unpaged arrays, invariants (block-id permutation, split + merge), and a set of
planted mistakes that must each fail at least one pin.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.helpers import fp8_scales, logical_kv, np_raw, oracle_pool

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.strip() for l in f if l.strip() and not l.startswith("#")]


# --------------------------------------------------------------------------- KV size
def test_kv_size_matches_pages_worked_examples():
    for line in _lines("kv_size_examples.txt"):
        nums = line.split("|")[0].split()
        L, H, D, T, eb, want = (int(x) for x in nums)
        assert oracle.kv_bytes(L, H, D, T, eb) == want, line


def test_kv_size_printed_approximations():
    # the pages print these rounded: 2.5 MB, 640 GB, 16 GB, 512 MB (binary units)
    assert oracle.kv_bytes(80, 64, 128, 1, 2) / 2**20 == 2.5
    assert oracle.kv_bytes(80, 64, 128, 256 * 1024, 2) / 2**30 == 640
    assert oracle.kv_bytes(32, 32, 128, 32768, 2) / 2**30 == 16
    assert oracle.kv_bytes(1, 32, 128, 32768, 2) / 2**20 == 512


# --------------------------------------------------------------------------- E4M3
def test_e4m3_decode_spec_points():
    for line in _lines("e4m3_spec_values.txt"):
        code, val = line.split()
        got = oracle.e4m3_decode(np.array([int(code, 16)], np.uint8))[0]
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_decode_matches_library_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(lib)
    assert np.array_equal(ours[~both_nan], lib[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(lib))


def _nearest_code_bruteforce(y):
    """Reference encoder by exhaustive search over the 254 finite codes:
    nearest value, ties to the code with even mantissa, |y| > 448 saturates."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    out = np.empty(y.shape, np.uint8)
    for i, v in enumerate(y.astype(np.float64)):
        if math.isnan(v):
            out[i] = 0x7F
            continue
        neg = math.copysign(1.0, v) < 0
        a = abs(v)
        if a > 448:
            out[i] = 0xFE if neg else 0x7E
            continue
        pos_codes = codes[codes < 0x80]
        pos_vals = vals[codes < 0x80]
        d = np.abs(pos_vals - a)
        best = d.min()
        cand = pos_codes[d == best]
        c = cand[0] if len(cand) == 1 else [x for x in cand if x % 2 == 0][0]
        out[i] = (c | 0x80) if neg else c
    return out


@pytest.mark.parametrize("scale", [1.0, 0.5, 4.75 / 448, 3.0, 1e-3])
def test_e4m3_encode_exhaustive_over_bf16(scale):
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    got = oracle.e4m3_encode(x, scale)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        y = (x / np.float32(scale)).astype(np.float32)     # IEEE fp32 division
    want = _nearest_code_bruteforce(y)
    assert np.array_equal(got, want)
    # in range, the library's round-to-nearest-even conversion agrees
    finite = np.isfinite(y) & (np.abs(y) <= 448)
    lib = torch.from_numpy(y[finite]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[finite], lib)


def test_e4m3_encode_special_cases():
    enc = lambda v, s=1.0: int(oracle.e4m3_encode(np.array([v], np.float32), s)[0])
    assert enc(np.inf) == 0x7E and enc(-np.inf) == 0xFE
    assert enc(np.nan) == 0x7F
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert enc(464.0) == 0x7E and enc(1e30) == 0x7E and enc(-500.0) == 0xFE
    assert enc(2.0 ** -9) == 0x01
    assert enc(2.0 ** -10) == 0x00          # tie between 0 and 2^-9: even code 0
    assert enc(3 * 2.0 ** -10) == 0x02      # tie between 2^-9 and 2^-8: even code 2
    assert enc(1.0625) == 0x38              # tie between 1 and 1.125: even mantissa
    assert enc(1.1875) == 0x3A              # tie between 1.125 and 1.25: even mantissa
    assert enc(896.0, 2.0) == 0x7E          # x / scale = 448


# --------------------------------------------------------------------------- per-tensor scale
def _specials_array(dt, seed):
    """Random values of a dtype with the awkward ones planted: NaN, +-Inf, -0,
    subnormals of the dtype, and a largest magnitude that is negative."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(4099, generator=g, dtype=torch.float32) * 3.0
    x = x.to(dt)
    tiny = torch.finfo(dt).tiny                   # smallest normal: halve it for a subnormal
    plant = [float("nan"), float("inf"), float("-inf"), -0.0, tiny / 2, -tiny / 4, -37.25]
    for i, v in enumerate(plant):
        x[97 * (i + 1)] = v
    return x


@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
def test_absmax_is_the_largest_finite_magnitude(dt):
    """The per-tensor FP8 scale starts from the tensor's absolute maximum
    ("Unlocking long context" section 3.2).  Checked against numpy on the values
    torch decodes: NaN and +-Inf are left out, -0 and subnormals are ordinary
    values, and a negative element can hold the maximum magnitude."""
    name = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[dt]
    x = _specials_array(dt, seed=41)
    vals = x.to(torch.float64).numpy()
    want = float(np.abs(vals[np.isfinite(vals)]).max())
    assert want == 37.25                          # the planted negative maximum
    assert oracle.absmax(np_raw(x), name) == want
    # only non-finite values, only zeros, and the empty tensor: 0
    bad = torch.tensor([float("nan"), float("inf"), float("-inf")], dtype=torch.float32).to(dt)
    assert oracle.absmax(np_raw(bad), name) == 0.0
    assert oracle.absmax(np_raw(torch.tensor([0.0, -0.0]).to(dt)), name) == 0.0
    assert oracle.absmax(np_raw(torch.zeros(0, dtype=dt)), name) == 0.0
    # a lone subnormal is the maximum
    sub = torch.tensor([0.0, torch.finfo(dt).tiny / 8]).to(dt)
    assert oracle.absmax(np_raw(sub), name) == float(sub[1].double())


def test_fp8_scale_closed_forms():
    """scale = amax / 448 in fp32 ("Unlocking long context" section 3.2; 448 is the
    largest finite E4M3 value): exact values where the quotient is a power of
    two, exact scaling by powers of two, and 1 for an all-zero tensor."""
    assert oracle.fp8_scale(0.0) == 1.0
    assert oracle.fp8_scale(448.0) == 1.0
    assert oracle.fp8_scale(896.0) == 2.0
    assert oracle.fp8_scale(3.5) == 2.0 ** -7
    assert oracle.fp8_scale(7.0 * 2.0 ** -20) == 2.0 ** -26
    for k in range(-30, 31):
        assert oracle.fp8_scale(37.25 * 2.0 ** k) == oracle.fp8_scale(37.25) * 2.0 ** k


def test_fp8_scale_stores_the_largest_value_as_448():
    """With the scale, the tensor's largest magnitude encodes to the largest E4M3
    code (0x7E, or 0xFE for a negative value) and nothing saturates beyond it;
    the scale is the correctly rounded quotient (within half an fp32 ulp)."""
    rng = np.random.default_rng(5)
    amax = np.concatenate([rng.lognormal(0.0, 6.0, 2000), [1e-30, 3e-5, 65504.0, 3e38]])
    amax = amax.astype(np.float32)
    for a in amax:
        sc = oracle.fp8_scale(float(a))
        assert int(oracle.e4m3_encode(np.array([a], np.float32), sc)[0]) == 0x7E
        assert int(oracle.e4m3_encode(np.array([-a], np.float32), sc)[0]) == 0xFE
        exact = float(a) / 448.0
        assert abs(sc - exact) <= 0.5 * np.spacing(np.float32(exact)) * (1 + 1e-12)


# --------------------------------------------------------------------------- attention
def _naive(q, K, V, scale):
    """Library naive attention on unpaged arrays: softmax(q K^T * scale) V, the
    definition printed in "Unlocking long context" section 4.1."""
    w = softmax(scale * (K @ q))
    return w @ V, w


def _naive_case(case, tens, kv_f64=None, k_scale=1.0, v_scale=1.0):
    G = case.num_q_heads // case.num_kv_heads
    q = tens.q.double().cpu().numpy()
    out = np.zeros((case.batch, case.num_q_heads, case.head_dim))
    for s, (K, V) in enumerate(kv_f64 or logical_kv(case, tens)):
        for h in range(case.num_q_heads):
            hk = h // G
            out[s, h], _ = _naive(q[s, h], K[:, hk] * k_scale, V[:, hk] * v_scale, case.scale)
    return out


def _small_cases():
    return [
        wl.tiny_gqa2_d64_f32(),
        wl.make_case("mha_bf16", [1, 17, 50], 3, 3, 32, 16, "bf16", "bf16", "bf16", seed=5),
        wl.make_case("gqa4_f16_bs32", [33, 64, 70], 8, 2, 16, 32, "f16", "f16", "f16", seed=6),
        wl.make_case("gqa8_bf16_prefix", [20, 70, 40], 16, 2, 16, 16, "bf16", "bf16", "bf16",
                     seed=7, shared_prefix_tokens=32),
        wl.make_case("layers3_layer1_bs64", [5, 64, 130], 4, 2, 16, 64, "bf16", "bf16", "bf16",
                     seed=8, num_layers=3, layer=1),
    ]


def _run_oracle(case, tens, pool, k_scale=1.0, v_scale=1.0, **kw):
    return oracle.decode(np_raw(tens.q), case.q_dtype, pool, case.kv_dtype, case.geometry,
                         case.layer, case.tables, case.seq_lens, case.scale, k_scale, v_scale,
                         **kw)


@pytest.mark.parametrize("case", _small_cases(), ids=lambda c: c.name)
def test_paged_equals_unpaged_naive_attention(case):
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    out, lse, wsum = _run_oracle(case, tens, pool)
    ref = _naive_case(case, tens)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(wsum, 1.0, rtol=0, atol=1e-14)


def test_fp8_paged_equals_naive_on_dequantised_values():
    case = wl.fp8_batch(batch=2, tokens=300, heads=(4, 2, 64), seed=11)
    case.seq_lens = np.array([300, 123], np.int32)
    tens = wl.make_tensors(case)
    ks, vs = fp8_scales(tens)
    pool = oracle_pool(case, tens, ks, vs, include_new=True)
    out, _, _ = _run_oracle(case, tens, pool, ks, vs)
    # dequantise with the library's decoder, through the generator's own values
    kv = []
    for K, V in logical_kv(case, tens):
        Kq = oracle.e4m3_encode(K.astype(np.float32), ks)
        Vq = oracle.e4m3_encode(V.astype(np.float32), vs)
        dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
        kv.append((dec(Kq), dec(Vq)))
    ref = _naive_case(case, tens, kv, ks, vs)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_block_id_permutation_invariance():
    base = wl.make_case("perm", [45, 9, 160], 4, 2, 32, 16, "bf16", "bf16", "bf16", seed=21)
    tens = wl.make_tensors(base)
    outs = []
    for seed in (1, 2, 3):
        c = wl.make_case("perm", base.seq_lens, 4, 2, 32, 16, "bf16", "bf16", "bf16", seed=21)
        rng = np.random.default_rng(seed)
        perm = rng.permutation(c.num_blocks).astype(np.int32)
        c.tables, _, _ = wl._build_tables(c.seq_lens, 16, c.num_blocks, perm)
        pool = oracle_pool(c, tens, include_new=True)
        outs.append(_run_oracle(c, tens, pool)[0])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_single_token_returns_v0_exactly():
    case = wl.make_case("one", [1, 1], 4, 2, 64, 16, "f32", "f32", "f32", seed=31)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    out, _, wsum = _run_oracle(case, tens, pool)
    v = tens.v_new.double().numpy()
    for h in range(4):
        assert np.array_equal(out[:, h], v[:, h // 2])
    assert np.array_equal(wsum, np.ones_like(wsum))


def test_identical_v_rows_return_that_row():
    case = wl.make_case("samev", [77, 130], 4, 2, 32, 16, "f32", "f32", "f32", seed=41)
    tens = wl.make_tensors(case)
    row = torch.randn(2, 32, generator=torch.Generator().manual_seed(3))
    tens.v_tokens[:] = row
    tens.v_new[:] = row
    pool = oracle_pool(case, tens, include_new=True)
    out, _, _ = _run_oracle(case, tens, pool)
    want = np.broadcast_to(row.double().numpy()[None, [0, 0, 1, 1]], out.shape)
    np.testing.assert_allclose(out, want, rtol=1e-14, atol=1e-15)


def test_zero_query_gives_mean_of_v():
    case = wl.make_case("q0", [50, 3], 4, 2, 32, 16, "f32", "f32", "f32", seed=51)
    tens = wl.make_tensors(case)
    tens.q.zero_()
    pool = oracle_pool(case, tens, include_new=True)
    out, lse, _ = _run_oracle(case, tens, pool)
    for s, (K, V) in enumerate(logical_kv(case, tens)):
        for h in range(4):
            np.testing.assert_allclose(out[s, h], V[:, h // 2].mean(0), rtol=0, atol=1e-13)
            assert abs(lse[s, h] - math.log(case.seq_lens[s])) < 1e-13


def test_empty_range_gives_zero_and_minus_inf():
    case = wl.make_case("empty", [20], 2, 1, 16, 16, "f32", "f32", "f32", seed=61)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    out, lse, _ = _run_oracle(case, tens, pool, tok_begin=[5], tok_end=[5])
    assert np.all(out == 0) and np.all(lse == -np.inf)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_then_merge_equals_unsplit(seed):
    case = wl.make_case("split", [300, 47, 1], 8, 2, 32, 16, "bf16", "bf16", "bf16",
                        seed=70 + seed)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    full, full_lse, _ = _run_oracle(case, tens, pool)
    rng = np.random.default_rng(seed)
    S = 6
    bounds = []
    for n in case.seq_lens:
        # random cut points, including empty and single-token partitions
        cuts = np.sort(rng.integers(0, n + 1, size=S - 1))
        if n > 2:
            cuts[0] = cuts[1] = min(cuts[1], n - 1)        # an empty partition
            cuts[2] = min(cuts[1] + 1, n)                  # a single-token partition
            cuts = np.sort(cuts)
        bounds.append(np.concatenate([[0], cuts, [n]]))
    bounds = np.array(bounds, dtype=np.int32)
    R = case.batch * case.num_q_heads
    po = np.zeros((R, S, case.head_dim))
    pl = np.zeros((R, S))
    for p in range(S):
        o, l, _ = _run_oracle(case, tens, pool, tok_begin=bounds[:, p], tok_end=bounds[:, p + 1])
        po[:, p] = o.reshape(R, -1)
        pl[:, p] = l.reshape(R)
    mo, ml = oracle.merge(po, pl)
    np.testing.assert_allclose(mo, full.reshape(R, -1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, full_lse.reshape(R), rtol=0, atol=1e-12)


def test_merge_weights_and_degenerate_rows():
    rng = np.random.default_rng(9)
    po = rng.standard_normal((3, 4, 8))
    pl = np.array([[0.5, -np.inf, 2.0, -np.inf],
                   [-np.inf] * 4,
                   [1.0, 1.0, 1.0, 1.0]])
    out, lse = oracle.merge(po, pl)
    w = np.exp(np.array([0.5, 2.0]) - 2.0)
    np.testing.assert_allclose(out[0], (w[0] * po[0, 0] + w[1] * po[0, 2]) / w.sum(), atol=1e-15)
    assert np.all(out[1] == 0) and lse[1] == -np.inf
    np.testing.assert_allclose(out[2], po[2].mean(0), atol=1e-15)
    np.testing.assert_allclose(lse[2], 1.0 + math.log(4), atol=1e-15)


# --------------------------------------------------------------------------- append
def test_append_index_worked_example():
    for line in _lines("append_example.txt"):
        bs, tok, blk_i, off = (int(x) for x in line.split())
        case = wl.make_case("ex", [tok + 1], 2, 1, 8, bs, "f32", "f32", "f32", seed=81)
        tens = wl.make_tensors(case)
        pool = np.zeros(oracle.kv_bytes(1, 1, 8, case.num_blocks * bs, 4), np.uint8)
        oracle.append(pool, "f32", case.geometry, 0, np_raw(tens.k_new), np_raw(tens.v_new),
                      "f32", case.tables, np.array([tok], np.int32))
        p = pool.view(np.float32).reshape(case.num_blocks, 2, 1, 1, bs, 8)
        blk = case.tables[0, blk_i]
        assert np.array_equal(p[blk, 0, 0, 0, off], tens.k_new.numpy()[0, 0])
        assert np.array_equal(p[blk, 1, 0, 0, off], tens.v_new.numpy()[0, 0])
        assert np.count_nonzero(p) == np.count_nonzero(tens.k_new.numpy()) + \
            np.count_nonzero(tens.v_new.numpy())


def test_append_order_invariance_and_no_collisions():
    case = wl.make_case("ord", [40, 17, 33], 4, 2, 16, 16, "bf16", "bf16", "bf16", seed=91)
    tens = wl.make_tensors(case)
    a = oracle_pool(case, tens)
    perm = torch.randperm(tens.tok_seq.shape[0], generator=torch.Generator().manual_seed(1))
    for f in ("k_tokens", "v_tokens", "tok_seq", "tok_pos"):
        setattr(tens, f, getattr(tens, f)[perm].contiguous())
    b = oracle_pool(case, tens)
    assert np.array_equal(a, b)
    # every written element is distinct: as many nonzero bf16 words as tokens x heads x D x 2
    T = tens.tok_seq.shape[0]
    assert np.count_nonzero(a.view(np.uint16)) == T * 2 * 16 * 2


def test_append_rejects_out_of_range():
    case = wl.make_case("bad", [10], 2, 1, 8, 16, "f32", "f32", "f32", seed=95)
    tens = wl.make_tensors(case)
    pool = np.zeros(oracle.kv_bytes(1, 1, 8, case.num_blocks * 16, 4), np.uint8)
    with pytest.raises(ValueError):
        oracle.append(pool, "f32", case.geometry, 0, np_raw(tens.k_new), np_raw(tens.v_new),
                      "f32", case.tables, np.array([16], np.int32))


# --------------------------------------------------------------------------- planted mistakes
MUTANTS = {
    1: "kv head = hq % Hkv instead of hq // G",
    2: "token index off by one",
    3: "head-dim reversed in q.k",
    4: "softmax scale dropped",
    5: "sign of the exponent flipped",
    6: "K read in place of V",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistakes_fail_a_pin(mutant):
    case = wl.make_case("mut", [37, 70], 8, 2, 32, 16, "f32", "f32", "f32", seed=99)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    good, _, _ = _run_oracle(case, tens, pool)
    bad, _, _ = _run_oracle(case, tens, pool, mutant=mutant)
    ref = _naive_case(case, tens)
    np.testing.assert_allclose(good, ref, atol=1e-12)
    assert np.max(np.abs(bad - ref)) > 1e-6, MUTANTS[mutant]


# --------------------------------------------------------------------------- multi-token decode
def _mq_q(case, q_len, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(case.batch, q_len, case.num_q_heads, case.head_dim, generator=g).to(
        wl.TORCH_DT[case.q_dtype])


@pytest.mark.parametrize("q_len", [1, 2, 5])
def test_multi_token_decode_equals_causal_naive_attention(q_len):
    case = wl.make_case("mq", [q_len, 40, 77], 8, 2, 32, 16, "bf16", "bf16", "bf16", seed=120)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    q = _mq_q(case, q_len)
    out, lse = oracle.decode_mq(np_raw(q), "bf16", pool, "bf16", case.geometry, 0, case.tables,
                                case.seq_lens, q_len, case.scale)
    qd = q.double().numpy()
    G = case.num_q_heads // case.num_kv_heads
    for s, (K, V) in enumerate(logical_kv(case, tens)):
        n = int(case.seq_lens[s])
        for i in range(q_len):
            end = n - q_len + i + 1          # causal: keys up to the query's own position
            for h in range(case.num_q_heads):
                ref, w = _naive(qd[s, i, h], K[:end, h // G], V[:end, h // G], case.scale)
                np.testing.assert_allclose(out[s, i, h], ref, rtol=0, atol=1e-12)


def test_multi_token_decode_with_one_token_is_single_query_decode():
    case = wl.make_case("mq1", [33, 100], 8, 2, 32, 16, "f32", "f32", "f32", seed=121)
    tens = wl.make_tensors(case)
    pool = oracle_pool(case, tens, include_new=True)
    a, la = oracle.decode_mq(np_raw(tens.q).reshape(2, 1, 8, 32), "f32", pool, "f32",
                             case.geometry, 0, case.tables, case.seq_lens, 1, case.scale)
    b, lb, _ = _run_oracle(case, tens, pool)
    assert np.array_equal(a[:, 0], b) and np.array_equal(la[:, 0], lb)


# --------------------------------------------------------------------------- block-wise FP8 scales
def _bs_setup(case, tens, group_tokens=0):
    geom = case.geometry
    nb = case.num_blocks
    scales = np.zeros((nb, 2, case.num_layers, case.num_kv_heads), np.float32)
    seq = np.concatenate([np_raw(tens.tok_seq), np.arange(case.batch, dtype=np.int32)])
    pos = np.concatenate([np_raw(tens.tok_pos), np_raw(tens.new_pos)])
    k = np.concatenate([np_raw(tens.k_tokens), np_raw(tens.k_new)])
    v = np.concatenate([np_raw(tens.v_tokens), np_raw(tens.v_new)])
    oracle.block_scales(scales, geom, case.layer, k, v, "bf16", case.tables, seq, pos,
                        group_tokens)
    pool = np.zeros(oracle.kv_bytes(case.num_layers, case.num_kv_heads, case.head_dim,
                                    nb * case.block_size, 1), np.uint8)
    oracle.append_tokens(pool, "e4m3", geom, case.layer, k, v, "bf16", case.tables, seq, pos,
                         block_scales=scales)
    return scales, pool


def test_uniform_block_scales_equal_the_per_tensor_path():
    case = wl.make_case("bs_uni", [100, 33], 8, 2, 32, 16, "e4m3", "bf16", "bf16", seed=130)
    tens = wl.make_tensors(case)
    ks = 0.0123
    uni = np.full((case.num_blocks, 2, 1, 2), ks, np.float32)
    a = oracle_pool(case, tens, ks, ks, include_new=True)
    b = np.zeros_like(a)
    seq = np.concatenate([np_raw(tens.tok_seq), np.arange(2, dtype=np.int32)])
    pos = np.concatenate([np_raw(tens.tok_pos), np_raw(tens.new_pos)])
    oracle.append_tokens(b, "e4m3", case.geometry, 0,
                         np.concatenate([np_raw(tens.k_tokens), np_raw(tens.k_new)]),
                         np.concatenate([np_raw(tens.v_tokens), np_raw(tens.v_new)]), "bf16",
                         case.tables, seq, pos, block_scales=uni)
    assert np.array_equal(a, b)
    o1, l1, _ = _run_oracle(case, tens, a, ks, ks)
    o2, l2, _ = oracle.decode(np_raw(tens.q), "bf16", b, "e4m3", case.geometry, 0, case.tables,
                              case.seq_lens, case.scale, 99.0, 99.0, block_scales=uni)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_block_scales_put_each_tiles_largest_value_at_448():
    case = wl.make_case("bs_max", [70, 300], 8, 2, 32, 16, "e4m3", "bf16", "bf16", seed=131)
    tens = wl.make_tensors(case)
    scales, pool = _bs_setup(case, tens)
    codes = pool.reshape(case.num_blocks, 2, 1, 2, 16, 32)
    used = sorted({int(b) for b in case.tables[case.tables >= 0]})
    for blk in used:
        for kv in range(2):
            for h in range(2):
                assert scales[blk, kv, 0, h] > 0
                tile = codes[blk, kv, 0, h]
                assert np.any((tile == 0x7E) | (tile == 0xFE)), (blk, kv, h)


def test_block_scaled_decode_equals_naive_on_dequantised_values():
    case = wl.make_case("bs_naive", [150, 61], 8, 2, 32, 16, "e4m3", "bf16", "bf16", seed=132)
    tens = wl.make_tensors(case)
    scales, pool = _bs_setup(case, tens)
    out, _, _ = oracle.decode(np_raw(tens.q), "bf16", pool, "e4m3", case.geometry, 0,
                              case.tables, case.seq_lens, case.scale, block_scales=scales)
    dec = torch.from_numpy(pool).view(torch.float8_e4m3fn).double().numpy().reshape(
        case.num_blocks, 2, 1, 2, 16, 32) * scales[:, :, :, :, None, None]
    kv = []
    for s in range(case.batch):
        n = int(case.seq_lens[s])
        blocks = case.tables[s, :(n + 15) // 16]
        K = dec[blocks, 0, 0].transpose(0, 2, 1, 3).reshape(-1, 2, 32)[:n]
        V = dec[blocks, 1, 0].transpose(0, 2, 1, 3).reshape(-1, 2, 32)[:n]
        kv.append((K, V))
    ref = _naive_case(case, tens, kv)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_block_scales_are_more_accurate_than_one_scale_on_spiky_keys():
    case = wl.make_case("bs_spiky", [2000], 8, 2, 32, 16, "e4m3", "bf16", "bf16", seed=133,
                        spike_frac=0.01)
    tens = wl.make_tensors(case)
    exact_case = wl.make_case("bs_spiky", [2000], 8, 2, 32, 16, "bf16", "bf16", "bf16", seed=133,
                              spike_frac=0.01)
    exact, _, _ = _run_oracle(exact_case, tens, oracle_pool(exact_case, tens, include_new=True))
    ks, vs = fp8_scales(tens)
    per_tensor, _, _ = _run_oracle(case, tens, oracle_pool(case, tens, ks, vs, include_new=True),
                                   ks, vs)
    scales, pool = _bs_setup(case, tens)
    blockwise, _, _ = oracle.decode(np_raw(tens.q), "bf16", pool, "e4m3", case.geometry, 0,
                                    case.tables, case.seq_lens, case.scale, block_scales=scales)
    assert np.abs(blockwise - exact).max() < np.abs(per_tensor - exact).max()


# --------------------------------------------------------------------------- scale groups
def _groups(case, S):
    """(sequence, first entry, entries) of every scale group of S tokens."""
    bs = case.block_size
    out = []
    for sq in range(case.batch):
        n = int(case.seq_lens[sq])
        for e0 in range(0, (n + bs - 1) // bs, S // bs):
            out.append((sq, e0, case.tables[sq, e0:min(e0 + S // bs, (n + bs - 1) // bs)]))
    return out


@pytest.mark.parametrize("S", [64, 128])
def test_scale_groups_share_one_scale_and_store_their_max_at_448(S):
    """One scale per S tokens ("Unlocking long context" section 3.2, 64-128
    tokens): every block of a group holds the same scale, and the group's
    largest element encodes to the largest E4M3 code, in K and in V."""
    case = wl.make_case(f"grp{S}", [700, 333, 64, 1], 8, 2, 32, 16, "e4m3", "bf16", "bf16",
                        seed=140, spike_frac=0.01)
    tens = wl.make_tensors(case)
    scales, pool = _bs_setup(case, tens, S)
    codes = pool.reshape(case.num_blocks, 2, 1, 2, 16, 32)
    for sq, e0, blocks in _groups(case, S):
        for kv in range(2):
            for h in range(2):
                sc = scales[blocks, kv, 0, h]
                assert np.all(sc == sc[0]) and sc[0] > 0, (sq, e0, kv, h)
                n = int(case.seq_lens[sq])
                toks = codes[blocks, kv, 0, h].reshape(-1, 32)[:n - e0 * 16]
                assert np.any((toks == 0x7E) | (toks == 0xFE)), (sq, e0, kv, h)


def test_scale_groups_nest_and_reduce_to_per_block_scales():
    """Scale groups of 128 tokens are the larger of their two 64-token halves'
    scales (the maximum commutes with the correctly rounded division), and
    groups of one block (S = block size, or 0) are the per-block scales."""
    case = wl.make_case("grp_nest", [1000, 129, 300], 8, 2, 32, 16, "e4m3", "bf16", "bf16",
                        seed=141, spike_frac=0.01)
    tens = wl.make_tensors(case)
    s64, _ = _bs_setup(case, tens, 64)
    s128, _ = _bs_setup(case, tens, 128)
    for sq, e0, blocks in _groups(case, 128):
        lo, hi = blocks[:4], blocks[4:]
        want = s64[lo[0]] if hi.size == 0 else np.maximum(s64[lo[0]], s64[hi[0]])
        for b in blocks:
            assert np.array_equal(s128[b], want), (sq, e0)
    s16, _ = _bs_setup(case, tens, 16)
    s0, _ = _bs_setup(case, tens, 0)
    assert np.array_equal(s16, s0)
    # one block per group is the per-block result: each block's largest value at 448
    used = sorted({int(b) for b in case.tables[case.tables >= 0]})
    assert np.array_equal(s16[used], s0[used])


def test_scale_group_size_must_be_a_multiple_of_the_block_size():
    case = wl.make_case("grp_bad", [40], 8, 2, 32, 16, "e4m3", "bf16", "bf16", seed=142)
    tens = wl.make_tensors(case)
    with pytest.raises(ValueError):
        _bs_setup(case, tens, 24)
    with pytest.raises(ValueError):
        _bs_setup(case, tens, 8)
