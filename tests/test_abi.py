"""C-ABI library checks that need no GPU: it builds, loads, exports every
symbol include/pkv.h declares, sizes pools by the pages' formula, runs the host
block allocator, and rejects bad arguments before any device work."""
import ctypes
import os
import re

import pytest

import oracle
from paged_kv_cache_215_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    pkv_build.build()
    from paged_kv_cache_215_gb300 import pkv as mod
    return mod


def test_library_exports_every_declared_symbol(pkv):
    hdr = open(os.path.join(ROOT, "include", "pkv.h")).read()
    declared = set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(\w+)\s*\(", hdr))
    assert len(declared) >= 20
    lib = ctypes.CDLL(pkv_build.SO)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared == set(pkv.EXPORTS)


def test_pool_bytes_is_the_pages_formula(pkv):
    for (L, hq, hkv, D, bs, nb, dt, eb) in [(1, 32, 8, 128, 16, 9012, "bf16", 2),
                                            (80, 64, 8, 128, 32, 7, "f16", 2),
                                            (2, 4, 2, 64, 16, 32, "f32", 4),
                                            (1, 32, 8, 128, 16, 1000, "e4m3", 1)]:
        g = pkv.geometry(L, hq, hkv, D, bs, nb, dt)
        assert pkv.kv_pool_bytes(g) == oracle.kv_bytes(L, hkv, D, nb * bs, eb)
    assert pkv.kv_pool_bytes(pkv.geometry(1, 3, 2, 128, 16, 10, "bf16")) == 0   # 3 % 2 != 0
    assert pkv.kv_pool_bytes(pkv.geometry(1, 2, 2, 100, 16, 10, "bf16")) == 0   # D % 8 != 0


class FakePool:
    """A pool whose device pointer is never dereferenced (allocator only)."""

    def __init__(self, pkv, nb=10):
        self.pkv = pkv
        self.g = pkv.geometry(1, 4, 2, 64, 16, nb, "bf16")
        h = ctypes.c_void_p()
        rc = pkv.lib().kv_pool_create(ctypes.byref(self.g), ctypes.c_void_p(1 << 20),
                                      pkv.kv_pool_bytes(self.g), None, ctypes.byref(h))
        assert rc == 0
        self.h = h

    def alloc(self, n):
        out = (ctypes.c_int32 * max(n, 1))()
        rc = self.pkv.lib().kv_pool_alloc(self.h, n, out)
        return rc, list(out[:n])

    def call(self, name, ids):
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        return getattr(self.pkv.lib(), name)(self.h, len(ids), arr)

    def ref(self, i):
        return self.pkv.lib().kv_pool_refcount(self.h, i)

    def nfree(self):
        return self.pkv.lib().kv_pool_num_free(self.h)

    def close(self):
        self.pkv.lib().kv_pool_destroy(self.h)


def test_allocator_all_or_nothing(pkv):
    p = FakePool(pkv, nb=10)
    rc, ids = p.alloc(4)
    assert rc == 0 and len(set(ids)) == 4 and p.nfree() == 6
    rc, _ = p.alloc(7)
    assert rc == pkv.PKV_ENOMEM and p.nfree() == 6          # nothing taken
    rc, more = p.alloc(6)
    assert rc == 0 and p.nfree() == 0 and not set(more) & set(ids)
    assert p.call("kv_pool_free", ids + more) == 0 and p.nfree() == 10
    assert all(p.ref(i) == 0 for i in range(10))
    p.close()


def test_allocator_refcounts_share_and_free(pkv):
    p = FakePool(pkv, nb=6)
    _, ids = p.alloc(2)
    assert p.call("kv_pool_share", ids) == 0 and p.call("kv_pool_share", ids[:1]) == 0
    assert p.ref(ids[0]) == 3 and p.ref(ids[1]) == 2
    assert p.call("kv_pool_free", ids) == 0
    assert p.ref(ids[0]) == 2 and p.ref(ids[1]) == 1 and p.nfree() == 4
    # freeing more references than exist fails and changes nothing
    assert p.call("kv_pool_free", [ids[1], ids[1]]) == pkv.PKV_EINVAL and p.ref(ids[1]) == 1
    assert p.call("kv_pool_free", [ids[1]]) == 0 and p.nfree() == 5
    assert p.call("kv_pool_share", [ids[1]]) == pkv.PKV_EINVAL     # sharing a free block
    p.close()


def test_allocator_reserve(pkv):
    p = FakePool(pkv, nb=8)
    assert p.call("kv_pool_reserve", [5, 2, 7]) == 0
    assert [p.ref(i) for i in range(8)] == [0, 0, 1, 0, 0, 1, 0, 1]
    assert p.call("kv_pool_reserve", [1, 2]) == pkv.PKV_EINVAL      # 2 is taken
    assert p.call("kv_pool_reserve", [1, 1]) == pkv.PKV_EINVAL      # repeated
    assert p.call("kv_pool_reserve", [8]) == pkv.PKV_EINVAL         # out of range
    assert p.ref(1) == 0 and p.nfree() == 5
    rc, ids = p.alloc(5)
    assert rc == 0 and sorted(ids) == [0, 1, 3, 4, 6]
    p.close()


def test_decode_rejects_bad_arguments_before_device_work(pkv):
    p = FakePool(pkv, nb=8)
    L = pkv.lib()
    x = ctypes.c_void_p(1 << 20)
    common = dict(out=x, od=pkv.PKV_BF16, q=x, qd=pkv.PKV_BF16, layer=0, tab=x, mb=4, lens=x,
                  B=2, maxlen=64, scale=0.125, ks=1.0, vs=1.0, S=0, ws=x, wsb=1 << 20)

    def call(**kw):
        a = dict(common, **kw)
        return L.paged_decode_attention(a["out"], a["od"], a["q"], a["qd"], p.h, a["layer"],
                                        a["tab"], a["mb"], a["lens"], a["B"], a["maxlen"],
                                        a["scale"], a["ks"], a["vs"], a["S"], a["ws"], a["wsb"],
                                        None)
    assert call(B=0) == 0                                  # empty batch: no-op
    assert call(layer=1) == pkv.PKV_EINVAL                 # layer out of range
    assert call(B=-1) == pkv.PKV_EINVAL
    assert call(maxlen=65) == pkv.PKV_EINVAL               # longer than the table holds
    assert call(od=pkv.PKV_FP8_E4M3) == pkv.PKV_EINVAL     # out dtype
    assert call(q=ctypes.c_void_p((1 << 20) + 2)) == pkv.PKV_EINVAL   # misaligned q
    assert call(tab=None) == pkv.PKV_EINVAL
    assert call(S=-2) == pkv.PKV_EINVAL
    p.close()


def test_shared_prefix_decode_rejects_bad_arguments_before_device_work(pkv):
    p = FakePool(pkv, nb=8)                                # bf16, head_dim 64, bs 16
    L = pkv.lib()
    x = ctypes.c_void_p(1 << 20)
    common = dict(ptab=x, pblocks=2, plen=32, plens=x, B=2, maxlen=64, ks=1.0, vs=1.0)

    def call(**kw):
        a = dict(common, **kw)
        return L.paged_decode_attention_cascade(x, pkv.PKV_BF16, x, pkv.PKV_BF16, p.h, 0,
                                                a["ptab"], a["pblocks"], a["plen"], a["plens"],
                                                x, 4, x, a["B"], a["maxlen"], 0.125, a["ks"],
                                                a["vs"], x, 1 << 20, None, None)
    assert call(B=0) == 0                                  # empty batch: no-op
    assert call(plen=8) == pkv.PKV_EINVAL                  # not a multiple of the block size
    assert call(pblocks=1) == pkv.PKV_EINVAL               # longer than the prefix table
    assert call(ptab=None) == pkv.PKV_EINVAL
    assert call(plens=None) == pkv.PKV_EINVAL
    assert call(maxlen=65) == pkv.PKV_EINVAL               # longer than the tables hold
    assert call() == pkv.PKV_EUNSUPPORTED                  # head_dim 64: no tcgen05 kernel
    p.close()


def test_append_rejects_dtype_mismatch(pkv):
    p = FakePool(pkv, nb=8)
    x = ctypes.c_void_p(1 << 20)
    rc = pkv.lib().kv_append(p.h, 0, x, x, pkv.PKV_F32, x, 4, x, 2, 1.0, 1.0, None)
    assert rc == pkv.PKV_EINVAL                            # f32 into a bf16 pool
    rc = pkv.lib().kv_append(p.h, 3, x, x, pkv.PKV_BF16, x, 4, x, 2, 1.0, 1.0, None)
    assert rc == pkv.PKV_EINVAL                            # layer
    p.close()


def test_strerror_names_every_status(pkv):
    names = {pkv.strerror(c) for c in range(-6, 1)}
    assert len(names) == 7 and "unknown status" not in names


def _c_kind(ctype):
    t = " ".join(ctype.replace("const", " ").split())
    if "*" in t or t in ("cudaStream_t",):
        return "ptr"
    if t in ("float",):
        return "f32"
    if t in ("double",):
        return "f64"
    if t in ("size_t",):
        return "u64"                            # ctypes.c_size_t is c_uint64 on LP64
    if t in ("int64_t", "long long"):
        return "i64"
    if t in ("uint64_t", "unsigned long long"):
        return "u64"
    if t in ("int", "int32_t", "pkv_dtype"):
        return "i32"
    raise AssertionError(f"unclassified C type {ctype!r}")


def _ct_kind(ct):
    if ct in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(ct, type) and
                                                     issubclass(ct, ctypes._Pointer)):
        return "ptr"
    table = {ctypes.c_float: "f32", ctypes.c_double: "f64", ctypes.c_size_t: "u64",
             ctypes.c_int64: "i64", ctypes.c_uint64: "u64", ctypes.c_int: "i32",
             ctypes.c_int32: "i32"}
    return table[ct]


def test_binding_argument_lists_match_the_header(pkv):
    """Every prototype in include/pkv.h against the ctypes argument list the
    binding installs: same count, and pointer / 32-bit int / float / 64-bit
    unsigned (size_t) / 64-bit int in every position (a stale binding would pass
    wrong values)."""
    hdr = open(os.path.join(ROOT, "include", "pkv.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    protos = re.findall(r"PKV_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)\s*;", hdr)
    assert len(protos) == len(pkv.EXPORTS)
    lib = pkv.lib()
    for name, params in protos:
        params = " ".join(params.split())
        args = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        # drop the parameter name: the last identifier of each declaration
        kinds = [_c_kind(re.sub(r"\b\w+$", "", a).strip() or a) for a in args]
        got = [_ct_kind(t) for t in (getattr(lib, name).argtypes or [])]
        assert kinds == got, f"{name}: header {kinds} binding {got}"


def _prep(pkv, p, lens, tables, new=None):
    import numpy as np
    lens = np.asarray(lens, np.int32)
    first = np.full(len(lens), 77, np.int32)
    newp = None
    if new is not None:
        new = np.asarray(new, np.int32)
        newp = new.ctypes.data
    rc = pkv.lib().kv_pool_prepare_append(p.h, len(lens), lens.ctypes.data, newp,
                                          tables.ctypes.data, tables.shape[1],
                                          first.ctypes.data, None)
    return rc, first


def test_prepare_append_takes_a_block_exactly_when_a_token_starts_one(pkv):
    """The pages' append_token: a block is allocated when the new token's
    position is a multiple of the block size (block size 16 here)."""
    import numpy as np
    p = FakePool(pkv, nb=20)
    _, ids = p.alloc(2)
    tables = np.full((4, 6), -1, np.int32)
    tables[0, 0] = ids[0]                                 # 16 tokens: the next starts block 1
    tables[1, 0] = ids[1]                                 # 5 tokens: room left in block 0
    # sequences 2 and 3 hold no token yet: each needs its block 0
    free0 = p.nfree()
    rc, first = _prep(pkv, p, [16, 5, 0, 0], tables)
    assert rc == 0
    assert list(first) == [1, -1, 0, 0]
    assert tables[1, 1] == -1 and tables[0, 0] == ids[0] and tables[1, 0] == ids[1]
    new = [int(tables[0, 1]), int(tables[2, 0]), int(tables[3, 0])]
    assert len(set(new) | set(ids)) == 5 and all(p.ref(i) == 1 for i in new)
    assert p.nfree() == free0 - 3
    p.close()


def test_prepare_append_chunk_spans_several_blocks(pkv):
    import numpy as np
    p = FakePool(pkv, nb=20)
    tables = np.full((2, 8), -1, np.int32)
    _, ids = p.alloc(1)
    tables[0, 0] = ids[0]
    rc, first = _prep(pkv, p, [10, 0], tables, new=[40, 17])   # 10+40 -> 4 blocks; 17 -> 2
    assert rc == 0 and list(first) == [1, 0]
    assert (tables[0, :4] >= 0).all() and tables[0, 4] == -1
    assert (tables[1, :2] >= 0).all() and tables[1, 2] == -1
    assert p.nfree() == 20 - 1 - 3 - 2
    # k = 0 changes nothing
    before = tables.copy()
    rc, first = _prep(pkv, p, [50, 17], tables, new=[0, 0])
    assert rc == 0 and list(first) == [-1, -1] and np.array_equal(tables, before)
    p.close()


def test_prepare_append_is_all_or_nothing(pkv):
    import numpy as np
    p = FakePool(pkv, nb=5)
    tables = np.full((3, 4), -1, np.int32)
    rc, _ = _prep(pkv, p, [0, 0, 0], tables, new=[32, 32, 17])   # 2 + 2 + 2 > 5
    assert rc == pkv.PKV_ENOMEM and p.nfree() == 5 and (tables == -1).all()
    rc, _ = _prep(pkv, p, [0, 0, 0], tables, new=[65, 1, 1])     # 5 blocks > 4 entries
    assert rc == pkv.PKV_EINVAL and p.nfree() == 5 and (tables == -1).all()
    rc, _ = _prep(pkv, p, [-1, 0, 0], tables)
    assert rc == pkv.PKV_EINVAL and p.nfree() == 5
    rc, _ = _prep(pkv, p, [0, 0, 0], tables, new=[32, 32, 16])   # exactly 5
    assert rc == 0 and p.nfree() == 0
    p.close()


def test_prepare_append_copy_of_a_shared_tail_is_planned_in_order(pkv):
    """Two sequences share a partly filled tail block.  Without a device the
    copy cannot be issued, so the call reports PKV_ECUDA and leaves pool and
    tables exactly as they were (the copy itself is exercised on the GPU); a
    shared *full* block needs no copy (the next token starts a new block)."""
    import numpy as np
    p = FakePool(pkv, nb=8)
    _, ids = p.alloc(2)
    p.call("kv_pool_share", ids)                          # both blocks shared by 2 tables
    tables = np.full((2, 4), -1, np.int32)
    tables[:, 0], tables[:, 1] = ids[0], ids[1]
    before, free0 = tables.copy(), p.nfree()
    rc, _ = _prep(pkv, p, [20, 20], tables)               # tail block ids[1] has room
    assert rc == pkv.PKV_ECUDA
    assert np.array_equal(tables, before) and p.nfree() == free0
    assert p.ref(ids[1]) == 2
    rc, first = _prep(pkv, p, [32, 32], tables)           # full: each starts a new block
    assert rc == 0 and list(first) == [2, 2] and p.nfree() == free0 - 2
    assert p.ref(ids[0]) == 2 and p.ref(ids[1]) == 2
    # not enough blocks for the copy either: PKV_ENOMEM before any copy is tried
    q = FakePool(pkv, nb=2)
    _, qids = q.alloc(2)
    q.call("kv_pool_share", qids[:1])
    t2 = np.full((2, 2), -1, np.int32)
    t2[:, 0] = qids[0]
    rc, _ = _prep(pkv, q, [3, 3], t2)
    assert rc == pkv.PKV_ENOMEM and q.ref(qids[0]) == 2
    p.close()
    q.close()


def test_prepare_append_rejects_a_dead_tail_entry(pkv):
    import numpy as np
    p = FakePool(pkv, nb=4)
    tables = np.full((1, 2), -1, np.int32)
    tables[0, 0] = 3                                      # never taken: refcount 0
    rc, _ = _prep(pkv, p, [5], tables)
    assert rc == pkv.PKV_EINVAL and p.nfree() == 4 and tables[0, 0] == 3
    p.close()
