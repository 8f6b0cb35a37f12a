"""Thin Python binding of the C ABI in include/pkv.h (argument marshalling only).

Torch tensors provide device memory and the current CUDA stream; every step of
the computation runs in the library's CUDA kernels.  The library must have been
built (``paged_kv_cache_215_gb300.build.build()``); importing this module
without it raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

PKV_OK, PKV_EINVAL, PKV_ENOMEM, PKV_ECUDA, PKV_EBOUNDS, PKV_ETIMEOUT, PKV_EUNSUPPORTED = \
    0, -1, -2, -3, -4, -5, -6
PKV_F32, PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2, 3
STATUS_BYTES = 16

DTYPE_CODE = {"f32": PKV_F32, "f16": PKV_F16, "bf16": PKV_BF16, "e4m3": PKV_FP8_E4M3}
TORCH_CODE = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
ELEM_BYTES = {PKV_F32: 4, PKV_F16: 2, PKV_BF16: 2, PKV_FP8_E4M3: 1}


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


class Geometry(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32)]


class LaunchOpts(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("kv_heads_per_cta", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("phase", ctypes.c_int32), ("pdl", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


def _load() -> ctypes.CDLL:
    path = _build.SO
    if not os.path.exists(path):
        raise ImportError(f"the CUDA library {path} is not built; run "
                          "paged_kv_cache_215_gb300.build.build() (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    I64 = ctypes.c_int64
    G = ctypes.POINTER(Geometry)
    sig = {
        "kv_pool_bytes": (Z, [G]),
        "kv_pool_create": (I, [G, P, Z, P, ctypes.POINTER(P)]),
        "kv_pool_destroy": (I, [P]),
        "kv_pool_geometry": (I, [P, G]),
        "kv_pool_alloc": (I, [P, I, P]),
        "kv_pool_reserve": (I, [P, I, P]),
        "kv_pool_free": (I, [P, I, P]),
        "kv_pool_share": (I, [P, I, P]),
        "kv_pool_refcount": (I, [P, ctypes.c_int32]),
        "kv_pool_num_free": (I, [P]),
        "kv_pool_cow": (I, [P, ctypes.c_int32, P, P]),
        "kv_pool_prepare_append": (I, [P, I, P, P, P, I, P, P]),
        "kv_append": (I, [P, I, P, P, I, P, I, P, I, F, F, P]),
        "kv_append_tokens": (I, [P, I, P, P, I, P, I, I, P, P, I64, F, F, P]),
        "kv_absmax": (I, [P, I, I64, P, P]),
        "kv_fp8_scale": (I, [P, I, P, P]),
        "kv_pool_set_block_scales": (I, [P, P]),
        "kv_block_scales": (I, [P, I, P, P, I, P, I, I, P, P, I64, I, P]),
        "paged_decode_workspace_bytes": (Z, [G, I, I, I]),
        "paged_decode_workspace_bytes_mq": (Z, [G, I, I, I, I]),
        "paged_decode_attention_mq": (I, [P, I, P, I, I, P, I, P, I, P, I, I, F, F, F, I, P, Z,
                                          ctypes.POINTER(LaunchOpts), P]),
        "paged_decode_attention": (I, [P, I, P, I, P, I, P, I, P, I, I, F, F, F, I, P, Z, P]),
        "paged_decode_attention_ex": (I, [P, I, P, I, P, I, P, I, P, I, I, F, F, F, I, P, Z,
                                          ctypes.POINTER(LaunchOpts), P]),
        "merge_partials": (I, [P, I, P, P, I, I, I, I, P]),
        "paged_decode_attention_partial": (I, [P, P, P, I, P, I, P, I, P, I, I, F, F, F, P, Z, P]),
        "paged_decode_step": (I, [P, I, P, I, P, P, I, P, I, P, I, P, I, I, F, F, F, I, P, Z,
                                  ctypes.POINTER(LaunchOpts), P]),
        "paged_decode_attention_static": (I, [P, I, P, I, P, I, P, I, P, I, I, F, F, F, I, P]),
        "paged_decode_attention_cascade": (I, [P, I, P, I, P, I, P, I, I, P, P, I, P, I, I, F, F,
                                               F, P, Z, ctypes.POINTER(LaunchOpts), P]),
        "paged_decode_workspace_bytes_cascade": (Z, [G, I, I, I, I]),
        "pkv_check_status": (I, [P, P]),
        "pkv_wait_selftest": (I, [P, P]),
        "pkv_strerror": (ctypes.c_char_p, [I]),
        "pkv_launch_count": (ctypes.c_uint64, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTS = ("kv_pool_bytes", "kv_pool_create", "kv_pool_destroy", "kv_pool_geometry",
           "kv_pool_alloc", "kv_pool_reserve", "kv_pool_free", "kv_pool_share",
           "kv_pool_refcount", "kv_pool_num_free", "kv_pool_cow", "kv_pool_prepare_append",
           "kv_append",
           "kv_append_tokens", "kv_absmax", "kv_fp8_scale", "paged_decode_workspace_bytes",
           "kv_pool_set_block_scales", "kv_block_scales",
           "paged_decode_attention", "paged_decode_attention_ex", "merge_partials",
           "paged_decode_attention_partial",
           "paged_decode_attention_static", "paged_decode_step",
           "paged_decode_attention_mq", "paged_decode_workspace_bytes_mq",
           "paged_decode_attention_cascade", "paged_decode_workspace_bytes_cascade",
           "pkv_check_status", "pkv_wait_selftest", "pkv_strerror", "pkv_launch_count")


def lib() -> ctypes.CDLL:
    return _lib


def strerror(code: int) -> str:
    return _lib.pkv_strerror(code).decode()


def _check(rc: int, what: str):
    if rc != PKV_OK:
        raise PkvError(rc, what)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.is_contiguous(), "tensors passed to the library must be contiguous"
    return t.data_ptr()


def _i32(x: Sequence[int]):
    arr = (ctypes.c_int32 * len(x))(*[int(v) for v in x])
    return arr


def geometry(num_layers, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
             kv_dtype) -> Geometry:
    code = DTYPE_CODE[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    return Geometry(num_layers, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, code)


def kv_pool_bytes(geom: Geometry) -> int:
    return int(_lib.kv_pool_bytes(ctypes.byref(geom)))


def launch_count() -> int:
    return int(_lib.pkv_launch_count())


def launch_opts(kernel=0, ctas_per_sm=0, kv_heads_per_cta=0, stages=0, phase=0,
                pdl=0) -> LaunchOpts:
    o = LaunchOpts()
    o.kernel, o.ctas_per_sm, o.kv_heads_per_cta, o.stages, o.phase, o.pdl = \
        kernel, ctas_per_sm, kv_heads_per_cta, stages, phase, pdl
    return o


class KVPool:
    """A paged KV pool: caller-owned device storage [NB, 2, L, Hkv, bs, D] plus the
    library's host state (block allocator, TMA descriptors)."""

    def __init__(self, geom: Geometry, device="cuda", storage: Optional[torch.Tensor] = None):
        self.geom = geom
        self.nbytes = kv_pool_bytes(geom)
        if self.nbytes == 0:
            raise PkvError(PKV_EINVAL, "kv_pool_bytes")
        self.storage = storage if storage is not None else \
            torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.status = torch.zeros(STATUS_BYTES // 4, dtype=torch.int32, device=self.storage.device)
        h = ctypes.c_void_p()
        _check(_lib.kv_pool_create(ctypes.byref(geom), _ptr(self.storage), self.storage.numel(),
                                   _ptr(self.status), ctypes.byref(h)), "kv_pool_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            _lib.kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def kv_dtype(self) -> int:
        return self.geom.kv_dtype

    def view(self) -> torch.Tensor:
        """The storage as [NB, 2, L, Hkv, bs, D] elements (uint8 for E4M3)."""
        g = self.geom
        dt = {PKV_F32: torch.float32, PKV_F16: torch.float16, PKV_BF16: torch.bfloat16,
              PKV_FP8_E4M3: torch.uint8}[g.kv_dtype]
        return self.storage.view(dt).view(g.num_blocks, 2, g.num_layers, g.num_kv_heads,
                                          g.block_size, g.head_dim)

    # ---- host block allocator
    def alloc(self, n: int):
        out = (ctypes.c_int32 * max(n, 1))()
        _check(_lib.kv_pool_alloc(self.handle, n, out), "kv_pool_alloc")
        return list(out[:n])

    def reserve(self, ids):
        _check(_lib.kv_pool_reserve(self.handle, len(ids), _i32(ids)), "kv_pool_reserve")

    def free(self, ids):
        _check(_lib.kv_pool_free(self.handle, len(ids), _i32(ids)), "kv_pool_free")

    def share(self, ids):
        _check(_lib.kv_pool_share(self.handle, len(ids), _i32(ids)), "kv_pool_share")

    def refcount(self, block_id: int) -> int:
        return int(_lib.kv_pool_refcount(self.handle, block_id))

    def num_free(self) -> int:
        return int(_lib.kv_pool_num_free(self.handle))

    def cow(self, block_id: int, stream=None) -> int:
        out = ctypes.c_int32()
        _check(_lib.kv_pool_cow(self.handle, block_id, ctypes.byref(out), _stream(stream)),
               "kv_pool_cow")
        return out.value

    def prepare_append(self, seq_lens, tables, new_tokens=None, stream=None):
        """Extend the host tables (numpy int32 [B, max_blocks], updated in place) for
        the next tokens of every sequence, copying shared tail blocks first; returns
        each row's first changed entry (-1: unchanged)."""
        import numpy as np
        assert tables.dtype == np.int32 and tables.flags["C_CONTIGUOUS"]
        B = tables.shape[0]
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        newt = None if new_tokens is None else np.ascontiguousarray(new_tokens, dtype=np.int32)
        first = np.empty(B, dtype=np.int32)
        _check(_lib.kv_pool_prepare_append(self.handle, B, lens.ctypes.data,
                                           None if newt is None else newt.ctypes.data,
                                           tables.ctypes.data, tables.shape[1],
                                           first.ctypes.data, _stream(stream)),
               "kv_pool_prepare_append")
        return first

    # ---- append (reshape_and_cache)
    def append(self, layer, k, v, tables, positions, k_scale=1.0, v_scale=1.0, stream=None):
        _check(_lib.kv_append(self.handle, layer, _ptr(k), _ptr(v), TORCH_CODE[k.dtype],
                              _ptr(tables), tables.shape[1], _ptr(positions), positions.shape[0],
                              k_scale, v_scale, _stream(stream)), "kv_append")

    def append_tokens(self, layer, k, v, tables, seq_ids, positions, k_scale=1.0, v_scale=1.0,
                      stream=None):
        _check(_lib.kv_append_tokens(self.handle, layer, _ptr(k), _ptr(v), TORCH_CODE[k.dtype],
                                     _ptr(tables), tables.shape[1], tables.shape[0],
                                     _ptr(seq_ids), _ptr(positions), seq_ids.shape[0], k_scale,
                                     v_scale, _stream(stream)), "kv_append_tokens")

    def set_block_scales(self, scales: Optional[torch.Tensor]):
        """Attach a [NB, 2, L, Hkv] float32 device tensor of per-tile E4M3 scales."""
        self.block_scales = scales
        _check(_lib.kv_pool_set_block_scales(self.handle, _ptr(scales)), "kv_pool_set_block_scales")

    def compute_block_scales(self, layer, k, v, tables, seq_ids, positions, group_tokens=0,
                             stream=None):
        """Block-wise scales of the scale groups (group_tokens positions; 0: one
        block) the tokens land in, into the attached scale array."""
        _check(_lib.kv_block_scales(self.handle, layer, _ptr(k), _ptr(v), TORCH_CODE[k.dtype],
                                    _ptr(tables), tables.shape[1], tables.shape[0],
                                    _ptr(seq_ids), _ptr(positions), positions.shape[0],
                                    group_tokens, _stream(stream)), "kv_block_scales")

    def check_status(self, stream=None) -> int:
        return int(_lib.pkv_check_status(self.handle, _stream(stream)))

    def wait_selftest(self, stream=None):
        """Launch the failure-detection self-test (a bounded wait that runs out,
        about 1 s); the next check_status returns PKV_ETIMEOUT."""
        _check(_lib.pkv_wait_selftest(self.handle, _stream(stream)), "pkv_wait_selftest")


def kv_absmax(x: torch.Tensor, out: torch.Tensor, stream=None):
    _check(_lib.kv_absmax(_ptr(x), TORCH_CODE[x.dtype], x.numel(), _ptr(out), _stream(stream)),
           "kv_absmax")


def kv_fp8_scale(amax: torch.Tensor, out: torch.Tensor, stream=None):
    """The library's per-tensor E4M3 scale of a tensor whose pieces' kv_absmax
    results are `amax` (float32, device), written to out[0]."""
    _check(_lib.kv_fp8_scale(_ptr(amax), amax.numel(), _ptr(out), _stream(stream)),
           "kv_fp8_scale")


def fp8_scales(k_parts, v_parts, stream=None):
    """Per-tensor E4M3 scales (k_scale, v_scale) of K and V held in pieces (for
    example the cached tokens and the new ones): kv_absmax of every piece, then
    kv_fp8_scale of each tensor, on the device; the two floats are read back."""
    dev = k_parts[0].device
    amax = torch.zeros(len(k_parts) + len(v_parts), dtype=torch.float32, device=dev)
    for i, x in enumerate(list(k_parts) + list(v_parts)):
        kv_absmax(x, amax[i:i + 1], stream)
    sc = torch.empty(2, dtype=torch.float32, device=dev)
    nk = len(k_parts)
    kv_fp8_scale(amax[:nk], sc[0:1], stream)
    kv_fp8_scale(amax[nk:], sc[1:2], stream)
    k, v = sc.cpu().tolist()
    return k, v


def workspace_bytes(geom: Geometry, batch: int, max_seq_len: int, num_splits: int = 0) -> int:
    return int(_lib.paged_decode_workspace_bytes(ctypes.byref(geom), batch, max_seq_len,
                                                 num_splits))


def paged_decode_attention(out, q, pool: KVPool, layer, tables, seq_lens, max_seq_len, scale,
                           k_scale=1.0, v_scale=1.0, num_splits=0, workspace=None, opts=None,
                           stream=None):
    if workspace is None:
        nb = workspace_bytes(pool.geom, q.shape[0], max_seq_len, num_splits)
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=pool.storage.device)
    args = (_ptr(out), TORCH_CODE[out.dtype], _ptr(q), TORCH_CODE[q.dtype], pool.handle, layer,
            _ptr(tables), tables.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, scale,
            k_scale, v_scale, num_splits, _ptr(workspace), workspace.numel())
    if opts is None:
        rc = _lib.paged_decode_attention(*args, _stream(stream))
    else:
        rc = _lib.paged_decode_attention_ex(*args, ctypes.byref(opts), _stream(stream))
    _check(rc, "paged_decode_attention")
    return out


def paged_decode_attention_partial(out, lse, q, pool: KVPool, layer, tables, seq_lens,
                                   max_seq_len, scale, k_scale=1.0, v_scale=1.0, workspace=None,
                                   stream=None):
    """Partial attention over the tokens this pool holds: fp32 out [B, Hq, D] and
    the natural log-sum-exp lse [B, Hq] of every row (for merging key ranges)."""
    if workspace is None:
        nb = workspace_bytes(pool.geom, q.shape[0], max_seq_len, 0)
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=pool.storage.device)
    assert out.dtype == torch.float32 and lse.dtype == torch.float32
    _check(_lib.paged_decode_attention_partial(
        _ptr(out), _ptr(lse), _ptr(q), TORCH_CODE[q.dtype], pool.handle, layer, _ptr(tables),
        tables.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, scale, k_scale, v_scale,
        _ptr(workspace), workspace.numel(), _stream(stream)), "paged_decode_attention_partial")
    return out, lse


def paged_decode_attention_static(out, q, pool: KVPool, layer, tables, seq_lens, max_seq_len,
                                  scale, k_scale=1.0, v_scale=1.0, num_splits=0, stream=None):
    """paged_decode_attention without a workspace argument: the library's built-in
    scratch array holds the partial results (see include/pkv.h)."""
    _check(_lib.paged_decode_attention_static(
        _ptr(out), TORCH_CODE[out.dtype], _ptr(q), TORCH_CODE[q.dtype], pool.handle, layer,
        _ptr(tables), tables.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, scale, k_scale,
        v_scale, num_splits, _stream(stream)), "paged_decode_attention_static")
    return out


def paged_decode_step(out, q, k_new, v_new, pool: KVPool, layer, tables, seq_lens, max_seq_len,
                      scale, k_scale=1.0, v_scale=1.0, num_splits=0, workspace=None, opts=None,
                      stream=None):
    """Store each sequence's new token at position seq_len - 1, then decode attention
    (fused into one attention launch on the tensor-core kernel)."""
    if workspace is None:
        nb = workspace_bytes(pool.geom, q.shape[0], max_seq_len, num_splits)
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=pool.storage.device)
    _check(_lib.paged_decode_step(
        _ptr(out), TORCH_CODE[out.dtype], _ptr(q), TORCH_CODE[q.dtype], _ptr(k_new), _ptr(v_new),
        TORCH_CODE[k_new.dtype], pool.handle, layer, _ptr(tables), tables.shape[1],
        _ptr(seq_lens), q.shape[0], max_seq_len, scale, k_scale, v_scale, num_splits,
        _ptr(workspace), workspace.numel(), None if opts is None else ctypes.byref(opts),
        _stream(stream)), "paged_decode_step")
    return out


def paged_decode_attention_mq(out, q, pool: KVPool, layer, tables, seq_lens, max_seq_len, scale,
                              k_scale=1.0, v_scale=1.0, num_splits=0, workspace=None, opts=None,
                              stream=None):
    """Causal attention of the last q_len tokens of every sequence (q, out:
    [B, q_len, Hq, D]) over the paged pool, the new tokens already stored."""
    B, q_len = q.shape[0], q.shape[1]
    if workspace is None:
        nb = int(_lib.paged_decode_workspace_bytes_mq(ctypes.byref(pool.geom), B, q_len,
                                                      max_seq_len, num_splits))
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=pool.storage.device)
    _check(_lib.paged_decode_attention_mq(
        _ptr(out), TORCH_CODE[out.dtype], _ptr(q), TORCH_CODE[q.dtype], q_len, pool.handle, layer,
        _ptr(tables), tables.shape[1], _ptr(seq_lens), B, max_seq_len, scale, k_scale, v_scale,
        num_splits, _ptr(workspace), workspace.numel(),
        None if opts is None else ctypes.byref(opts), _stream(stream)),
        "paged_decode_attention_mq")
    return out


def cascade_workspace_bytes(geom: Geometry, batch: int, max_blocks: int, max_seq_len: int,
                            prefix_len_max: int) -> int:
    return int(_lib.paged_decode_workspace_bytes_cascade(ctypes.byref(geom), batch, max_blocks,
                                                         max_seq_len, prefix_len_max))


def paged_decode_attention_cascade(out, q, pool: KVPool, layer, prefix_table, prefix_len_max,
                                   prefix_lens, tables, seq_lens, max_seq_len, scale,
                                   k_scale=1.0, v_scale=1.0, workspace=None, opts=None,
                                   stream=None):
    """Decode attention of sequences sharing a prefix of blocks: the prefix
    (prefix_table [P] int32, prefix_lens [B] int32 tokens per sequence) is read
    once for all of them; the result equals paged_decode_attention.  opts.kernel:
    0 automatic (a prefix that fits a quarter of L2 goes through the plain
    decode), 2 always the plain decode, 3 always the prefix pass."""
    B = q.shape[0]
    if workspace is None:
        nb = cascade_workspace_bytes(pool.geom, B, tables.shape[1], max_seq_len, prefix_len_max)
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=pool.storage.device)
    _check(_lib.paged_decode_attention_cascade(
        _ptr(out), TORCH_CODE[out.dtype], _ptr(q), TORCH_CODE[q.dtype], pool.handle, layer,
        _ptr(prefix_table), int(prefix_table.numel()) if prefix_table is not None else 0,
        prefix_len_max, _ptr(prefix_lens), _ptr(tables), tables.shape[1], _ptr(seq_lens), B,
        max_seq_len, scale, k_scale, v_scale, _ptr(workspace), workspace.numel(),
        ctypes.byref(opts) if opts is not None else None, _stream(stream)),
        "paged_decode_attention_cascade")
    return out


def merge_partials(out, part_o, part_lse, stream=None):
    B, H, S, D = part_o.shape
    _check(_lib.merge_partials(_ptr(out), TORCH_CODE[out.dtype], _ptr(part_o), _ptr(part_lse),
                               B, H, D, S, _stream(stream)), "merge_partials")
    return out
