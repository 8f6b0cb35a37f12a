"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (``paged_kv_cache_215_gb300``) never
imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over output rows);
this module compiles it with gcc and marshals numpy arrays through ctypes.
Each C function cites the passage of the source pages it follows.  Element
storage is passed raw: bf16 and f16 as uint16 bit patterns, E4M3 as uint8.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

# the oracle's own dtype codes (see oracle.c)
DT = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (OpenMP if available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _SO + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P, I, D, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float
            LL = ctypes.c_longlong
            L.or_decode.restype = I
            L.or_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, I, I, P, I, P, I,
                                    D, D, D, P, P, P, I, I, P]
            L.or_decode_mq.restype = I
            L.or_decode_mq.argtypes = [P, P, P, I, P, I, I, I, I, I, I, I, I, P, I, P, I, I,
                                       D, D, D, P]
            L.or_block_scales.restype = I
            L.or_block_scales.argtypes = [P, I, I, I, I, I, I, P, P, I, P, I, I, P, P, LL, I]
            L.or_append.restype = I
            L.or_append.argtypes = [P, I, I, I, I, I, I, I, P, P, I, P, I, P, I, F, F, P]
            L.or_append_tokens.restype = I
            L.or_append_tokens.argtypes = [P, I, I, I, I, I, I, I, P, P, I, P, I, I, P, P, LL,
                                           F, F, P]
            L.or_merge.restype = None
            L.or_merge.argtypes = [P, P, P, P, LL, I, I]
            L.or_absmax.restype = D
            L.or_absmax.argtypes = [P, I, LL]
            L.or_fp8_scale.restype = F
            L.or_fp8_scale.argtypes = [D]
            L.or_to_f64.restype = None
            L.or_to_f64.argtypes = [P, P, I, LL, D]
            L.or_e4m3_encode.restype = ctypes.c_uint8
            L.or_e4m3_encode.argtypes = [F, F]
            L.or_e4m3_encode_n.restype = None
            L.or_e4m3_encode_n.argtypes = [P, P, LL, F]
            L.or_e4m3_to_f64.restype = D
            L.or_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            L.or_f16_to_f64.restype = D
            L.or_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.or_bf16_to_f64.restype = D
            L.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.or_kv_bytes.restype = ctypes.c_uint64
            L.or_kv_bytes.argtypes = [ctypes.c_uint64] * 5
            L.or_num_threads.restype = I
            L.or_num_threads.argtypes = []
            _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _f32(a):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def num_threads() -> int:
    return lib().or_num_threads()


def kv_bytes(layers, kv_heads, head_dim, tokens, elem_bytes) -> int:
    """[MHPN 3.1] 2 x layers x kv_heads x head_dim x tokens x bytes."""
    return int(lib().or_kv_bytes(layers, kv_heads, head_dim, tokens, elem_bytes))


def e4m3_encode(x, scale: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().or_e4m3_encode_n(_ptr(out), _ptr(x), x.size, float(scale))
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib().or_to_f64(_ptr(out), _ptr(codes), DT["e4m3"], codes.size, 1.0)
    return out


def to_f64(raw, dtype: str, scale: float = 1.0) -> np.ndarray:
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size * raw.itemsize // ELEM_BYTES[dtype], dtype=np.float64)
    lib().or_to_f64(_ptr(out), _ptr(raw), DT[dtype], out.size, float(scale))
    return out


def absmax(raw, dtype: str) -> float:
    raw = np.ascontiguousarray(raw)
    n = raw.size * raw.itemsize // ELEM_BYTES[dtype]
    return float(lib().or_absmax(_ptr(raw), DT[dtype], n))


def fp8_scale(amax: float) -> float:
    """[UNLOCK 3.2] per-tensor E4M3 scale amax / 448 in fp32 (amax 0 gives 1)."""
    return float(lib().or_fp8_scale(float(amax)))


def decode(q, q_dtype, pool, kv_dtype, geom, layer, tables, seq_lens, scale,
           k_scale=1.0, v_scale=1.0, tok_begin=None, tok_end=None, rows=None,
           mutant=0, block_scales=None):
    """fp64 decode attention.  geom = dict(num_blocks, num_layers, num_kv_heads,
    block_size, head_dim, num_q_heads).  Returns (out [B,Hq,D], lse [B,Hq],
    wsum [B,Hq]) as fp64 arrays; rows not requested are NaN."""
    q = np.ascontiguousarray(q)
    pool = np.ascontiguousarray(pool)
    tables = _i32(tables)
    seq_lens = _i32(seq_lens)
    B = seq_lens.shape[0]
    Hq, D = geom["num_q_heads"], geom["head_dim"]
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    wsum = np.full((B, Hq), np.nan)
    tb, te, rr = _i32(tok_begin), _i32(tok_end), _i32(rows)
    max_blocks = tables.shape[1] if tables.ndim == 2 else 0
    rc = lib().or_decode(_ptr(out), _ptr(lse), _ptr(wsum), _ptr(q), DT[q_dtype], _ptr(pool),
                         DT[kv_dtype], geom["num_blocks"], geom["num_layers"],
                         geom["num_kv_heads"], geom["block_size"], D, Hq, layer,
                         _ptr(tables), max_blocks, _ptr(seq_lens), B, float(scale),
                         float(k_scale), float(v_scale), _ptr(tb), _ptr(te), _ptr(rr),
                         0 if rr is None else rr.size, int(mutant), _f32(block_scales))
    if rc != 0:
        raise ValueError(f"oracle decode rejected its inputs (code {rc})")
    return out, lse, wsum


def decode_mq(q, q_dtype, pool, kv_dtype, geom, layer, tables, seq_lens, q_len, scale,
              k_scale=1.0, v_scale=1.0, block_scales=None):
    """fp64 causal attention of the last q_len tokens of every sequence over its
    paged K/V.  q [B, q_len, Hq, D] -> (out [B, q_len, Hq, D], lse [B, q_len, Hq])."""
    q = np.ascontiguousarray(q)
    pool = np.ascontiguousarray(pool)
    tables = _i32(tables)
    seq_lens = _i32(seq_lens)
    B = seq_lens.shape[0]
    Hq, D = geom["num_q_heads"], geom["head_dim"]
    out = np.empty((B, q_len, Hq, D))
    lse = np.empty((B, q_len, Hq))
    rc = lib().or_decode_mq(_ptr(out), _ptr(lse), _ptr(q), DT[q_dtype], _ptr(pool), DT[kv_dtype],
                            geom["num_blocks"], geom["num_layers"], geom["num_kv_heads"],
                            geom["block_size"], D, Hq, layer, _ptr(tables), tables.shape[1],
                            _ptr(seq_lens), B, int(q_len), float(scale), float(k_scale),
                            float(v_scale), _f32(block_scales))
    if rc != 0:
        raise ValueError(f"oracle decode_mq rejected its inputs (code {rc})")
    return out, lse


def append(pool, kv_dtype, geom, layer, k, v, in_dtype, tables, positions,
           k_scale=1.0, v_scale=1.0, block_scales=None):
    """[ENG26 2.2] append_token into `pool` (modified in place)."""
    tables = _i32(tables)
    positions = _i32(positions)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    rc = lib().or_append(_ptr(pool), DT[kv_dtype], geom["num_blocks"], geom["num_layers"],
                         geom["num_kv_heads"], geom["block_size"], geom["head_dim"], layer,
                         _ptr(k), _ptr(v), DT[in_dtype], _ptr(tables), tables.shape[1],
                         _ptr(positions), positions.shape[0], float(k_scale), float(v_scale),
                         _f32(block_scales))
    if rc != 0:
        raise ValueError(f"oracle append rejected its inputs (code {rc})")


def append_tokens(pool, kv_dtype, geom, layer, k, v, in_dtype, tables, seq_ids, positions,
                  k_scale=1.0, v_scale=1.0, block_scales=None):
    """Bulk append: token i -> sequence seq_ids[i], position positions[i]."""
    tables = _i32(tables)
    seq_ids = _i32(seq_ids)
    positions = _i32(positions)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    rc = lib().or_append_tokens(_ptr(pool), DT[kv_dtype], geom["num_blocks"],
                                geom["num_layers"], geom["num_kv_heads"], geom["block_size"],
                                geom["head_dim"], layer, _ptr(k), _ptr(v), DT[in_dtype],
                                _ptr(tables), tables.shape[1], tables.shape[0], _ptr(seq_ids),
                                _ptr(positions), seq_ids.shape[0], float(k_scale),
                                float(v_scale), _f32(block_scales))
    if rc != 0:
        raise ValueError(f"oracle append_tokens rejected its inputs (code {rc})")


def block_scales(scales, geom, layer, k, v, in_dtype, tables, seq_ids, positions,
                 group_tokens=0):
    """[UNLOCK 3.2] block-wise scales amax / 448 of the scale groups (group_tokens
    consecutive positions of a sequence; 0: one block) these tokens land in,
    written into the slot of every block of each group (`scales`, [NB, 2, L, Hkv]
    float32, modified in place)."""
    tables = _i32(tables)
    seq_ids = _i32(seq_ids)
    positions = _i32(positions)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    rc = lib().or_block_scales(_f32(scales), geom["num_blocks"], geom["num_layers"],
                               geom["num_kv_heads"], geom["block_size"], geom["head_dim"], layer,
                               _ptr(k), _ptr(v), DT[in_dtype], _ptr(tables), tables.shape[1],
                               tables.shape[0], _ptr(seq_ids), _ptr(positions), seq_ids.shape[0],
                               int(group_tokens))
    if rc != 0:
        raise ValueError(f"oracle block_scales rejected its inputs (code {rc})")


def merge(part_o, part_lse):
    """[SEQPAR incremental softmax] LSE merge.  part_o [R, S, D], part_lse [R, S]
    (fp64) -> (out [R, D], lse [R])."""
    part_o = np.ascontiguousarray(part_o, dtype=np.float64)
    part_lse = np.ascontiguousarray(part_lse, dtype=np.float64)
    R, S, D = part_o.shape
    out = np.empty((R, D))
    lse = np.empty((R,))
    lib().or_merge(_ptr(out), _ptr(lse), _ptr(part_o), _ptr(part_lse), R, S, D)
    return out, lse
