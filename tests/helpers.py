"""Test helpers: build the oracle's own pool from a workload and read results."""
import numpy as np
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl


def np_raw(t):
    return wl.raw_numpy(t)


def oracle_pool(case, tens, k_scale=1.0, v_scale=1.0, include_new=False):
    """The oracle's pool: zeros, then every cached token appended by the oracle."""
    eb = case.kv_elem_bytes()
    nbytes = oracle.kv_bytes(case.num_layers, case.num_kv_heads, case.head_dim,
                             case.num_blocks * case.block_size, eb)
    pool = np.zeros(nbytes, dtype=np.uint8)
    in_dt = "bf16" if case.kv_dtype == "e4m3" else case.kv_dtype
    oracle.append_tokens(pool, case.kv_dtype, case.geometry, case.layer, np_raw(tens.k_tokens),
                         np_raw(tens.v_tokens), in_dt, case.tables, np_raw(tens.tok_seq),
                         np_raw(tens.tok_pos), k_scale, v_scale)
    if include_new:
        oracle.append(pool, case.kv_dtype, case.geometry, case.layer, np_raw(tens.k_new),
                      np_raw(tens.v_new), in_dt, case.tables, np_raw(tens.new_pos),
                      k_scale, v_scale)
    return pool


def fp8_scales(tens):
    """The oracle's per-tensor scales of all K (resp. V) tokens: its amax over the
    cached tokens and the new ones, then its scale rule."""
    ks = []
    for a, b in ((tens.k_tokens, tens.k_new), (tens.v_tokens, tens.v_new)):
        amax = max(oracle.absmax(np_raw(a), "bf16"), oracle.absmax(np_raw(b), "bf16"))
        ks.append(oracle.fp8_scale(amax))
    return float(ks[0]), float(ks[1])


def logical_kv(case, tens):
    """Contiguous per-sequence K and V (fp64), straight from the generator's
    arrays: no pool, no table."""
    k = tens.k_tokens.double().cpu().numpy()
    v = tens.v_tokens.double().cpu().numpy()
    seq = tens.tok_seq.cpu().numpy()
    pos = tens.tok_pos.cpu().numpy()
    kn = tens.k_new.double().cpu().numpy()
    vn = tens.v_new.double().cpu().numpy()
    out = []
    for s in range(case.batch):
        n = int(case.seq_lens[s])
        K = np.zeros((n, case.num_kv_heads, case.head_dim))
        V = np.zeros_like(K)
        m = seq == s
        K[pos[m]] = k[m]
        V[pos[m]] = v[m]
        K[n - 1] = kn[s]
        V[n - 1] = vn[s]
        out.append((K, V))
    return out
