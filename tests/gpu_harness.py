"""Drive the CUDA library through its binding for a workload, and build the
oracle's side of the same workload from the same generator tensors."""
import numpy as np
import torch

import oracle
from paged_kv_cache_215_gb300 import workloads as wl
from tests.helpers import np_raw

# Parity bounds on max |gpu - oracle| relative to max |V| of the sequence.
TOL = {"f32": 2e-3, "f16": 2e-3, "bf16": 2e-3, "e4m3": 5e-3}
OUT_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


class GpuCase:
    """A pool on the GPU filled through the library's own append path."""

    def __init__(self, case, tens=None, device="cuda", fill_byte=0):
        from paged_kv_cache_215_gb300 import pkv
        self.pkv = pkv
        self.case = case
        self.tens = tens if tens is not None else wl.make_tensors(case, device=device)
        t = self.tens
        mv = lambda x: x.to(device).contiguous()
        self.k_tokens, self.v_tokens = mv(t.k_tokens), mv(t.v_tokens)
        self.tok_seq, self.tok_pos = mv(t.tok_seq), mv(t.tok_pos)
        self.q, self.k_new, self.v_new, self.new_pos = mv(t.q), mv(t.k_new), mv(t.v_new), mv(t.new_pos)
        g = case
        self.geom = pkv.geometry(g.num_layers, g.num_q_heads, g.num_kv_heads, g.head_dim,
                                 g.block_size, g.num_blocks, g.kv_dtype)
        nbytes = pkv.kv_pool_bytes(self.geom)
        storage = torch.full((nbytes,), fill_byte, dtype=torch.uint8, device=device)
        self.pool = pkv.KVPool(self.geom, storage=storage)
        ids = case.tables[case.tables >= 0]
        uniq, counts = np.unique(ids, return_counts=True)
        self.pool.reserve(uniq.tolist())
        extra = np.repeat(uniq, counts - 1)
        if extra.size:
            self.pool.share(extra.tolist())
        self.tables = torch.from_numpy(case.tables).to(device)
        self.seq_lens = torch.from_numpy(case.seq_lens).to(device)
        self.max_seq_len = int(case.seq_lens.max()) if case.batch else 0
        self.k_scale = self.v_scale = 1.0
        if case.kv_dtype == "e4m3":
            # the library's per-tensor scales over the cached and the new tokens
            self.k_scale, self.v_scale = pkv.fp8_scales((self.k_tokens, self.k_new),
                                                        (self.v_tokens, self.v_new))
        if self.tok_seq.numel():
            self.pool.append_tokens(case.layer, self.k_tokens, self.v_tokens, self.tables,
                                    self.tok_seq, self.tok_pos, self.k_scale, self.v_scale)

    def fused_step(self, out_dtype="f32", num_splits=0, opts=None):
        """One decode step through paged_decode_step (store + attention in one launch)."""
        c = self.case
        out = torch.full((c.batch, c.num_q_heads, c.head_dim), float("nan"),
                         dtype=OUT_DT[out_dtype], device=self.q.device)
        self.pkv.paged_decode_step(out, self.q, self.k_new, self.v_new, self.pool, c.layer,
                                   self.tables, self.seq_lens, self.max_seq_len, c.scale,
                                   self.k_scale, self.v_scale, num_splits=num_splits, opts=opts)
        return out

    def step(self, out_dtype="f32", num_splits=0, opts=None, append=True):
        """One decode step: append the last token of every sequence, then attend."""
        c = self.case
        if append and c.batch:
            self.pool.append(c.layer, self.k_new, self.v_new, self.tables, self.new_pos,
                             self.k_scale, self.v_scale)
        out = torch.full((c.batch, c.num_q_heads, c.head_dim), float("nan"),
                         dtype=OUT_DT[out_dtype], device=self.q.device)
        self.pkv.paged_decode_attention(out, self.q, self.pool, c.layer, self.tables,
                                        self.seq_lens, self.max_seq_len, c.scale, self.k_scale,
                                        self.v_scale, num_splits=num_splits, opts=opts)
        return out

    def status(self):
        return self.pool.check_status()


def oracle_side(case, tens, seqs=None, k_scale=1.0, v_scale=1.0):
    """The oracle's pool (only the tokens of `seqs` when given) and its fp64
    result for every head of those sequences."""
    t = tens
    tok_seq = t.tok_seq.cpu()
    if seqs is None:
        keep = torch.ones_like(tok_seq, dtype=torch.bool)
        seqs = list(range(case.batch))
    else:
        keep = torch.isin(tok_seq, torch.tensor(seqs, dtype=tok_seq.dtype))
    eb = case.kv_elem_bytes()
    nbytes = oracle.kv_bytes(case.num_layers, case.num_kv_heads, case.head_dim,
                             case.num_blocks * case.block_size, eb)
    pool = np.zeros(nbytes, dtype=np.uint8)
    in_dt = "bf16" if case.kv_dtype == "e4m3" else case.kv_dtype
    kc = t.k_tokens.cpu()[keep]
    vc = t.v_tokens.cpu()[keep]
    oracle.append_tokens(pool, case.kv_dtype, case.geometry, case.layer, np_raw(kc), np_raw(vc),
                         in_dt, case.tables, np_raw(tok_seq[keep]), np_raw(t.tok_pos.cpu()[keep]),
                         k_scale, v_scale)
    sel = torch.tensor(seqs, dtype=torch.long)
    tab = case.tables[seqs]
    oracle.append(pool, case.kv_dtype, case.geometry, case.layer, np_raw(t.k_new.cpu()[sel]),
                  np_raw(t.v_new.cpu()[sel]), in_dt, tab, np_raw(t.new_pos.cpu()[sel]),
                  k_scale, v_scale)
    # full query array; rows restricted to the chosen sequences
    rows = np.concatenate([np.arange(s * case.num_q_heads, (s + 1) * case.num_q_heads)
                           for s in seqs]).astype(np.int32) if seqs else np.zeros(0, np.int32)
    out, lse, wsum = oracle.decode(np_raw(t.q.cpu()), case.q_dtype, pool, case.kv_dtype,
                                   case.geometry, case.layer, case.tables, case.seq_lens,
                                   case.scale, k_scale, v_scale, rows=rows)
    return pool, out, seqs


def vmax_per_seq(case, pool, seqs, v_scale):
    """max |V| (dequantised) over the tokens each sequence attends to, read from
    the oracle's pool through the tables."""
    dt = case.kv_dtype
    vals = oracle.to_f64(pool, dt, v_scale if dt == "e4m3" else 1.0)
    p = vals.reshape(case.num_blocks, 2, case.num_layers, case.num_kv_heads, case.block_size,
                     case.head_dim)
    res = {}
    for s in seqs:
        n = int(case.seq_lens[s])
        if n == 0:
            res[s] = 0.0                                  # nothing attended: output must be 0
            continue
        nb = (n + case.block_size - 1) // case.block_size
        blocks = case.tables[s, :nb]
        v = p[blocks, 1, case.layer]                      # [nb, Hkv, bs, D]
        v = v.transpose(0, 2, 1, 3).reshape(nb * case.block_size, case.num_kv_heads, -1)[:n]
        res[s] = float(np.abs(v).max()) if n else 0.0
    return res


def assert_parity(case, gpu_out, ref_out, pool, seqs, v_scale, what="", out_dtype="f32"):
    tol = TOL[case.kv_dtype]
    vm = vmax_per_seq(case, pool, seqs, v_scale)
    got = gpu_out.double().cpu().numpy()
    worst = 0.0
    for s in seqs:
        err = np.abs(got[s] - ref_out[s])
        bound = np.full_like(err, tol * vm[s])
        if out_dtype != "f32":
            # plus the rounding of the exact value to the output dtype (half an ulp)
            ulp = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}[out_dtype]
            bound = bound + ulp * np.abs(ref_out[s])
        assert np.all(np.isfinite(got[s])), f"{what}: non-finite output for sequence {s}"
        ratio = float(np.max(err / np.maximum(bound, 1e-30))) if err.size else 0.0
        worst = max(worst, ratio)
        assert np.all(err <= bound), \
            f"{what}: seq {s} max err {err.max():.3e} > bound ({tol} x max|V| {vm[s]:.3f})"
    return worst
