"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: sequence lengths, block-table entries (a seeded
permutation of the physical pool), logical per-token K/V values, the decode
query and the new token's k/v.  It holds none of the method's arithmetic: the
pool is filled by each side's own append path (the CUDA library on the GPU,
the oracle on the CPU), and nothing here computes slots, scores or encodings.

Shapes and value distributions follow the workloads the source pages discuss
(Llama-3-8B-like 32 query / 8 KV heads at head_dim 128; a 70B-like 64/8 shape;
block_size 16 and 32; 8K-average batches, 128K and 1M single requests):
  values        N(0, 1), drawn in fp32 and rounded to the storage dtype
  lengths       uniform integers, or log-uniform for the mixed 70B batch
  block ids     the first entries of a seeded permutation of the whole pool
  spikes        1% of token positions of a long request get K x 4 (all heads)
  shared prefix the first 4096 tokens' full blocks are one set of physical
                blocks referenced by every sequence's table
All draws come from torch.Generator objects seeded per case, on CPU or CUDA.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Case:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str                 # storage dtype of the pool: f32 | f16 | bf16 | e4m3
    q_dtype: str                  # dtype of q, k_new, v_new (bf16 values feed the E4M3 pool)
    out_dtype: str
    seq_lens: np.ndarray          # [B] int32, attention length after the step's append
    tables: np.ndarray            # [B, max_blocks] int32, -1 past the last used entry
    num_blocks: int
    num_layers: int = 1
    layer: int = 0
    seed: int = 0
    spike_frac: float = 0.0       # fraction of K rows scaled x4
    shared_prefix_tokens: int = 0
    shared_blocks: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks(self) -> int:
        return int(self.tables.shape[1])

    @property
    def geometry(self) -> dict:
        return dict(num_layers=self.num_layers, num_q_heads=self.num_q_heads,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    block_size=self.block_size, num_blocks=self.num_blocks)

    def kv_elem_bytes(self) -> int:
        return {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}[self.kv_dtype]

    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _build_tables(lens, bs, num_blocks, perm, shared_tokens=0):
    """Assign block ids from `perm` in order.  With shared_tokens > 0, the first
    floor(min(n, shared_tokens) / bs) entries of every table are one common
    list of blocks (the shared prefix); everything after is private."""
    B = len(lens)
    nblk = [(int(n) + bs - 1) // bs for n in lens]
    max_blocks = max(nblk) if B else 1
    tables = np.full((B, max(max_blocks, 1)), -1, dtype=np.int32)
    cursor = 0
    shared_full = shared_tokens // bs
    shared = np.asarray(perm[:shared_full], dtype=np.int32)
    cursor += shared_full
    for s in range(B):
        k = min(int(lens[s]), shared_tokens) // bs if shared_tokens else 0
        tables[s, :k] = shared[:k]
        rest = nblk[s] - k
        tables[s, k:nblk[s]] = perm[cursor:cursor + rest]
        cursor += rest
    return tables, cursor, shared


def make_case(name: str, seq_lens, num_q_heads, num_kv_heads, head_dim, block_size,
              kv_dtype, q_dtype, out_dtype, seed, pool_slack=0.10, spike_frac=0.0,
              shared_prefix_tokens=0, num_layers=1, layer=0) -> Case:
    lens = np.asarray(seq_lens, dtype=np.int32)
    bs = block_size
    need = sum((int(n) + bs - 1) // bs for n in lens)
    if shared_prefix_tokens:
        # blocks that every table shares are counted once
        sh = shared_prefix_tokens // bs
        need = sh + sum((int(n) + bs - 1) // bs - min(int(n), shared_prefix_tokens) // bs
                        for n in lens)
    num_blocks = max(int(math.ceil(need * (1.0 + pool_slack))), need, 1)
    perm = torch.randperm(num_blocks, generator=_gen(seed + 1000)).numpy().astype(np.int32)
    tables, used, shared = _build_tables(lens, bs, num_blocks, perm, shared_prefix_tokens)
    assert used <= num_blocks
    return Case(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, block_size=bs, kv_dtype=kv_dtype, q_dtype=q_dtype,
                out_dtype=out_dtype, seq_lens=lens, tables=tables, num_blocks=num_blocks,
                seed=seed, spike_frac=spike_frac, shared_prefix_tokens=shared_prefix_tokens,
                shared_blocks=shared, num_layers=num_layers, layer=layer)


# ---------------------------------------------------------------------------
# the five workload families, full size and scaled down for parity tests

def tiny_gqa2_d64_f32() -> Case:
    """2 sequences of 37 and 100 cached tokens plus one appended token each;
    4 query / 2 KV heads, head_dim 64, block_size 16, fp32, pool of 32 blocks."""
    lens = np.array([37 + 1, 100 + 1], dtype=np.int32)
    c = make_case("tiny_gqa2_d64_f32", lens, 4, 2, 64, 16, "f32", "f32", "f32", seed=1000)
    # a pool of exactly 32 blocks, ids from a seeded permutation of all 32
    perm = torch.randperm(32, generator=_gen(2000)).numpy().astype(np.int32)
    c.tables, _, _ = _build_tables(lens, 16, 32, perm)
    c.num_blocks = 32
    return c


def llama8b_batch(batch=32, lo=4096, hi=12288, seed=1001, block_size=16) -> Case:
    """32 query / 8 KV heads, head_dim 128, bf16, lengths uniform in [lo, hi]."""
    g = _gen(seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=g).numpy().astype(np.int32)
    return make_case(f"llama8b_decode_b{batch}_len{lo}-{hi}_bs{block_size}", lens, 32, 8, 128,
                     block_size, "bf16", "bf16", "bf16", seed=seed)


def long_context(tokens=131072, seed=1002, batch=1) -> Case:
    """Batch 1 (or `batch` such requests), 32 query / 8 KV heads, head_dim 128, bf16,
    1% of K rows x4."""
    return make_case(f"long_context_b{batch}_{tokens}", [tokens] * batch, 32, 8, 128, 16, "bf16",
                     "bf16", "bf16", seed=seed, spike_frac=0.01)


def fp8_batch(batch=8, tokens=32768, heads=(32, 8, 128), seed=1003) -> Case:
    """E4M3 pool with one fp32 scale per K and per V (amax / 448); bf16 q and out."""
    hq, hkv, d = heads
    return make_case(f"fp8_e4m3_b{batch}_{tokens}_h{hq}-{hkv}_d{d}", [tokens] * batch, hq, hkv,
                     d, 16, "e4m3", "bf16", "bf16", seed=seed)


def llama70b_prefix(batch=64, lo=512, hi=131072, block_size=16, prefix=4096, seed=1004) -> Case:
    """64 query / 8 KV heads, head_dim 128, bf16, lengths log-uniform in [lo, hi],
    the first `prefix` tokens' full blocks shared by every sequence."""
    g = _gen(seed)
    u = torch.rand((batch,), generator=g, dtype=torch.float64).numpy()
    lens = np.round(np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))).astype(np.int32)
    return make_case(f"llama70b_prefix_b{batch}_len{lo}-{hi}_bs{block_size}", lens, 64, 8, 128,
                     block_size, "bf16", "bf16", "bf16", seed=seed,
                     shared_prefix_tokens=prefix)


def llama8b_layers(num_layers=4, layer=2, batch=32, lo=4096, hi=12288, seed=1005) -> Case:
    """The 8B-shaped batch in a pool holding several layers; one layer is read."""
    g = _gen(seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=g).numpy().astype(np.int32)
    return make_case(f"llama8b_decode_b{batch}_len{lo}-{hi}_L{num_layers}_layer{layer}", lens, 32,
                     8, 128, 16, "bf16", "bf16", "bf16", seed=seed, num_layers=num_layers,
                     layer=layer)


def long_context_bs64(tokens=131072, seed=1006, batch=1) -> Case:
    """The 128K request in 64-token blocks."""
    return make_case(f"long_context_b{batch}_{tokens}_bs64", [tokens] * batch, 32, 8, 128, 64,
                     "bf16", "bf16", "bf16", seed=seed, spike_frac=0.01)


def shared_prefix_long(batch=32, prefix=65536, lo=64, hi=2048, seed=1010) -> Case:
    """Many requests over one long document: `batch` sequences whose first `prefix`
    tokens are one shared list of blocks, each followed by a private part of
    uniform [lo, hi] tokens; 32 query / 8 KV heads, head_dim 128, bf16, bs 16."""
    g = _gen(seed)
    lens = (prefix + torch.randint(lo, hi + 1, (batch,), generator=g)).numpy().astype(np.int32)
    return make_case(f"shared_prefix_{prefix // 1024}k_b{batch}", lens, 32, 8, 128, 16, "bf16",
                     "bf16", "bf16", seed=seed, shared_prefix_tokens=prefix)


def prefix_args(case: Case, used: Optional[int] = None):
    """(prefix table, prefix length, per-sequence prefix lengths) of a shared-prefix
    decode over the first `used` tokens (default all) of the case's shared blocks:
    sequence s uses min(n_s, used) rounded down to whole blocks."""
    bs = case.block_size
    used = case.shared_prefix_tokens if used is None else min(used, case.shared_prefix_tokens)
    used = used // bs * bs
    table = np.ascontiguousarray(case.shared_blocks[:used // bs]).astype(np.int32)
    lens = np.array([min(int(n), used) // bs * bs for n in case.seq_lens], dtype=np.int32)
    return table, used, lens


# Each full-size workload, drawn for `mult` times its batch (a data-parallel job
# over several GPUs draws one global batch of that many sequences and gives
# each GPU a share; mult = 1 is the single-GPU workload).
FULL = {
    "tiny": lambda mult=1: tiny_gqa2_d64_f32() if mult == 1 else make_case(
        f"tiny_x{mult}", [38, 101] * mult, 4, 2, 64, 16, "f32", "f32", "f32", seed=1000),
    "llama8b_b32_8k": lambda mult=1: llama8b_batch(batch=32 * mult),
    "long_128k": lambda mult=1: long_context(131072, batch=mult),
    "long_1m": lambda mult=1: long_context(1048576, batch=mult),
    "fp8_b8_32k": lambda mult=1: fp8_batch(batch=8 * mult),
    "llama70b_prefix_bs16": lambda mult=1: llama70b_prefix(batch=64 * mult, block_size=16),
    "llama70b_prefix_bs32": lambda mult=1: llama70b_prefix(batch=64 * mult, block_size=32),
    "long_128k_bs64": lambda mult=1: long_context_bs64(batch=mult),
    "llama8b_b32_8k_layers4": lambda mult=1: llama8b_layers(batch=32 * mult),
    "shared_prefix_64k_b32": lambda mult=1: shared_prefix_long(batch=32 * mult),
    # the 70B-shaped prefix batch with lengths 4K-8K (a 1.5 GB pool): the same
    # prefix pass (64 sequences x 8 query heads per KV head, a 4096-token prefix)
    # on a case small enough to profile
    "llama70b_prefix_small": lambda mult=1: llama70b_prefix(batch=64 * mult, lo=4096, hi=8192,
                                                           seed=1011),
}

# query tokens per sequence of the multi-token (speculative verification) measurements
MULTI_TOKEN = {"llama8b_b32_8k_q4": ("llama8b_b32_8k", 4)}


# ---------------------------------------------------------------------------
# tensors

@dataclass
class Tensors:
    k_tokens: torch.Tensor      # [T, Hkv, D] logical K of every cached token except each
    v_tokens: torch.Tensor      #   sequence's last one (which the decode step appends)
    tok_seq: torch.Tensor       # [T] int32 sequence index of each token
    tok_pos: torch.Tensor       # [T] int32 position of each token in its sequence
    q: torch.Tensor             # [B, Hq, D]
    k_new: torch.Tensor         # [B, Hkv, D] the last token of every sequence
    v_new: torch.Tensor
    new_pos: torch.Tensor       # [B] int32 = seq_lens - 1 (-1: an empty sequence, nothing to append)


def make_tensors(case: Case, device="cpu") -> Tensors:
    """Draw the logical K/V of every token, the query and the appended token.

    Tokens inside a shared prefix carry the same values in every sequence (they
    are the same physical blocks); everything else is drawn per sequence."""
    dev = torch.device(device)
    g = _gen(case.seed + 7, device=dev)
    B, Hkv, D, Hq = case.batch, case.num_kv_heads, case.head_dim, case.num_q_heads
    store = torch.bfloat16 if case.kv_dtype == "e4m3" else TORCH_DT[case.kv_dtype]
    lens = torch.as_tensor(case.seq_lens.astype(np.int64))
    T_all = int(lens.sum())
    P = case.shared_prefix_tokens
    if P:
        prefix_k = torch.randn((P, Hkv, D), generator=g, device=dev)
        prefix_v = torch.randn((P, Hkv, D), generator=g, device=dev)
    k_all = torch.randn((T_all, Hkv, D), generator=g, device=dev)
    v_all = torch.randn((T_all, Hkv, D), generator=g, device=dev)
    starts = torch.zeros(B + 1, dtype=torch.int64)
    starts[1:] = torch.cumsum(lens, 0)
    seq_of = torch.repeat_interleave(torch.arange(B), lens).to(dev)
    pos_of = (torch.arange(T_all) - torch.repeat_interleave(starts[:-1], lens)).to(dev)
    if P:
        in_prefix = pos_of < P
        k_all[in_prefix] = prefix_k[pos_of[in_prefix]]
        v_all[in_prefix] = prefix_v[pos_of[in_prefix]]
    if case.spike_frac > 0:
        gs = _gen(case.seed + 13)
        for s in range(B):
            n = int(case.seq_lens[s])
            k = int(math.floor(case.spike_frac * n))
            if k:
                rows = torch.randperm(n, generator=gs)[:k].to(dev) + int(starts[s])
                k_all[rows] *= 4.0
    k_all = k_all.to(store)
    v_all = v_all.to(store)
    qdt = TORCH_DT[case.q_dtype]
    q = torch.randn((B, Hq, D), generator=g, device=dev).to(qdt)
    nonempty = lens > 0
    last = (starts[1:] - 1).clamp(min=0).to(dev)
    keep = torch.ones(T_all, dtype=torch.bool, device=dev)
    keep[last[nonempty.to(dev)]] = False
    k_new = torch.zeros((B, Hkv, D), dtype=store, device=dev)
    v_new = torch.zeros((B, Hkv, D), dtype=store, device=dev)
    if T_all:
        ne = nonempty.to(dev)
        k_new[ne] = k_all[last[ne]]
        v_new[ne] = v_all[last[ne]]
    return Tensors(k_tokens=k_all[keep].contiguous(), v_tokens=v_all[keep].contiguous(),
                   tok_seq=seq_of[keep].to(torch.int32).contiguous(),
                   tok_pos=pos_of[keep].to(torch.int32).contiguous(),
                   q=q.contiguous(), k_new=k_new.contiguous(), v_new=v_new.contiguous(),
                   new_pos=(lens - 1).to(torch.int32).to(dev).contiguous())


def raw_numpy(t: torch.Tensor) -> np.ndarray:
    """Storage bytes of a tensor as a numpy array (bf16/f16 as uint16, fp8 as uint8)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.numpy()


def block_waste(case: Case) -> float:
    """Internal fragmentation of the tables: unused slots / allocated slots."""
    bs = case.block_size
    alloc = sum(((int(n) + bs - 1) // bs) * bs for n in case.seq_lens)
    return (alloc - case.total_tokens()) / max(alloc, 1)
