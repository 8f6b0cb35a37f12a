"""Decode across GPUs: which GPU owns which sequences, key ranges or heads.

Decode attention of one sequence reads only that sequence's blocks, so a batch
splits across GPUs by sequence with no exchange between them: each GPU holds
its sequences' blocks in its own pool, runs the whole step (append, attention,
merge) on them, and returns their outputs.  The only host-side decision is the
split; this module makes it: contiguous ranges of the global batch, cut at the
token-count quantiles so that every GPU reads about the same KV bytes (the
quantity the step's time follows), every sequence owned by exactly one rank.
Two splits with one exchange each are here too: a long sequence's keys cut
into block-aligned ranges (an all-gather of the partial outputs and their
log-sum-exp, then the merge), and the KV heads cut into ranges (an all-gather
of the outputs, concatenated along the heads).
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

from . import workloads as wl


def partition(seq_lens, world: int) -> List[Tuple[int, int]]:
    """Contiguous [lo, hi) ranges of sequences, one per rank, covering the batch
    once.  Rank r takes the sequences whose first token lies in the r-th
    1/world of all tokens (a sequence straddling a cut goes to the rank its
    start falls in); with no tokens at all, equal sequence counts."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    B = int(lens.shape[0])
    if world < 1:
        raise ValueError("world must be >= 1")
    total = int(lens.sum())
    if total == 0:
        cuts = [B * r // world for r in range(world + 1)]
    else:
        starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
        # first sequence whose start reaches r * total / world (exact integer test)
        cuts = [int(np.searchsorted(starts * world, r * total, side="left"))
                for r in range(world)] + [B]
        cuts[0] = 0
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def shard(case: "wl.Case", lo: int, hi: int) -> "wl.Case":
    """The sub-batch [lo, hi) of a case as a case of its own, for one rank: the
    sequences keep their lengths (and their shared prefix, if any), and get a
    pool and tables of the rank's own.  The whole batch is returned as is."""
    if lo == 0 and hi == case.batch:
        return case
    return wl.make_case(f"{case.name}_seqs{lo}-{hi}", case.seq_lens[lo:hi], case.num_q_heads,
                        case.num_kv_heads, case.head_dim, case.block_size, case.kv_dtype,
                        case.q_dtype, case.out_dtype, seed=case.seed + 7919 * (lo + 1),
                        spike_frac=case.spike_frac,
                        shared_prefix_tokens=case.shared_prefix_tokens,
                        num_layers=case.num_layers, layer=case.layer)


def rank_case(name: str, rank: int, world: int) -> "wl.Case":
    """Rank `rank`'s share of the global batch of workload `name` at `world` GPUs
    (weak scaling: the global batch is `world` times the single-GPU one)."""
    glob = wl.FULL[name](world)
    lo, hi = partition(glob.seq_lens, world)[rank]
    return shard(glob, lo, hi)


# ---------------------------------------------------------------------------
# One long sequence across GPUs: every rank holds a contiguous key range of it
# and attends over that range alone; the partial results meet once.

def key_ranges(n: int, world: int, block_size: int) -> List[Tuple[int, int]]:
    """Block-aligned contiguous [lo, hi) ranges of a sequence's n keys, one per
    rank (rank r: blocks [r * nb / world, (r + 1) * nb / world)), covering every
    key once; a rank may get an empty range.  Rank r holds its keys at local
    positions 0 .. hi - lo of its own tables."""
    if world < 1 or block_size < 1 or n < 0:
        raise ValueError("need world >= 1, block_size >= 1 and n >= 0")
    nb = (int(n) + block_size - 1) // block_size
    cuts = [min(int(n), (r * nb // world) * block_size) for r in range(world)] + [int(n)]
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def gather_and_merge(o_local, lse_local, merge, out, group=None):
    """The exchange of a key-range split ("Sequence-parallel engineering for
    long-context LLM inference", numerically stable incremental softmax, and its
    communication-cost section: one gather of every rank's partial output and
    log-sum-exp): all-gather this rank's fp32 partial o_local [B, H, D] and
    lse_local [B, H], stack them as [B, H, ranks, D] and [B, H, ranks], and let
    `merge(out, part_o, part_lse)` combine them (the library's merge_partials on
    GPUs).  Every rank ends with the whole result in `out`."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    os_ = [torch.empty_like(o_local) for _ in range(world)]
    ls_ = [torch.empty_like(lse_local) for _ in range(world)]
    dist.all_gather(os_, o_local.contiguous(), group=group)
    dist.all_gather(ls_, lse_local.contiguous(), group=group)
    part_o = torch.stack(os_, dim=2).contiguous()
    part_lse = torch.stack(ls_, dim=2).contiguous()
    return merge(out, part_o, part_lse)


# ---------------------------------------------------------------------------
# KV heads across GPUs: every rank holds all sequences' blocks for a contiguous
# range of KV heads (and attends with the query heads that read them); the
# outputs of the ranks are concatenated along the head dimension.

def head_ranges(num_kv_heads: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous [lo, hi) KV-head ranges of equal size, one per rank; rank r
    serves query heads [lo * G, hi * G) (query head h reads KV head h // G).
    num_kv_heads must be a multiple of world."""
    if world < 1 or num_kv_heads % world:
        raise ValueError("num_kv_heads must be a positive multiple of world")
    per = num_kv_heads // world
    return [(r * per, (r + 1) * per) for r in range(world)]


def gather_heads(o_local, out, group=None):
    """The exchange of the head split: all-gather every rank's output for its
    query heads, o_local [B, Hq / world, D], and concatenate them in rank order
    into out [B, Hq, D].  Every rank ends with the whole result."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(o_local) for _ in range(world)]
    dist.all_gather(parts, o_local.contiguous(), group=group)
    out.copy_(torch.cat(parts, dim=1))
    return out
