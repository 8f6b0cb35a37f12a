"""The decode entry point that allocates nothing (needs a GPU).

paged_decode_attention_static serves callers that cannot allocate device
memory when they run decode attention; its partial results live in a fixed
array inside the library.  Here it is called through the C ABI twice in a row,
with the automatic split and with a fixed split of three partitions per
sequence (so the array holds partials at different offsets from one call to
the next), and must match the fp64 oracle within the parity bound the other
GPU tests use (2e-3 x max|V| for bf16 KV, 5e-3 x max|V| for E4M3 KV) and agree
with paged_decode_attention given a caller-owned workspace.  A workspace
larger than the array must be refused with PKV_ENOMEM.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, TOL, assert_parity, oracle_side

pytestmark = pytest.mark.gpu


def _static_call(gc, out, num_splits=0):
    from paged_kv_cache_215_gb300 import pkv
    c = gc.case
    return pkv.lib().paged_decode_attention_static(
        out.data_ptr(), pkv.TORCH_CODE[out.dtype], gc.q.data_ptr(), pkv.TORCH_CODE[gc.q.dtype],
        gc.pool.handle, c.layer, gc.tables.data_ptr(), gc.tables.shape[1],
        gc.seq_lens.data_ptr(), c.batch, gc.max_seq_len, ctypes.c_float(c.scale),
        ctypes.c_float(gc.k_scale), ctypes.c_float(gc.v_scale), num_splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", [
    wl.llama8b_batch(batch=6, lo=300, hi=3000, seed=31),
    wl.make_case("fp8_static", [2500, 40, 1], 32, 8, 128, 16, "e4m3", "bf16", "bf16", seed=32),
    wl.llama70b_prefix(batch=5, lo=512, hi=9000, block_size=32, seed=33),
], ids=lambda c: c.name)
def test_static_scratch_matches_oracle_and_workspace_entry_point(case):
    from paged_kv_cache_215_gb300 import build
    build.build()
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    ws_out = gc.step(out_dtype="f32")                 # appends the new tokens; caller workspace
    assert_parity(case, ws_out, ref, pool, seqs, gc.v_scale, f"{case.name} workspace")
    vmax = max(float(gc.v_tokens.float().abs().max()), float(gc.v_new.float().abs().max()))
    bound = TOL[case.kv_dtype] * vmax
    # the automatic split, a fixed split, then the automatic split again: each call
    # finds what the previous one left in the shared array
    for splits in (0, 0, 3, 3, 0):
        out = torch.full_like(ws_out, float("nan"))
        assert _static_call(gc, out, splits) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert_parity(case, out, ref, pool, seqs, gc.v_scale, f"{case.name} static s{splits}")
        assert float((out - ws_out).abs().max()) <= bound
    assert gc.status() == 0


def test_static_scratch_rejects_oversized_workspace():
    from paged_kv_cache_215_gb300 import pkv
    # 4096 sequences x 64 query heads split 16 ways needs far more than the array holds
    g = pkv.geometry(1, 64, 8, 128, 16, 64, "bf16")
    pool = pkv.KVPool(g)
    need = pkv.workspace_bytes(g, 4096, 16 * 16, 16)
    assert need > 16 << 20
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = pkv.lib().paged_decode_attention_static(
        dummy.data_ptr(), pkv.PKV_F32, dummy.data_ptr(), pkv.PKV_BF16, pool.handle, 0,
        dummy.data_ptr(), 16, dummy.data_ptr(), 4096, 16 * 16, ctypes.c_float(0.1),
        ctypes.c_float(1.0), ctypes.c_float(1.0), 16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pkv.PKV_ENOMEM
