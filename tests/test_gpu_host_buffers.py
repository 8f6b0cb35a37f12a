"""Decode steps whose inputs and output live in pinned host memory (needs a GPU).

A serving loop on a Grace host can hand paged_decode_step host buffers directly:
the attention kernel reads q, the new token's k and v and the lengths from
pinned host memory over the CPU-GPU link, and the merge (or the attention
kernel, for a sequence one CTA covers) writes out there; the workspace the
binding allocates stays on the pool's device.  The result must be the
device-buffer result bit for bit, and match the fp64 oracle within the parity
bound (2e-3 x max|V| for 16-bit KV, 5e-3 x max|V| for E4M3), for plain and
programmatic-dependent launches, on bf16, f16 and E4M3 pools, with sequences
that span many CTAs and sequences of 1 and 40 tokens that one CTA covers.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, assert_parity, oracle_side

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("case", [
    wl.llama8b_batch(batch=5, lo=200, hi=3000, seed=61),
    wl.make_case("host_f16", [6000, 40, 1], 32, 8, 128, 16, "f16", "f16", "f16", seed=62),
    wl.make_case("host_fp8", [2500, 40, 1], 32, 8, 128, 16, "e4m3", "bf16", "bf16", seed=64),
    wl.make_case("host_long", [20000], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=63),
], ids=lambda c: getattr(c, "name", str(c)))
def test_host_inputs_and_output_match_device_buffers(case, pdl):
    from paged_kv_cache_215_gb300 import build, pkv
    build.build()
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    opts = pkv.launch_opts(pdl=pdl)
    dev_out = gc.fused_step(out_dtype="f32", opts=opts)
    torch.cuda.synchronize()
    pin = lambda x: x.detach().cpu().contiguous().pin_memory()
    hq, hk, hv = pin(gc.q), pin(gc.k_new), pin(gc.v_new)
    hl = torch.from_numpy(case.seq_lens).pin_memory()
    host_out = torch.full(dev_out.shape, float("nan"), dtype=torch.float32).pin_memory()
    for _ in range(3):                       # the same token stored again each time
        pkv.paged_decode_step(host_out, hq, hk, hv, gc.pool, case.layer, gc.tables, hl,
                              gc.max_seq_len, case.scale, gc.k_scale, gc.v_scale, opts=opts)
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert torch.equal(host_out, dev_out.cpu())
    pool, ref, seqs = oracle_side(case, tens, None, gc.k_scale, gc.v_scale)
    assert_parity(case, host_out, ref, pool, seqs, gc.v_scale, f"{case.name} host buffers")

