"""Failure detection on the GPU without a fault (needs a GPU): a bounded wait
that runs out is reported through the pool's status word as PKV_ETIMEOUT, the
kernel returns instead of spinning, and the context keeps computing correct
results afterwards."""
import time

import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, assert_parity, oracle_side

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_timeout_and_context_survives():
    from paged_kv_cache_215_gb300 import build
    build.build()
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("fail_small", [100, 37], 32, 8, 128, 16, "bf16", "bf16", "bf16", seed=95)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    assert gc.status() == 0
    t0 = time.perf_counter()
    gc.pool.wait_selftest()                     # a barrier nothing arrives on
    assert gc.status() == pkv.PKV_ETIMEOUT
    waited = time.perf_counter() - t0
    assert 0.5 < waited < 30, waited            # the 1 s bound, not a hang
    assert gc.status() == 0                     # reading the word cleared it
    pool, ref, seqs = oracle_side(case, tens, None)
    out = gc.step()
    torch.cuda.synchronize()
    assert gc.status() == 0
    assert_parity(case, out, ref, pool, seqs, 1.0, case.name)
