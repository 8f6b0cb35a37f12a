"""A call split by opts.phase (needs a GPU): phase 1 (the attention launches) then
phase 2 (the merge) on the same stream and workspace must give the output of
the whole call (phase 0) bit for bit, for the plain decode (balanced and fixed
split) and for the shared-prefix decode (prefix pass and plain routes), and
that output must match the fp64 oracle (max |err| <= 2e-3 x max|V|)."""
import pytest
import torch

from paged_kv_cache_215_gb300 import workloads as wl
from tests.gpu_harness import GpuCase, assert_parity, oracle_side

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_215_gb300 import build
    build.build()


@pytest.mark.parametrize("splits", [0, 3])
def test_decode_phases_compose_to_the_whole_call(splits):
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("phases_decode", [3000, 17, 1, 900], 32, 8, 128, 16, "bf16", "bf16",
                        "bf16", seed=170)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos)
    ws = torch.empty(pkv.workspace_bytes(gc.geom, case.batch, gc.max_seq_len, splits),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for phases in ((0,), (1, 2)):
        out = torch.full((case.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        for ph in phases:
            pkv.paged_decode_attention(out, gc.q, gc.pool, case.layer, gc.tables, gc.seq_lens,
                                       gc.max_seq_len, case.scale, num_splits=splits,
                                       workspace=ws, opts=pkv.launch_opts(phase=ph))
        torch.cuda.synchronize()
        assert gc.status() == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    assert_parity(case, outs[0], ref, pool, seqs, 1.0, f"decode phases splits {splits}",
                  out_dtype="bf16")


@pytest.mark.parametrize("route", [3, 2], ids=["prefix_pass", "plain"])
def test_shared_prefix_phases_compose_to_the_whole_call(route):
    from paged_kv_cache_215_gb300 import pkv
    case = wl.make_case("phases_casc", [1500, 300, 2600, 640], 32, 8, 128, 16, "bf16", "bf16",
                        "bf16", seed=171, shared_prefix_tokens=640)
    tens = wl.make_tensors(case)
    gc = GpuCase(case, tens)
    pool, ref, seqs = oracle_side(case, tens, None)
    gc.pool.append(case.layer, gc.k_new, gc.v_new, gc.tables, gc.new_pos)
    table, P, lens = wl.prefix_args(case)
    table = torch.from_numpy(table).cuda()
    lens = torch.from_numpy(lens).cuda()
    ws = torch.empty(pkv.cascade_workspace_bytes(gc.geom, case.batch, case.max_blocks,
                                                 gc.max_seq_len, P),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for phases in ((0,), (1, 2)):
        out = torch.full((case.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        for ph in phases:
            pkv.paged_decode_attention_cascade(out, gc.q, gc.pool, case.layer, table, P, lens,
                                               gc.tables, gc.seq_lens, gc.max_seq_len, case.scale,
                                               workspace=ws,
                                               opts=pkv.launch_opts(kernel=route, phase=ph))
        torch.cuda.synchronize()
        assert gc.status() == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    assert_parity(case, outs[0], ref, pool, seqs, 1.0, f"shared-prefix phases route {route}",
                  out_dtype="bf16")
