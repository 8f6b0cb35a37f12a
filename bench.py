"""Benchmark: paged decode attention over a PagedAttention KV cache on GB300.

One step = one decode step of one layer: append the new token's k/v of every
sequence into its pool slot, then paged decode attention over all cached
tokens (the split-KV attention kernel and the log-sum-exp merge).  Inputs are
seeded synthetic tensors resident in HBM; the KV pool of the headline workload
(537 MB) is far larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: one global batch of N times the single-GPU workload
is split by sequence across the ranks (paged_kv_cache_215_gb300.dp: contiguous
ranges balanced by token count; decode has no exchange between sequences), the
time is the max over ranks and `value` is the sum of all ranks' KV bytes over
that time (weak scaling).
`--impl reference` times the fp64 CPU oracle on the host cores instead.
Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

from paged_kv_cache_215_gb300 import dp
from paged_kv_cache_215_gb300 import workloads as wl

METRIC = "paged decode attn KV GB/s (fraction of HBM peak); decode tokens/s at 128K"
UNIT = "GB/s"
PRIMARY = "long_128k"
SECONDARY = ["llama8b_b32_8k", "long_1m", "fp8_b8_32k", "llama70b_prefix_bs16",
             "llama70b_prefix_bs32", "long_128k_bs64", "llama8b_b32_8k_layers4"]
MODEL_LAYERS = {"long_128k": 32, "long_1m": 32, "llama8b_b32_8k": 32, "fp8_b8_32k": 32,
                "llama70b_prefix_bs16": 80, "llama70b_prefix_bs32": 80, "long_128k_bs64": 32,
                "llama8b_b32_8k_layers4": 32, "llama70b_prefix_small": 80,
                "shared_prefix_64k_b32": 32, "tiny": 1}
KERNEL_SOURCES = ["paged_kv_cache_215_gb300/csrc/decode_mma.cu",
                  "paged_kv_cache_215_gb300/csrc/decode_mma.cuh",
                  "paged_kv_cache_215_gb300/csrc/decode_mma_bf16.cu",
                  "paged_kv_cache_215_gb300/csrc/decode_mma_fp8.cu",
                  "paged_kv_cache_215_gb300/csrc/device.cuh"]


# ---------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """dram bytes per launch of the attention kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"decode_mma_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_hash():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.2)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l.split(", ") for l in self.lines if l and l[0].isdigit()]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def kv_bytes(case):
    return int(case.seq_lens.astype(np.int64).sum()) * 2 * case.num_kv_heads * case.head_dim * \
        case.kv_elem_bytes()


def algorithmic_attn_bytes(case):
    """What one decode-step attention launch must move: every cached K/V element
    once, q in, out, the table entries it follows, and the new token's k/v in and
    stored."""
    q = case.batch * case.num_q_heads * case.head_dim * 2
    out = case.batch * case.num_q_heads * case.head_dim * 2
    tables = sum((int(n) + case.block_size - 1) // case.block_size for n in case.seq_lens) * 4
    new = case.batch * 2 * case.num_kv_heads * case.head_dim * (2 + case.kv_elem_bytes())
    return kv_bytes(case) + q + out + tables + new


def algorithmic_unique_bytes(case):
    """algorithmic_attn_bytes with every shared block counted once: what one
    launch must read from HBM at the least."""
    return algorithmic_attn_bytes(case) - kv_bytes(case) + unique_kv_bytes(case)


def unique_kv_bytes(case):
    if not case.shared_prefix_tokens:
        return kv_bytes(case)
    bs = case.block_size
    per_tok = 2 * case.num_kv_heads * case.head_dim * case.kv_elem_bytes()
    shared = [min(int(n), case.shared_prefix_tokens) // bs * bs for n in case.seq_lens]
    dup = sum(shared) - max(shared)
    return kv_bytes(case) - dup * per_tok


# ---------------------------------------------------------------------------- our arm
class Workload:
    def __init__(self, name, device, case=None):
        from paged_kv_cache_215_gb300 import pkv
        self.pkv = pkv
        self.name = name
        self.case = case if case is not None else wl.FULL[name]()
        c = self.case
        self.tens = wl.make_tensors(c, device=device)
        t = self.tens
        self.geom = pkv.geometry(c.num_layers, c.num_q_heads, c.num_kv_heads, c.head_dim,
                                 c.block_size, c.num_blocks, c.kv_dtype)
        self.pool = pkv.KVPool(self.geom, device=device)
        self.pool.storage.zero_()
        ids = c.tables[c.tables >= 0]
        uniq, counts = np.unique(ids, return_counts=True)
        self.pool.reserve(uniq.tolist())
        if (counts > 1).any():
            self.pool.share(np.repeat(uniq, counts - 1).tolist())
        self.tables = torch.from_numpy(c.tables).to(device)
        self.seq_lens = torch.from_numpy(c.seq_lens).to(device)
        self.max_len = int(c.seq_lens.max())
        self.ks = self.vs = 1.0
        if c.kv_dtype == "e4m3":
            self.ks, self.vs = pkv.fp8_scales((t.k_tokens, t.k_new), (t.v_tokens, t.v_new))
        self.pool.append_tokens(c.layer, t.k_tokens, t.v_tokens, self.tables, t.tok_seq,
                                t.tok_pos, self.ks, self.vs)
        # the logical token arrays are no longer needed on the device
        self.tens.k_tokens = self.tens.v_tokens = None
        self.out = torch.empty(c.batch, c.num_q_heads, c.head_dim,
                               dtype=wl.TORCH_DT[c.out_dtype], device=device)
        nb = pkv.workspace_bytes(self.geom, c.batch, self.max_len, 0)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=device)
        self.o_attn = pkv.launch_opts(phase=1)
        self.o_attn_pdl = pkv.launch_opts(phase=1, pdl=1)
        self.o_merge = pkv.launch_opts(phase=2)
        torch.cuda.synchronize()

    def step(self, opts=None, q=None, k=None, v=None, seq_lens=None):
        """One decode step: store every sequence's new token and attend (one attention
        launch with the store fused in, plus the merge)."""
        c = self.case
        t = self.tens
        self.pkv.paged_decode_step(self.out, t.q if q is None else q, t.k_new if k is None else k,
                                   t.v_new if v is None else v, self.pool, c.layer, self.tables,
                                   self.seq_lens if seq_lens is None else seq_lens, self.max_len,
                                   c.scale, self.ks, self.vs, 0, self.ws, opts)

    def close(self):
        self.pool.close()


def time_steps(w, steps, warmup, split_phases=False, graph_chunk=0):
    """Warm-up, then `steps` timed decode steps on the current stream.

    split_phases: launch the attention kernel (phase 1) and the merge (phase 2)
    separately, with events around each attention launch (for the roofline).
    graph_chunk > 0: capture that many consecutive steps (chained with
    programmatic dependent launch) in one CUDA graph and replay it.
    Returns (total ms, per-step attention ms list, launches per step)."""
    from paged_kv_cache_215_gb300 import pkv
    stream = torch.cuda.current_stream()
    pdl = pkv.launch_opts(pdl=1)
    for _ in range(warmup):
        w.step(pdl)
    torch.cuda.synchronize()
    n0 = pkv.launch_count()
    w.step(pdl)
    torch.cuda.synchronize()
    per_step = pkv.launch_count() - n0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps if split_phases else 0)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph_chunk:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            w.step(pdl)                     # first call outside capture (one-time set-up)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for _ in range(graph_chunk):
                w.step(pdl)
        reps = max(1, steps // graph_chunk)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) * steps / (reps * graph_chunk), [], per_step
    start.record(stream)
    for i in range(steps):
        if split_phases:
            ev[i][0].record(stream)
            w.step(w.o_attn)
            ev[i][1].record(stream)
            w.step(w.o_merge)
        else:
            w.step(pdl)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end), [a.elapsed_time(b) for a, b in ev], per_step


def time_attention_graph(w, steps, chunk=10):
    """The attention kernel alone, as it runs inside the step: `chunk` launches
    chained with programmatic dependent launch, captured in one CUDA graph and
    replayed; milliseconds per launch."""
    stream = torch.cuda.current_stream()
    for _ in range(3):
        w.step(w.o_attn_pdl)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(chunk):
            w.step(w.o_attn_pdl)
    reps = max(1, steps // chunk)
    g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        g.replay()
    e.record(stream)
    torch.cuda.synchronize()
    del g
    return s.elapsed_time(e) / (reps * chunk)


def time_e2e(w, steps, warmup):
    """Through the C ABI from pinned host memory, every step: the host->device copy
    of that step's inputs (q, the new k and v, the lengths, packed in one pinned
    staging buffer the way a serving loop stages them), the decode step (store +
    attention + merge, its launches chained with programmatic dependent launch),
    and the device->host copy of its output.  Steps are pipelined over two
    staging slots and two output buffers on three streams: step i+1's inputs
    travel while step i computes, and step i's output travels while step i+1
    computes; each slot is reused only after the step that last used it has
    finished with it.  Ten steps are captured in one CUDA graph and replayed.
    Byte counts are the staging buffer and the output, per step."""
    c = w.case
    t = w.tens
    parts = {k: getattr(t, k).contiguous() for k in ("q", "k_new", "v_new")}
    parts["seq_lens"] = torch.from_numpy(c.seq_lens).to(w.seq_lens.device)
    offs, total = {}, 0
    for k, v in parts.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    hosts, devs, views, outs, outs_h = [], [], [], [], []
    for _ in range(2):
        host = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k, v in parts.items():
            nb = v.numel() * v.element_size()
            host[offs[k]:offs[k] + nb].copy_(v.cpu().contiguous().view(torch.uint8).reshape(-1))
        dev = torch.empty(total, dtype=torch.uint8, device="cuda")
        hosts.append(host)
        devs.append(dev)
        views.append({k: dev[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype)
                      .view(v.shape) for k, v in parts.items()})
        outs.append(torch.empty_like(w.out))
        outs_h.append(torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory())
    h2d = total
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ev_in = [ev(), ev()]        # slot's inputs are on the device
    ev_done = [ev(), ev()]      # slot's step finished (inputs read, output written)
    ev_out = [ev(), ev()]       # slot's output is on the host
    pdl = w.pkv.launch_opts(pdl=1)
    saved_out = w.out

    def step(i, first, comp):
        k = i % 2
        with torch.cuda.stream(s_in):
            if not first[k]:
                s_in.wait_event(ev_done[k])
            devs[k].copy_(hosts[k], non_blocking=True)
            ev_in[k].record(s_in)
        comp.wait_event(ev_in[k])
        if not first[k]:
            comp.wait_event(ev_out[k])
        w.out = outs[k]
        v = views[k]
        w.step(pdl, q=v["q"], k=v["k_new"], v=v["v_new"], seq_lens=v["seq_lens"])
        ev_done[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[k])
            outs_h[k].copy_(outs[k], non_blocking=True)
            ev_out[k].record(s_out)
        first[k] = False

    def run(n):
        # the copy streams fork from the stream that runs the steps (the capture
        # stream inside a graph capture) and join it again at the end
        comp = torch.cuda.current_stream()
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        first = [True, True]
        for i in range(n):
            step(i, first, comp)
        comp.wait_event(ev_out[0])
        comp.wait_event(ev_out[1])

    for _ in range(warmup):
        run(2)
    torch.cuda.synchronize()
    chunk = 10
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(chunk)
    reps = max(1, steps // chunk)
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        graph.replay()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / (reps * chunk)
    del graph
    w.out = saved_out
    return ms, h2d, d2h


def time_e2e_zero_copy(w, steps, warmup, slots=3):
    """Through the C ABI with every step's inputs in pinned host memory and its
    output written to pinned host memory: the attention kernel reads q, the new
    k and v and the lengths over the CPU-GPU link (NVLink-C2C on a Grace host)
    and the merge writes out there, so no copy operation sits between the
    launches and consecutive steps stay chained with programmatic dependent
    launch.  `slots` sets of host buffers rotate; ten steps are captured in one
    CUDA graph, and eager launches are timed too (the faster is returned, with its
    name).  Bytes per step: the input tensors read and the output written."""
    c = w.case
    t = w.tens
    pin = lambda x: x.detach().cpu().contiguous().pin_memory()
    ins = [{"q": pin(t.q), "k": pin(t.k_new), "v": pin(t.v_new),
            "seq_lens": torch.from_numpy(c.seq_lens).pin_memory()} for _ in range(slots)]
    outs = [torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory() for _ in range(slots)]
    h2d = sum(x.numel() * x.element_size() for x in ins[0].values())
    d2h = outs[0].numel() * outs[0].element_size()
    pdl = w.pkv.launch_opts(pdl=1)
    saved_out = w.out

    def run(n):
        for i in range(n):
            k = i % slots
            w.out = outs[k]
            w.step(pdl, q=ins[k]["q"], k=ins[k]["k"], v=ins[k]["v"], seq_lens=ins[k]["seq_lens"])

    for _ in range(warmup):
        run(slots)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    chunk = 10
    reps = max(1, steps // chunk)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        run(chunk)
    e.record(stream)
    torch.cuda.synchronize()
    eager = s.elapsed_time(e) / (reps * chunk)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(chunk)
    graph.replay()
    torch.cuda.synchronize()
    s.record(stream)
    for _ in range(reps):
        graph.replay()
    e.record(stream)
    torch.cuda.synchronize()
    replay = s.elapsed_time(e) / (reps * chunk)
    del graph
    w.out = saved_out
    return (eager, "eager launches") if eager <= replay else (replay, "cuda-graph replay"), h2d, d2h


def cpu_baseline(w, budget_s=15.0):
    """The fp64 oracle, as it stands, on this host's cores: a bounded sample of
    query rows of the same workload (its own pool built by its own append)."""
    import oracle
    c = w.case
    tens = wl.make_tensors(c, device="cuda")
    raw = wl.raw_numpy
    eb = c.kv_elem_bytes()
    pool = np.zeros(oracle.kv_bytes(c.num_layers, c.num_kv_heads, c.head_dim,
                                    c.num_blocks * c.block_size, eb), dtype=np.uint8)
    in_dt = "bf16" if c.kv_dtype == "e4m3" else c.kv_dtype
    oracle.append_tokens(pool, c.kv_dtype, c.geometry, c.layer, raw(tens.k_tokens),
                         raw(tens.v_tokens), in_dt, c.tables, raw(tens.tok_seq), raw(tens.tok_pos),
                         w.ks, w.vs)
    q = raw(tens.q)
    del tens
    rows_all = c.batch * c.num_q_heads
    per_row_bytes = kv_bytes(c) / rows_all
    done_rows, spent, n = 0, 0.0, max(1, oracle.num_threads())
    while spent < budget_s:
        rows = (np.arange(done_rows, done_rows + n) % rows_all).astype(np.int32)
        t0 = time.perf_counter()
        oracle.decode(q, c.q_dtype, pool, c.kv_dtype, c.geometry, c.layer, c.tables, c.seq_lens,
                      c.scale, w.ks, w.vs, rows=rows)
        spent += time.perf_counter() - t0
        done_rows += rows.size
    gbs = done_rows * per_row_bytes / spent / 1e9
    return {"value": gbs, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done_rows} (sequence, query head) rows (the workload has {rows_all}), "
                      f"fp64, {spent:.1f} s; GB/s counts each row's share of the KV bytes"}


def measure(name, steps, warmup, device, with_clocks=False, gpu_index=0, e2e=True, graph=True,
            case=None):
    w = Workload(name, device, case)
    c = w.case
    peak, peak_kind = peaks()
    sampler = ClockSampler(gpu_index) if with_clocks else None
    # headline: the production step -- fused store + attention, then the merge,
    # consecutive steps chained with programmatic dependent launch
    if sampler:
        sampler.start()
    eager_ms, _, per_step = time_steps(w, steps, warmup)
    graph_ms = time_steps(w, steps, 3, graph_chunk=10)[0] if graph else None
    clocks = sampler.stop() if sampler else None
    # the attention kernel alone: back to back inside a CUDA graph (as in the
    # step), and per launch with events around it on its stream
    attn_graph_ms = time_attention_graph(w, steps) if graph else None
    _, attn, _ = time_steps(w, steps, 3, split_phases=True)
    eager = eager_ms / steps
    gstep = graph_ms / steps if graph_ms else None
    ms = min(eager, gstep) if gstep else eager
    attn_iso_ms = float(np.mean(attn))
    attn_ms = attn_graph_ms if attn_graph_ms else attn_iso_ms
    # the roofline counts what one launch must read from HBM: blocks shared by
    # several sequences once (their repeats come from L2)
    alg = algorithmic_unique_bytes(c)
    res = {
        "ms_per_step": ms,
        "ms_per_step_eager": eager,
        "ms_per_step_graph": gstep,
        "timing": "cuda-graph replay of 10-step chunks" if (gstep and gstep <= eager)
                  else "eager launches",
        "kv_bytes": kv_bytes(c),
        "kv_gbs": unique_kv_bytes(c) / (ms * 1e-3) / 1e9,
        "attn_kernel_us": attn_ms * 1e3,
        "attn_kernel_timing": "10 launches chained with PDL in a CUDA graph, replayed"
                              if attn_graph_ms else "CUDA events around each launch",
        "attn_kernel_isolated_us": attn_iso_ms * 1e3,
        "attn_kernel_isolated_median_us": float(np.median(attn)) * 1e3,
        "attn_kernel_isolated_p10_p90_us": [float(np.percentile(attn, 10)) * 1e3,
                                            float(np.percentile(attn, 90)) * 1e3],
        "algorithmic_bytes": alg,
        "roofline": {
            "bound": "hbm",
            "achieved": alg / (attn_ms * 1e-3) / 1e9,
            "peak": peak, "unit": "GB/s",
            "frac": alg / (attn_ms * 1e-3) / 1e9 / peak,
            "traffic": profiled_traffic(name),
            "peak_kind": peak_kind,
        },
        "tokens_per_s_per_layer": c.batch / (ms * 1e-3),
        "decode_tokens_per_s_model": c.batch / (ms * 1e-3 * MODEL_LAYERS[name]),
        "model_layers": MODEL_LAYERS[name],
        "gpu_launches": per_step * steps,
        "launches_per_step": per_step,
        "clocks": clocks,
        "batch": c.batch,
        "seq_len_max": int(c.seq_lens.max()),
        "block_waste": wl.block_waste(c),
    }
    if c.shared_prefix_tokens:
        # every sequence's whole KV counted, shared blocks once per sequence
        res["logical_kv_gbs"] = kv_bytes(c) / (ms * 1e-3) / 1e9
        res["unique_kv_bytes"] = unique_kv_bytes(c)
    if e2e:
        (z_ms, z_how), zi, zo = time_e2e_zero_copy(w, max(10, steps // 10), 3)
        e_ms, h2d, d2h = time_e2e(w, max(10, steps // 10), 3)
        res["e2e"] = {"value": kv_bytes(c) / (z_ms * 1e-3) / 1e9, "unit": UNIT,
                      "ms_per_step": z_ms, "h2d_bytes_per_step": zi, "d2h_bytes_per_step": zo,
                      "transfer": "zero-copy: the kernels read each step's inputs from pinned "
                                  "host memory and write its output to pinned host memory "
                                  "(NVLink-C2C); " + z_how,
                      "explicit_copies": {"value": kv_bytes(c) / (e_ms * 1e-3) / 1e9,
                                          "ms_per_step": e_ms, "h2d_bytes_per_step": h2d,
                                          "d2h_bytes_per_step": d2h,
                                          "transfer": "cudaMemcpyAsync H2D of a pinned staging "
                                                      "buffer and D2H of the output each step, "
                                                      "on side streams, graph replay"}}
    return w, res


def aggregate_ranks(ms_per_step, kv_bytes_per_step, device="cpu"):
    """Whole-job throughput over all ranks: every rank ran its own batch (no data
    exchange), the job took as long as the slowest rank, and the job moved the
    sum of all ranks' KV bytes.  Returns (max ms per step, GB/s of the job)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms_per_step, kv_bytes_per_step / (ms_per_step * 1e-3) / 1e9
    t = torch.tensor([ms_per_step, float(kv_bytes_per_step)], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    ms = float(mx[0].item())
    return ms, float(t[1].item()) / (ms * 1e-3) / 1e9


def measure_multi_token(base, q_len, steps, device):
    """Multi-token decode (q_len new tokens per sequence, causal within the chunk)
    on a full-size workload, the new tokens already stored: one attention launch
    plus the merge per step, chained with programmatic dependent launch and
    replayed from a CUDA graph (as the decode step); the attention kernel alone
    is also timed with CUDA events (phase 1, for the roofline)."""
    from paged_kv_cache_215_gb300 import pkv
    w = Workload(base, device)
    c = w.case
    g = torch.Generator(device=device).manual_seed(77)
    q = torch.randn(c.batch, q_len, c.num_q_heads, c.head_dim, generator=g,
                    device=device).to(torch.bfloat16)
    out = torch.empty(c.batch, q_len, c.num_q_heads, c.head_dim, dtype=torch.bfloat16,
                      device=device)
    nb = int(pkv.lib().paged_decode_workspace_bytes_mq(ctypes.byref(w.geom), c.batch, q_len,
                                                       w.max_len, 0))
    ws = torch.empty(nb, dtype=torch.uint8, device=device)
    pdl, attn = pkv.launch_opts(pdl=1), pkv.launch_opts(phase=1)

    def step(o):
        pkv.paged_decode_attention_mq(out, q, w.pool, c.layer, w.tables, w.seq_lens, w.max_len,
                                      c.scale, w.ks, w.vs, 0, ws, opts=o)
    stream = torch.cuda.current_stream()
    for _ in range(5):
        step(pdl)
    torch.cuda.synchronize()
    chunk = 10
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(chunk):
            step(pdl)
    reps = max(1, steps // chunk)
    graph.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        graph.replay()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / (reps * chunk)
    s.record(stream)
    for _ in range(steps):
        step(attn)
    e.record(stream)
    torch.cuda.synchronize()
    attn_us = s.elapsed_time(e) / steps * 1e3
    del graph
    w.close()
    del w
    torch.cuda.empty_cache()
    kvb = kv_bytes(c)
    return {"q_len": q_len, "ms_per_step": ms, "attn_kernel_us": attn_us,
            "kv_gbs": kvb / (ms * 1e-3) / 1e9,
            "roofline_frac": kvb / (attn_us * 1e-6) / 1e9 / peaks()[0],
            "query_tokens_per_s_per_layer": c.batch * q_len / (ms * 1e-3), "batch": c.batch,
            "timing": "cuda-graph replay of 10-step chunks; attention kernel alone by CUDA events"}


def measure_chunked_prefill(device, batch=4, context=16384, chunk=2048, steps=20, kv="bf16"):
    """Chunked prefill on the tcgen05 kernel: `batch` sequences of `context` tokens
    (32 query / 8 KV heads, D 128, bs 16, a bf16, f16 or E4M3 pool; f16 queries for
    an f16 pool, else bf16) whose
    last `chunk` tokens are the new queries, causal within the chunk.
    Work = 4 * D flops per (query head, visible key)."""
    from paged_kv_cache_215_gb300 import pkv
    tag = "" if kv == "bf16" else f"_{kv}"
    qd = "f16" if kv == "f16" else "bf16"
    case = wl.make_case(f"chunked_prefill{tag}_b{batch}_ctx{context}_chunk{chunk}",
                        [context] * batch, 32, 8, 128, 16, kv, qd, qd, seed=1007)
    t = wl.make_tensors(case, device=device)
    geom = pkv.geometry(1, 32, 8, 128, 16, case.num_blocks, kv)
    pool = pkv.KVPool(geom, device=device)
    pool.storage.zero_()
    ids = case.tables[case.tables >= 0]
    pool.reserve(np.unique(ids).tolist())
    tables = torch.from_numpy(case.tables).to(device)
    lens = torch.from_numpy(case.seq_lens).to(device)
    ks = vs = 1.0
    if kv == "e4m3":
        ks, vs = pkv.fp8_scales((t.k_tokens, t.k_new), (t.v_tokens, t.v_new))
    pool.append_tokens(0, t.k_tokens, t.v_tokens, tables, t.tok_seq, t.tok_pos, ks, vs)
    pool.append(0, t.k_new, t.v_new, tables, t.new_pos, ks, vs)
    g = torch.Generator(device=device).manual_seed(78)
    q = torch.randn(batch, chunk, 32, 128, generator=g, device=device).to(wl.TORCH_DT[qd])
    out = torch.empty(batch, chunk, 32, 128, dtype=wl.TORCH_DT[qd], device=device)
    ws = torch.empty(16, dtype=torch.uint8, device=device)

    def step():
        pkv.paged_decode_attention_mq(out, q, pool, 0, tables, lens, context, case.scale, ks, vs,
                                      workspace=ws)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    keys = sum(context - chunk + i + 1 for i in range(chunk))      # visible keys per query row
    flops = 4.0 * 128 * 32 * keys * batch
    assert pool.check_status() == 0
    pool.close()
    peak = bf16_peak()
    return {"workload": case.name, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "peak": peak, "unit": "TFLOP/s",
                         "frac": flops / (ms * 1e-3) / 1e12 / peak},
            "query_tokens_per_s": batch * chunk / (ms * 1e-3)}


CASCADE = ["shared_prefix_64k_b32", "llama70b_prefix_bs16"]


def measure_cascade(name, device, steps=20):
    """Decode attention (no append) of a batch whose sequences share a prefix of
    blocks: the plain path (every sequence reads the prefix) against the
    shared-prefix path (the prefix read once for all sequences on the tcgen05
    kernel, the private suffixes through the decode kernel).  Reported: times of
    the plain decode, the automatic route and the forced prefix pass; GB/s of
    the unique KV bytes (every block once: what the HBM must deliver) and of the
    logical bytes (every sequence's whole KV); and the prefix pass's own rate
    (phase 1: the suffix-table build and the tcgen05 pass over the prefix) in
    TFLOP/s, 4 x head_dim flops per (query head of a sequence, prefix key)."""
    from paged_kv_cache_215_gb300 import pkv
    w = Workload(name, device)
    c = w.case
    table, P, lens = wl.prefix_args(c)
    prefix_flops = 4.0 * c.head_dim * c.num_q_heads * float(lens.astype(np.int64).sum())
    table = torch.from_numpy(table).to(device)
    lens = torch.from_numpy(lens).to(device)
    out = torch.empty_like(w.out)
    ws = torch.empty(pkv.cascade_workspace_bytes(w.geom, c.batch, c.max_blocks, w.max_len, P),
                     dtype=torch.uint8, device=device)

    def cascade(route=0, phase=0):
        pkv.paged_decode_attention_cascade(out, w.tens.q, w.pool, c.layer, table, P, lens,
                                           w.tables, w.seq_lens, w.max_len, c.scale, workspace=ws,
                                           opts=pkv.launch_opts(kernel=route, phase=phase))

    def plain():
        pkv.paged_decode_attention(w.out, w.tens.q, w.pool, c.layer, w.tables, w.seq_lens,
                                   w.max_len, c.scale, workspace=w.ws)
    res = {}
    arms = (("plain", plain), ("cascade", cascade), ("prefix_pass", lambda: cascade(3)),
            ("prefix_pass_phase1", lambda: cascade(3, 1)))
    for nm, f in arms * 2:
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            f()
        e.record()
        torch.cuda.synchronize()
        res[nm] = min(res.get(nm, 1e9), s.elapsed_time(e) / steps * 1e3)
    status = w.pool.check_status()
    kvb, ukv = kv_bytes(c), unique_kv_bytes(c)
    w.close()
    del w
    torch.cuda.empty_cache()
    return {"batch": c.batch, "shared_prefix_tokens": P, "status": status,
            "plain_us": res["plain"], "cascade_us": res["cascade"],
            "forced_prefix_route_us": res["prefix_pass"],
            "prefix_pass_us": res["prefix_pass_phase1"],
            "prefix_pass_tflops": prefix_flops / (res["prefix_pass_phase1"] * 1e-6) / 1e12,
            "speedup": res["plain"] / res["cascade"],
            "unique_kv_bytes": ukv,
            "unique_kv_gbs_plain": ukv / (res["plain"] * 1e-6) / 1e9,
            "unique_kv_gbs_cascade": ukv / (res["cascade"] * 1e-6) / 1e9,
            "logical_kv_gbs_plain": kvb / (res["plain"] * 1e-6) / 1e9,
            "logical_kv_gbs_cascade": kvb / (res["cascade"] * 1e-6) / 1e9}


APPEND = ["llama8b_b32_8k", "fp8_b8_32k"]


def measure_append(name, device, calls=50, reps=4):
    """Latency of kv_append alone (reshape_and_cache of one new token per sequence,
    bf16 in, the pool's dtype stored) on the workload's pool: a CUDA graph of
    `calls` back-to-back appends, replayed; microseconds per call."""
    w = Workload(name, device)
    c, t = w.case, w.tens

    def app():
        w.pool.append(c.layer, t.k_new, t.v_new, w.tables, t.new_pos, w.ks, w.vs)
    app()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            app()
    g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / (calls * reps)
    assert w.pool.check_status() == 0
    per_tok = 2 * c.num_kv_heads * c.head_dim
    moved = c.batch * per_tok * (2 + c.kv_elem_bytes())       # bf16 in, pool dtype out
    w.close()
    return {"batch": c.batch, "kv_dtype": c.kv_dtype, "us_per_call": us,
            "bytes_per_call": moved, "timing": f"CUDA graph of {calls} appends, {reps} replays"}


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"])
    return 1900.0


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    from paged_kv_cache_215_gb300 import build
    if rank == 0:
        build.build()
    if ws > 1:
        dist.barrier()
    name = args.workload
    # this rank's share of the global batch (N times the single-GPU workload)
    case = dp.rank_case(name, rank, ws)
    w, res = measure(name, args.steps, args.warmup, device, with_clocks=True, gpu_index=local,
                     case=case)
    ms, value = aggregate_ranks(res["ms_per_step"], res["kv_bytes"], device)
    extra = {}
    if rank == 0 and not args.no_cpu_baseline:
        extra["cpu_baseline"] = cpu_baseline(w)
    w.close()
    del w
    torch.cuda.empty_cache()
    others = {}
    if rank == 0 and not args.only_primary:
        for other in SECONDARY:
            ow, ores = measure(other, max(50, args.steps // 20), args.warmup, device,
                               with_clocks=False, e2e=False)
            ow.close()
            del ow
            torch.cuda.empty_cache()
            others[other] = {k: ores[k] for k in ("ms_per_step", "ms_per_step_eager",
                                                  "ms_per_step_graph", "kv_gbs", "attn_kernel_us",
                                                  "attn_kernel_isolated_us",
                                                  "tokens_per_s_per_layer",
                                                  "decode_tokens_per_s_model", "batch",
                                                  "block_waste")}
            others[other]["roofline_frac"] = ores["roofline"]["frac"]
            others[other]["achieved_gbs"] = ores["roofline"]["achieved"]
            if "logical_kv_gbs" in ores:
                others[other]["logical_kv_gbs"] = ores["logical_kv_gbs"]
                others[other]["unique_kv_bytes"] = ores["unique_kv_bytes"]
    if rank == 0 and not args.only_primary:
        for mq_name, (base, q_len) in wl.MULTI_TOKEN.items():
            others[mq_name] = measure_multi_token(base, q_len, max(50, args.steps // 20), device)
        for kv in ("bf16", "e4m3"):
            cp = measure_chunked_prefill(device, kv=kv)
            others[cp.pop("workload")] = cp
        for cname in CASCADE:
            others[f"{cname}_shared_prefix_decode"] = measure_cascade(cname, device)
        for aname in APPEND:
            others[f"{aname}_append"] = measure_append(aname, device)
    if ws > 1:
        dist.barrier()
    if rank != 0:
        return
    c = wl.FULL[name]()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": c.kv_dtype, "data": "synthetic (seeded N(0,1))",
        "config": bench_config(c, ws),
        "decode_tokens_per_s": res["decode_tokens_per_s_model"],
        "decode_tokens_per_s_per_layer": res["tokens_per_s_per_layer"],
        "roofline": res["roofline"],
        "attn_kernel_us": res["attn_kernel_us"],
        "attn_kernel_timing": res["attn_kernel_timing"],
        "attn_kernel_isolated_us": res["attn_kernel_isolated_us"],
        "attn_kernel_isolated_median_us": res["attn_kernel_isolated_median_us"],
        "attn_kernel_isolated_p10_p90_us": res["attn_kernel_isolated_p10_p90_us"],
        "ms_per_step_eager": res["ms_per_step_eager"],
        "ms_per_step_graph": res["ms_per_step_graph"],
        "timing": res["timing"],
        "launches_per_step": res["launches_per_step"],
        "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"],
        "clocks": res["clocks"],
        "block_waste": res["block_waste"],
    }
    line.update(extra)
    if others:
        line["workloads"] = others
    print(json.dumps(line), flush=True)


def bench_config(c, world):
    """The line's config: the workload of one GPU, the global batch of the job."""
    return {"workload": c.name, "batch": c.batch, "global_batch": c.batch * world,
            "seq_len": int(c.seq_lens.max()), "q_heads": c.num_q_heads,
            "kv_heads": c.num_kv_heads, "head_dim": c.head_dim, "block_size": c.block_size,
            "kv_dtype": c.kv_dtype,
            "parallelism": f"dp{world} (the global batch split by sequence across GPUs, "
                           "no exchange)",
            "l2": "inputs larger than L2 (KV read per step >> 129 MB), no flush"}


# ---------------------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = args.workload
    c = wl.FULL[name]()
    tens = wl.make_tensors(c, device="cpu" if not torch.cuda.is_available() else "cuda")
    raw = wl.raw_numpy
    ks = vs = 1.0
    if c.kv_dtype == "e4m3":
        ka = max(oracle.absmax(raw(tens.k_tokens), "bf16"), oracle.absmax(raw(tens.k_new), "bf16"))
        va = max(oracle.absmax(raw(tens.v_tokens), "bf16"), oracle.absmax(raw(tens.v_new), "bf16"))
        ks, vs = oracle.fp8_scale(ka), oracle.fp8_scale(va)
    eb = c.kv_elem_bytes()
    pool = np.zeros(oracle.kv_bytes(c.num_layers, c.num_kv_heads, c.head_dim,
                                    c.num_blocks * c.block_size, eb), dtype=np.uint8)
    in_dt = "bf16" if c.kv_dtype == "e4m3" else c.kv_dtype
    oracle.append_tokens(pool, c.kv_dtype, c.geometry, c.layer, raw(tens.k_tokens),
                         raw(tens.v_tokens), in_dt, c.tables, raw(tens.tok_seq), raw(tens.tok_pos),
                         ks, vs)
    q = raw(tens.q)
    knew, vnew, npos = raw(tens.k_new), raw(tens.v_new), raw(tens.new_pos)
    del tens
    rows_all = c.batch * c.num_q_heads
    per_row = kv_bytes(c) / rows_all
    threads = oracle.num_threads()

    def step(rows):
        oracle.append(pool, c.kv_dtype, c.geometry, c.layer, knew, vnew, in_dt, c.tables, npos,
                      ks, vs)
        oracle.decode(q, c.q_dtype, pool, c.kv_dtype, c.geometry, c.layer, c.tables, c.seq_lens,
                      c.scale, ks, vs, rows=rows)

    # size one step's sample so that the whole run takes about two minutes
    probe = np.arange(min(threads, rows_all), dtype=np.int32)
    t0 = time.perf_counter()
    step(probe)
    per_row_s = (time.perf_counter() - t0) / probe.size
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_rows = int(max(1, min(rows_all, budget / max(per_row_s, 1e-9))))
    cursor = 0

    def next_rows():
        nonlocal cursor
        r = (np.arange(n_rows) + cursor) % rows_all
        cursor = (cursor + n_rows) % rows_all
        return r.astype(np.int32)

    for _ in range(args.warmup):
        step(next_rows())
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(next_rows())
    total = time.perf_counter() - t0
    value = args.steps * n_rows * per_row / total / 1e9
    sample = (f"{n_rows} of {rows_all} (sequence, query head) rows per step, fp64 oracle "
              f"(append + paged decode), GB/s counts each row's share of the KV bytes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": bench_config(c, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=PRIMARY, choices=sorted(wl.FULL))
    ap.add_argument("--only-primary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the chunked-prefill (tcgen05) case and print its JSON")
    ap.add_argument("--cascade-only", action="store_true",
                    help="time only the shared-prefix decode workloads and print their JSON")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        from paged_kv_cache_215_gb300 import build
        build.build()
        for kv in ("bf16", "e4m3"):
            print(json.dumps(measure_chunked_prefill("cuda", steps=args.steps, kv=kv)), flush=True)
    elif args.cascade_only:
        from paged_kv_cache_215_gb300 import build
        build.build()
        names = CASCADE if args.workload == PRIMARY else [args.workload]
        for cname in names:
            r = measure_cascade(cname, "cuda", steps=args.steps)
            print(json.dumps({"workload": f"{cname}_shared_prefix_decode", **r}), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
