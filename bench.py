#!/usr/bin/env python
"""Benchmark of one full verify step on synthetic data.

A step is one pass of the whole hot path over one batch: tree-verify
attention with chunk salience for every layer (scores summed over layers),
top-k chunk selection plus window gathered into the compact cache, and tree
acceptance.  Default workload: Llama-3.1-8B KV shapes at 128K context with a
64-node tree, 32 layers, greedy acceptance over a 128,256-token vocabulary.

Prints one JSON line (rank 0).  `value` is microseconds per verify step per
layer (step time / layers; with N replicas, the whole job's step time per
layer-step: ms / (layers * N)), so lower is better.  Inputs stay resident in
HBM; every layer's K/V cache is a distinct 537 MB tensor, larger than L2.

--impl reference times the float64 CPU oracle on the host cores instead:
each step is one whole layer of the same workload (every kv head) plus its
retrieval and acceptance, and the per-layer figure is extrapolated to the
workload's layer count with the factor stated in the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

# The oracle's BLAS runs on every host core this process may use: the thread
# count is fixed before NumPy (or torch) is first imported.
CORES = len(os.sched_getaffinity(0))
for _var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_var] = str(CORES)

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("µs/verify-step/layer and KV GB/s (% HBM peak) at 128K ctx, "
          "64-node tree")
UNIT = "us/verify-step/layer"
DEFAULT_WORKLOAD = "llama8b-128k-32l"
FALLBACK_HBM_GBS = 6800.0
EV_PER_STEP = 1       # split-pass launches bracketed by events per step
CPU_BASELINE_LAYERS = 4   # whole layers the CPU baseline times


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank float over the process group (timings: the job is as
    slow as its slowest replica)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _kv_bytes(wl, st):
    return sum((L + T) for L, T in zip(st.ctx_lens, st.tree_sizes)) * \
        wl.num_kv_heads * wl.head_dim * 2 * 2


def _q_bytes(wl, st):
    return st.n_nodes * wl.num_q_heads * wl.head_dim * 2


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region:
    the sampler is started (and its first sample awaited) before the region,
    and only samples stamped inside the region's host-clock window are kept;
    when the region is shorter than the sampling period and none falls
    inside, the sample nearest to it is reported with samples = 0."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ds_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_ready(self, timeout_s: float = 3.0):
        """Blocks until nvidia-smi has written its first sample."""
        t_end = time.time() + timeout_s
        while self.proc is not None and time.time() < t_end:
            if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                return
            time.sleep(0.01)

    def stop(self, t0: float = None, t1: float = None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_samples(lines, t0, t1)


def sampled_launches(steps: int, layers: int, per_step: int):
    """(step, layer) pairs whose split pass is bracketed by events:
    `per_step` consecutive layers per step, starting at layer s * per_step
    (mod layers) in step s, so the sample rotates through every layer (all
    layers of a step when it has no more than `per_step`)."""
    if layers <= per_step:
        return [(s, l) for s in range(steps) for l in range(layers)]
    return [(s, (s * per_step + j) % layers) for s in range(steps) for j in range(per_step)]


def parse_clock_samples(lines, t0=None, t1=None):
    """Summary of nvidia-smi csv lines (timestamp first) within [t0, t1]
    (host epoch seconds); the nearest sample when none is inside."""
    import datetime
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
             "sw_power_cap"]
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            rows.append((ts, float(parts[2]), float(parts[3]),
                         [n for n, v in zip(names, parts[6:10])
                          if v.lower().startswith("active")]))
        except ValueError:
            continue
    if not rows:
        return None
    inside = rows if t0 is None else [r for r in rows if t0 <= r[0] <= t1]
    n_inside = len(inside)
    if not inside:
        mid = 0.5 * (t0 + t1)
        inside = [min(rows, key=lambda r: abs(r[0] - mid))]
    reasons = sorted({n for r in inside for n in r[3]})
    return {"sm_mhz": statistics.median(r[1] for r in inside),
            "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
            "samples": n_inside}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)

def oracle_time(wl, st, layers, src, accept_inp):
    """Times the float64 oracle on whole layers of one step: verify attention
    of every kv head for each layer given (all query heads, all nodes, chunk
    scores summed over those layers), then the top-k gather with the
    workload's local RoPE over the whole source cache (K and V of every kv
    head), then acceptance.  Returns a dict of wall-clock seconds."""
    import numpy as np
    import torch
    from oracle import ref
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    t_layers = []
    total = 0.0
    for q, k, v in layers:
        t0 = time.perf_counter()
        _, scores, _ = ref.verify_attention(
            f64(q), f64(k), f64(v), st.page_table.numpy(), st.ctx_lens,
            st.tree_offsets, st.parents, wl.page_size, wl.chunk_size)
        total = total + scores
        t_layers.append(time.perf_counter() - t0)
    sk, sv = src
    cap = wl.top_k * wl.chunk_size + wl.window
    t0 = time.perf_counter()
    ref.gather_compact(bits(sk), bits(sv), st.page_table.numpy(), st.ctx_lens,
                       total, wl.page_size, wl.chunk_size, wl.top_k, wl.window,
                       cap, rope_base=wl.rope_base)
    t_gather = time.perf_counter() - t0
    t0 = time.perf_counter()
    tl = accept_inp.target_logits.cpu().numpy()
    toks = accept_inp.draft_tokens.cpu().numpy()
    if wl.accept == "reject":
        ref.rejection_accept(tl, accept_inp.draft_logits.cpu().numpy(), toks,
                             st.parents, st.tree_offsets,
                             accept_inp.uniforms.cpu().numpy())
    else:
        ref.greedy_accept(tl, toks, st.parents, st.tree_offsets)
    t_accept = time.perf_counter() - t0
    return {"layers": t_layers, "gather": t_gather, "accept": t_accept}


def oracle_summary(wl, t):
    """Per-layer figure of a whole step from timed layers: the mean timed
    layer stands for each of the workload's layers (extrapolation factor =
    layers / timed layers), retrieval and acceptance are timed in full and
    spread over the layers like the GPU figure."""
    n = len(t["layers"])
    per_layer_s = (statistics.mean(t["layers"]) * wl.layers + t["gather"] +
                   t["accept"]) / wl.layers
    return {
        "value_us": per_layer_s * 1e6,
        "timed_layers": n,
        "timed_kv_heads": wl.num_kv_heads,
        "extrapolation_factor": wl.layers / n,
        "extrapolated": n < wl.layers,
        "layer_s": [round(x, 3) for x in t["layers"]],
        "gather_s": round(t["gather"], 3),
        "accept_s": round(t["accept"], 3),
        "sample": (f"{n} whole layer(s) of verify attention (all "
                   f"{wl.num_kv_heads} kv heads, all query heads and nodes) "
                   f"timed and taken x{wl.layers / n:g} for the step's "
                   f"{wl.layers} layers; top-k gather with local RoPE and "
                   f"{wl.accept} acceptance timed in full; divided by "
                   f"{wl.layers} layers"),
    }


def cpu_inputs(wl, n_layers):
    from long_context_speculative_ds_gb300 import synth
    st = synth.make_structure(wl)
    layers = [synth.make_layer(st, l, device="cpu") for l in range(n_layers)]
    src = synth.make_source_cache(st, device="cpu")
    mode = "reject" if wl.accept == "reject" else "greedy"
    acc = synth.make_accept_inputs(st, mode)
    return st, layers, src, acc


def run_reference(args, wl, rank, world):
    """The reference arm: the float64 oracle on the host cores.  Each step
    runs one whole layer (every kv head) plus the retrieval and acceptance;
    `ms_per_step` is that step's measured wall time, and `value` is the
    per-layer figure of a whole step with the layer time taken for each of
    the workload's layers (the fields say by how much)."""
    if rank != 0:
        return
    st, layers, src, acc = cpu_inputs(wl, 1)
    for _ in range(args.warmup):
        oracle_time(wl, st, layers, src, acc)
    runs = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        t = oracle_time(wl, st, layers, src, acc)
        runs.append((time.perf_counter() - t0, t))
    step_s = statistics.mean(r[0] for r in runs)
    merged = {"layers": [x for r in runs for x in r[1]["layers"]],
              "gather": statistics.mean(r[1]["gather"] for r in runs),
              "accept": statistics.mean(r[1]["accept"] for r in runs)}
    summ = oracle_summary(wl, merged)
    summ["timed_layers"] = 1
    summ["extrapolation_factor"] = wl.layers
    summ["layer_s"] = [round(statistics.mean(merged["layers"]), 3)]
    us = summ.pop("value_us")
    kvb = _kv_bytes(wl, st)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": _config(wl, st),
        "kv_gbs": round(kvb / (us * 1e-6) / 1e9, 3),
        "cpu_baseline": {"value": round(us, 3), "unit": UNIT, "cores": CORES,
                         "kind": "oracle", **summ},
        "e2e": {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(wl, st, kv_layout="NHD"):
    return {"workload": wl.name, "batch": wl.batch, "kv_layout": kv_layout,
            "ctx_lens": st.ctx_lens if wl.batch <= 8 else "ragged",
            "tree_nodes": st.tree_sizes, "layers": wl.layers,
            "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads,
            "head_dim": wl.head_dim, "page_size": wl.page_size,
            "chunk_size": wl.chunk_size, "top_k": wl.top_k,
            "window": wl.window, "vocab": wl.vocab, "accept": wl.accept,
            "rope_base": wl.rope_base, "kv_commit": True,
            "split_events": f"{EV_PER_STEP} split pass per step bracketed by events, "
                            "the layer rotating with the step",
            "l2": "inputs larger than L2: every layer has its own "
                  f"{_kv_bytes(wl, st) / 1e6:.0f} MB K/V cache"}


def _traffic_for(src_path: str):
    """DRAM bytes per launch of the split pass from the committed ncu summary,
    valid only while the kernel source (comments aside) is unchanged since
    the capture."""
    p = os.path.join(ROOT, "profiles", "verify_split_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_code_sha256") != code_sha256(src_path):
        return None
    return d.get("dram_bytes_per_launch_full_size")


def code_sha256(src_path: str) -> str:
    """sha256 of a C++/CUDA source with comments and blank space removed, so
    that edits to comments alone do not invalidate counters taken from it
    (string literals in the kernel sources hold no comment markers)."""
    import re
    text = open(src_path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = re.sub(r"\s+", " ", text).strip()
    return hashlib.sha256(text.encode()).hexdigest()


# ---------------------------------------------------------------------------
# the other workloads, measured in the same process after the headline

OTHER_WORKLOADS = ("llama8b-32k", "llama8b-64k", "qwen3-8b-ragged-b8")
OTHER_LAYERS = 4      # distinct layer caches per workload, rotated (> L2)


def workload_block(name, dev, peak, reps=6):
    """Split pass, whole verify call, retrieval and acceptance of one of the
    other workloads: OTHER_LAYERS layers with their own caches are verified
    back to back `reps` times with the split pass of every layer bracketed
    by CUDA events (the split-pass figure; the events break the dependent
    launch of the next kernel), then `reps` times again with no event
    between kernels (the verify-call figure)."""
    import torch
    from long_context_speculative_ds_gb300 import binding, synth
    from long_context_speculative_ds_gb300.step import StepInputs, VerifyStep
    wl = synth.WORKLOADS[name]
    nl = min(OTHER_LAYERS, wl.layers) if wl.layers > 1 else OTHER_LAYERS
    st = synth.make_structure(wl)
    qs, ks, vs = [], [], []
    for l in range(nl):
        q, k, v = synth.make_layer(st, l, device=dev)
        qs.append(q); ks.append(k); vs.append(v)
    sk, sv = synth.make_source_cache(st, device=dev)
    mode = "reject" if wl.accept == "reject" else "greedy"
    acc = synth.make_accept_inputs(st, mode, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    inp = StepInputs(page_table=st.page_table.to(dev),
                     ctx_lens=torch.tensor(st.ctx_lens, **i32),
                     tree_offsets=torch.tensor(st.tree_offsets, **i32),
                     parents=torch.tensor(st.parents, **i32),
                     q=qs, k_cache=ks, v_cache=vs, src_k=sk, src_v=sv,
                     target_logits=acc.target_logits, draft_logits=acc.draft_logits,
                     draft_tokens=acc.draft_tokens, uniforms=acc.uniforms)
    step = VerifyStep(inp, chunk_size=wl.chunk_size, top_k=wl.top_k, window=wl.window,
                      accept_mode=mode, rope_base=wl.rope_base)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nl)] for _ in range(reps)]
    for e_a, e_b in (e for row in evs for e in row):   # torch creates them on first record
        e_a.record()
        e_b.record()
    pargs = [[binding.verify_args(
        inp.q[l], inp.k_cache[l], inp.v_cache[l], inp.page_table, inp.ctx_lens,
        inp.tree_offsets, inp.parents, chunk_size=wl.chunk_size, out=step.out[l],
        chunk_scores=step.scores, workspace=step.ws_verify, accumulate=l > 0,
        prof_events=evs[r][l]) for l in range(nl)] for r in range(reps)]
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    for r in range(reps):
        for l in range(nl):
            binding.ds_verify_attn(pargs[r][l])
    torch.cuda.synchronize()
    assert step.device_status() == 0
    split_us = statistics.median(a.elapsed_time(b) * 1e3 for row in evs for a, b in row)
    # whole verify calls back to back, with no event between their kernels
    # (an event pair ends the dependent-launch overlap of the next kernel)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(reps):
        for l in range(nl):
            step.verify_layer(l)
    c1.record()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    verify_us = c0.elapsed_time(c1) * 1e3 / (reps * nl)

    def alone(fn, n=10):
        fn()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(n):
            fn()
        a1.record()
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) * 1e3 / n
    gather_us = alone(step.gather)
    accept_us = alone(step.accept)
    assert step.device_status() == 0
    alg = _kv_bytes(wl, st) + _q_bytes(wl, st)
    achieved = alg / (split_us * 1e-6) / 1e9
    accept_bytes = st.n_nodes * wl.vocab * 4 * (2 if mode == "reject" else 1)
    out = {
        "batch": wl.batch, "ctx_lens": st.ctx_lens, "tree_nodes": st.tree_sizes,
        "layers_rotated": nl,
        "split_pass_us": round(split_us, 2),
        "split_pass_gbs": round(achieved, 1),
        "split_pass_frac": round(achieved / peak, 4),
        "algorithmic_bytes_per_layer": alg,
        "verify_call_us": round(verify_us, 2),
        "verify_call_frac": round(alg / (verify_us * 1e-6) / 1e9 / peak, 4),
        "retrieval_us": round(gather_us, 2),
        "accept_us": round(accept_us, 2), "accept_mode": mode,
        "accept_gbs": round(accept_bytes / (accept_us * 1e-6) / 1e9, 1),
    }
    del step, inp, qs, ks, vs, sk, sv, acc
    torch.cuda.empty_cache()
    return out


def _end_to_end(step, inp, args, world, dev, barrier):
    """Per step: copy the step's inputs from pinned host memory (on a side
    stream, overlapping the verify of earlier layers), run the step through
    the library, read the results back, and wait for them; wall-clock timed.
    The step is captured once as a CUDA graph (`VerifyStep.capture_from_host`)
    and replayed each step, as a serving loop would: every copy and kernel
    runs every step, with one launch from the host."""
    import torch
    from long_context_speculative_ds_gb300.step import StepInputs
    pin = lambda t: None if t is None else t.cpu().pin_memory()
    host = StepInputs(
        page_table=pin(inp.page_table), ctx_lens=pin(inp.ctx_lens),
        tree_offsets=pin(inp.tree_offsets), parents=pin(inp.parents),
        q=[pin(x) for x in inp.q], k_cache=[], v_cache=[], src_k=None,
        src_v=None, target_logits=pin(inp.target_logits),
        draft_logits=pin(inp.draft_logits), draft_tokens=pin(inp.draft_tokens),
        uniforms=pin(inp.uniforms))
    host_out = {n: torch.empty_like(getattr(step, n), device="cpu").pin_memory()
                for n in ("out_path", "out_n", "out_bonus", "out_chunk_ids",
                          "out_len")}
    for _ in range(max(1, min(args.warmup, 2))):
        step.run_from_host(host, host_out)
    torch.cuda.synchronize()
    step.capture_from_host(host, host_out)
    for _ in range(max(1, min(args.warmup, 2))):
        step.replay()
    torch.cuda.synchronize()
    barrier()
    h2d = d2h = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        h2d, d2h = step.replay()
        torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    if world > 1:
        e2e_ms = max_over_ranks(e2e_ms, dev)
    return e2e_ms, h2d, d2h


def run_ours(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from long_context_speculative_ds_gb300 import binding, synth
    from long_context_speculative_ds_gb300 import build as bld
    from long_context_speculative_ds_gb300.step import StepInputs, VerifyStep

    if not bld.up_to_date():
        if world > 1:
            raise RuntimeError("library not built; run __graft_entry__.build()")
        bld.build()
    binding.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    st = synth.make_structure(wl)
    qs, ks, vs = [], [], []
    for l in range(wl.layers):
        q, k, v = synth.make_layer(st, l, device=dev, layout=args.kv_layout)
        qs.append(q); ks.append(k); vs.append(v)
    sk, sv = synth.make_source_cache(st, device=dev, layout=args.kv_layout)
    mode = "reject" if wl.accept == "reject" else "greedy"
    acc = synth.make_accept_inputs(st, mode, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    inp = StepInputs(page_table=st.page_table.to(dev),
                     ctx_lens=torch.tensor(st.ctx_lens, **i32),
                     tree_offsets=torch.tensor(st.tree_offsets, **i32),
                     parents=torch.tensor(st.parents, **i32),
                     q=qs, k_cache=ks, v_cache=vs, src_k=sk, src_v=sv,
                     target_logits=acc.target_logits,
                     draft_logits=acc.draft_logits,
                     draft_tokens=acc.draft_tokens, uniforms=acc.uniforms)
    step = VerifyStep(inp, chunk_size=wl.chunk_size, top_k=wl.top_k,
                      window=wl.window, accept_mode=mode,
                      kv_layout=args.kv_layout, with_commit=True,
                      rope_base=wl.rope_base)
    # events around a sample of the split-pass launches (each event pair
    # sits between two kernels of the step, breaks their dependent launch
    # and costs the step a few microseconds): EV_PER_STEP launches per step,
    # the layer rotating with the step so that the sample covers the layers
    sampled = sampled_launches(args.steps, wl.layers, EV_PER_STEP)
    evs = [(torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in sampled]
    for e_a, e_b in evs:      # torch creates the CUDA event on first record
        e_a.record()
        e_b.record()
    torch.cuda.synchronize()
    prof_args = {}
    for (s_, l), ev in zip(sampled, evs):
        prof_args[(s_, l)] = binding.verify_args(
            inp.q[l], inp.k_cache[l], inp.v_cache[l], inp.page_table,
            inp.ctx_lens, inp.tree_offsets, inp.parents,
            chunk_size=wl.chunk_size, out=step.out[l],
            chunk_scores=step.scores, workspace=step.ws_verify,
            kv_layout=args.kv_layout, accumulate=l > 0, prof_events=ev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0

    sampler = ClockSampler(local_rank)
    sampler.start()
    sampler.wait_ready()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_region0 = time.time()
    e0.record()
    for s in range(args.steps):
        for l in range(wl.layers):
            binding.ds_verify_attn(prof_args.get((s, l), step.verify_args[l]))
        step.gather()
        step.accept()
        step.commit()
    e1.record()
    torch.cuda.synchronize()
    t_region1 = time.time()
    barrier()
    clocks = sampler.stop(t_region0, t_region1)
    ms = e0.elapsed_time(e1) / args.steps
    split_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if world > 1:
        ms = max_over_ranks(ms, dev)

    # the post-accept commit alone, on each tree's deepest root-to-leaf path
    # (the longest accepted path the tree allows): it moves n rows per
    # sequence, K and V, in every layer (read + write)
    deep, n_acc = [], []
    for b in range(wl.batch):
        n0 = st.tree_offsets[b]
        par = st.parents[n0:n0 + st.tree_sizes[b]]
        depth = [0] * len(par)
        for j in range(1, len(par)):
            depth[j] = depth[par[j]] + 1
        leaf = max(range(len(par)), key=lambda j: (depth[j], -j)) if par else 0
        chain = []
        while par and leaf > 0:
            chain.append(leaf)
            leaf = par[leaf]
        chain.reverse()
        deep.append(chain + [-1] * (binding.DS_MAX_TREE_NODES - len(chain)))
        n_acc.append(len(chain))
    c_new = torch.empty(wl.batch, **i32)
    c_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    c_args = binding.commit_args(inp.k_cache, inp.v_cache, inp.page_table, inp.ctx_lens,
                                 inp.tree_offsets, torch.tensor(deep, **i32),
                                 torch.tensor(n_acc, **i32), new_ctx_lens=c_new,
                                 workspace=c_ws, kv_layout=args.kv_layout)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    reps = 20
    binding.ds_kv_commit(c_args)
    c0.record()
    for _ in range(reps):
        binding.ds_kv_commit(c_args)
    c1.record()
    torch.cuda.synchronize()
    assert binding.ds_device_status(c_ws) == 0
    commit_us = c0.elapsed_time(c1) * 1e3 / reps
    commit_bytes = sum(n_acc) * wl.num_kv_heads * wl.head_dim * 2 * 2 * 2 * wl.layers

    # retrieval (top-k + gather) and acceptance alone, each over its own
    # algorithmic bytes: the compact tokens' K and V read and written; the
    # logits read (target, plus draft for rejection)
    def _alone(fn):
        fn()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(reps):
            fn()
        a1.record()
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) * 1e3 / reps
    gather_us = _alone(step.gather)
    accept_us = _alone(step.accept)
    assert step.device_status() == 0
    compact_tokens = int(step.out_len.sum().item())
    gather_bytes = compact_tokens * wl.num_kv_heads * wl.head_dim * 2 * 2 * 2
    accept_bytes = st.n_nodes * wl.vocab * 4 * (2 if mode == "reject" else 1)

    # compact append between retrievals: the root and the accepted path
    # (1 + n tokens) appended behind a compact cache with room for them
    cap2 = step.capacity + 64
    kvh, hd = wl.num_kv_heads, wl.head_dim
    a_k = torch.zeros(wl.batch, cap2, kvh, hd, dtype=torch.bfloat16, device=dev)
    a_v = torch.zeros_like(a_k)
    a_pos = torch.empty(wl.batch, cap2, **i32)
    a_len = torch.empty(wl.batch, **i32)
    a_ids = torch.empty(wl.batch, max(wl.top_k, 1), **i32)
    a_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    binding.ds_chunk_topk_gather(binding.gather_args(
        step.scores, inp.ctx_lens, inp.src_k, inp.src_v, inp.page_table,
        chunk_size=wl.chunk_size, top_k=wl.top_k, window=wl.window, out_k=a_k,
        out_v=a_v, out_positions=a_pos, out_len=a_len, out_chunk_ids=a_ids,
        workspace=a_ws, kv_layout=args.kv_layout, rope_base=wl.rope_base))
    n_app = [1 + n for n in n_acc]
    to_t = inp.ctx_lens + torch.tensor(n_app, **i32)
    app_args = binding.append_args(inp.src_k, inp.src_v, inp.page_table, inp.ctx_lens,
                                   to_t, out_k=a_k, out_v=a_v, out_positions=a_pos,
                                   out_len=a_len, workspace=a_ws,
                                   kv_layout=args.kv_layout, rope_base=wl.rope_base)
    a_reps = max(1, min(5, 64 // max(n_app)))
    c0.record()
    for _ in range(a_reps):
        binding.ds_compact_append(app_args)
    c1.record()
    torch.cuda.synchronize()
    assert binding.ds_device_status(a_ws) == 0
    append_us = c0.elapsed_time(c1) * 1e3 / a_reps
    append_bytes = sum(n_app) * kvh * hd * 2 * 2 * 2   # K and V, read + write
    del a_k, a_v

    # end to end: pinned host inputs in, results out, every step
    e2e_ms, h2d, d2h = (None, 0, 0) if args.no_e2e else \
        _end_to_end(step, inp, args, world, dev, barrier)
    assert step.device_status() == 0

    if rank != 0:
        return
    kvb = _kv_bytes(wl, st)
    peak, peak_kind = _peaks()
    us = ms * 1e3 / (wl.layers * world)
    kv_gbs = kvb * wl.layers * world / (ms * 1e-3) / 1e9
    alg_bytes = kvb + _q_bytes(wl, st)
    achieved = alg_bytes / (split_ms * 1e-3) / 1e9
    src = os.path.join(ROOT, "long_context_speculative_ds_gb300", "csrc",
                       "verify_tc.cu")
    line = {
        "metric": METRIC, "value": round(us, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": _config(wl, st, args.kv_layout),
        "kv_gbs": round(kv_gbs, 1),
        "hbm_frac": round(kv_gbs / peak, 4),
        "roofline": {"kernel": "verify split pass", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "split_pass_us": round(split_ms * 1e3, 2),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "traffic": _traffic_for(src)},
        "e2e": {"value": None if e2e_ms is None else
                round(e2e_ms * 1e3 / (wl.layers * world), 3),
                "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "committed and tree K/V stay resident (model state);"
                        " per-step Q, tree, page table, logits, uniforms in,"
                        " path/bonus/chunk ids out; the step (copies and"
                        " kernels) captured once as a CUDA graph, replayed"
                        " and waited for every step"},
        "gather": {"us": round(gather_us, 2), "compact_tokens": compact_tokens,
                   "algorithmic_bytes": gather_bytes,
                   "gbs": round(gather_bytes / (gather_us * 1e-6) / 1e9, 1),
                   "rope": wl.rope_base > 0},
        "accept": {"us": round(accept_us, 2), "mode": mode,
                   "algorithmic_bytes": accept_bytes,
                   "gbs": round(accept_bytes / (accept_us * 1e-6) / 1e9, 1)},
        "kv_commit": {"us": round(commit_us, 2), "accepted": n_acc,
                      "algorithmic_bytes": commit_bytes,
                      "gbs": round(commit_bytes / (commit_us * 1e-6) / 1e9, 1)
                      if commit_us > 0 else None},
        "compact_append": {"us": round(append_us, 2), "rows": n_app,
                           "algorithmic_bytes": append_bytes,
                           "note": "not in the step: the step retrieves every cycle"},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    if not args.no_workloads and wl.name == DEFAULT_WORKLOAD:
        del inp, step, qs, ks, vs, sk, sv, acc
        torch.cuda.empty_cache()
        line["workloads"] = {n: workload_block(n, dev, peak) for n in OTHER_WORKLOADS}
    if world == 1 and not args.no_cpu_baseline:
        n_cpu = min(CPU_BASELINE_LAYERS, wl.layers)
        cst, clayers, csrc, cacc = cpu_inputs(wl, n_cpu)
        summ = oracle_summary(wl, oracle_time(wl, cst, clayers, csrc, cacc))
        us_cpu = summ.pop("value_us")
        line["cpu_baseline"] = {"value": round(us_cpu, 1), "unit": UNIT,
                                "cores": CORES, "kind": "oracle", **summ}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the 32K, 64K and ragged workloads' block")
    ap.add_argument("--kv-layout", choices=["NHD", "HND"], default="NHD")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count (profiling runs)")
    args = ap.parse_args()
    from long_context_speculative_ds_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.layers:
        wl = wl.replace(layers=args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
