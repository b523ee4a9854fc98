"""Benchmark of one DDTree verify step on GB300.

A step is the whole hot path on one batch: ddt_build_tree_visibility (tree
build and mask compile, one launch) -> ddt_verify_attn (split-KV partial +
combine) -> ddt_accept, captured once in a CUDA graph and replayed.  Inputs are seeded
and synthetic (workload "single_p4096_b32_h64": 1 request, prefix 4096,
budget 32, 64 heads, 576-wide bf16 latent rows in a 65536-row pool) and
resident in HBM.  Instead of flushing L2 the timed loop replays, round-robin,
enough independent copies of the step's buffers that their inputs cover three
L2s, so each replay reads cold data; the same graphs timed with a 256 MiB L2
flush before each replay (cold code as well) are printed beside it.

The reported metric is verify-attention TFLOP/s: algorithmic attention FLOPs
(2 * (576 + 512) per visible (query-head, kv) pair) per second of the whole
step.  KV GB/s, steps/s, a roofline object for ddt_verify_attn (timed with
CUDA events inside the same region), an end-to-end figure through host
buffers (one packed copy each way), the CPU oracle timed on the host cores,
the times of the KV commit and the sampling accept on their own (not part of
the step), and of the autoregressive step and a 128-token prefill chunk of the
same path, are printed beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --timeline [--workload W]   # per-kernel offsets inside a step

For N > 1 every rank runs its own copy of the workload (weak scaling, no
collective on the data path); the time is the max over ranks.  Under torchrun
the ranks come from its environment; without it, ``--gpus N`` starts the N
ranks itself (one process per GPU, rendezvous on 127.0.0.1).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "single_p4096_b32_h64"
METRIC = "verify-attn TFLOP/s and KV GB/s per step, % of roofline, 1xGB300"
# DRAM bytes (read + write) of one ddt_verify_attn call (partial + combine kernels) on
# this workload, from an ncu capture of both kernels (dram__bytes_read.sum +
# dram__bytes_write.sum per launch); valid only for the kernel sources it was taken
# from (their digests below): a change to them turns the field back to null.
PROFILE_TRAFFIC = {
    "bytes": 7314944 + 0 + 17345792 + 0,
    "sources": {
        "tree_speculative_decoding_gb300/csrc/ddt_attn_tc.cu":
            "dec334a03a3bce0678d35e19a04e4e3c7c40c8f0dd2989d8c6d888bb5fe998cd",
        "tree_speculative_decoding_gb300/csrc/ddt_attn_combine.cu":
            "fdca4d973e73b3ae2f8c739a639b1e174297c9d7950436970856c620e376355a",
        "tree_speculative_decoding_gb300/csrc/ddt_sm100.cuh":
            "25dcc37765dc9a4ca61c25bc5dd6eebe865d0a236e3a913d3add0bd656fc9804",
    },
}


def source_digest(rel):
    """sha256 of a source file's code with comments and whitespace removed, so that
    an edit to comments alone keeps a profile valid while any code change voids it."""
    import hashlib
    import re
    with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


def profiled_traffic():
    """The profiled DRAM bytes if the attention sources are unchanged since, else None."""
    for rel, digest in PROFILE_TRAFFIC["sources"].items():
        try:
            if source_digest(rel) != digest:
                return None
        except OSError:
            return None
    return PROFILE_TRAFFIC["bytes"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# -- timing aggregation shared by all ranks (tested on CPU with gloo) -----------
def reduce_over_ranks(elapsed_s: float, units: float, dist=None):
    """Max of the per-rank elapsed time and sum of per-rank units (FLOPs)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return elapsed_s, units
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        except Exception:
            pass
        if self.path:
            os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def replica_count(per_replica_bytes, l2_bytes, cover=3, lo=2, hi=64):
    """How many independent copies of a step's buffers make its inputs (the
    KV rows it reads plus its input arena) cover `cover` L2s when replayed
    round-robin, between `lo` and `hi`."""
    need = -(-cover * int(l2_bytes) // max(1, int(per_replica_bytes)))
    return max(lo, min(hi, need))


def workload_config(wl):
    """The workload's shape, as both arms report it."""
    return {"workload": wl.name, "batch": wl.B, "heads": wl.H, "prefix": int(wl.prefix_len[0]),
            "budget": int(wl.budget[0]), "q_len": int(wl.q_len[0]), "topk": wl.K,
            "pool_rows": wl.pool_rows}


def run_device(args, rank, world, local_rank):
    import torch

    from tree_speculative_decoding_gb300 import workloads
    from tree_speculative_decoding_gb300.metrics import algorithmic_bytes, attn_flops, kv_bytes
    from tree_speculative_decoding_gb300.pipeline import VerifyStep

    dist = None
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)

    wl = workloads.preset(args.workload)
    # Inputs larger than L2 instead of a flush: R independent copies of the step's
    # buffers (inputs, KV pool, outputs, workspace), replayed round-robin, with R
    # chosen so that the step inputs of all copies (the KV rows the step reads plus
    # its input arena) fill at least three L2s.  Every replay then finds its data
    # cold while the kernels' code stays cached, as in a serving loop.
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 132 * 2 ** 20)
    st = VerifyStep(wl, dev)
    kvb = kv_bytes(wl.kv_indptr)
    per_replica = kvb + st.inputs.buf.numel()
    n_rep = replica_count(per_replica, l2_bytes)
    replicas = [st] + [VerifyStep(wl, dev) for _ in range(n_rep - 1)]
    for r in replicas:
        r.run()
    torch.cuda.synchronize()
    for r in replicas:
        r.check_device_errors()
    depth = st.depth.cpu().numpy()
    flops = attn_flops(wl.prefix_len, depth, wl.qo_indptr, wl.H)

    # the step is the one-call C-ABI step (ddt_verify_step): tree + mask,
    # attention, accept, captured once per copy and replayed; ddt_verify_attn
    # alone (partial + combine) is captured too, for the roofline object
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    step_graphs, attn_graphs = [], []
    for r in replicas:
        g, a = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                r.run_one_call(stream=stream)
            with torch.cuda.graph(a, stream=stream):
                r.verify_attn(stream=stream)
        step_graphs.append(g)
        attn_graphs.append(a)
    torch.cuda.synchronize()
    for g in step_graphs + attn_graphs:      # first replay of each graph (upload), untimed
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()

    # kernels launched per step: tree + mask (one launch), attention partial (+ combine), accept
    launches_per_step = st.launches_per_step
    turn = [0]

    def replay(graphs, ev):
        """Replays the next copy's graph between two events; step and
        attention replays share one counter, so a copy comes back only after
        every other copy has run."""
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            graphs[turn[0] % n_rep].replay()
            ev[1].record(stream)
        turn[0] += 1

    def new_events(n):
        return [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
                for _ in range(n)]

    for ev in new_events(args.warmup):
        replay(step_graphs, ev)
    torch.cuda.synchronize()

    events, attn_events = new_events(args.steps), new_events(args.steps)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            replay(step_graphs, events[i])
            replay(attn_graphs, attn_events[i])
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = clk.summary()
    step_ms = [a.elapsed_time(b) for a, b in events]
    attn_ms = [a.elapsed_time(b) for a, b in attn_events]
    elapsed = sum(step_ms) / 1e3
    elapsed_max, flops_all = reduce_over_ranks(elapsed, flops * args.steps, dist)

    # the same two graphs of copy 0 with the 256 MiB L2 flush before each replay
    # instead of the rotation (cold code and cold data), for comparison
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flushed_n = min(args.steps, 500)
    fl_step, fl_attn = new_events(flushed_n), new_events(flushed_n)
    for i in range(flushed_n):
        for g, ev in ((step_graphs[0], fl_step[i]), (attn_graphs[0], fl_attn[i])):
            with torch.cuda.stream(stream):
                flush.zero_()
                ev[0].record(stream)
                g.replay()
                ev[1].record(stream)
    torch.cuda.synchronize()
    flushed = {"ms_per_step": round(statistics.mean(a.elapsed_time(b) for a, b in fl_step), 5),
               "verify_attn_ms": round(statistics.mean(a.elapsed_time(b) for a, b in fl_attn), 5),
               "steps": flushed_n}

    # end to end through host buffers, one C-ABI call per step: a library-owned
    # graph (ddt_step_graph_create_io) that copies the step's inputs (one packed
    # buffer) from pinned host memory, runs the step and copies its result back to
    # pinned host memory: the accept results (accepted path, committed tokens,
    # bonus token, new lengths), which is what the host needs every step; the
    # attention output stays on the device for the layer after it.  The same with
    # the attention output and lse copied back too is timed beside it.  One such
    # graph per copy, rotated as in the timed loop.
    h_in = st.inputs.buf.cpu().pin_memory()
    h_res = torch.empty(st.results_bytes, dtype=torch.uint8).pin_memory()
    h_all = torch.empty_like(st.outputs.buf, device="cpu").pin_memory()
    h2d = h_in.numel() * h_in.element_size()

    def e2e_time(h_out):
        graphs = [r.step_graph(host_io=(h_in, h_out)) for r in replicas]
        for g in graphs:
            g.launch(stream)
        torch.cuda.synchronize()
        evs = new_events(max(10, args.steps // 10))
        for i, ev in enumerate(evs):
            with torch.cuda.stream(stream):
                ev[0].record(stream)
                graphs[i % n_rep].launch(stream)
                ev[1].record(stream)
        torch.cuda.synchronize()
        for g in graphs:
            g.close()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    e2e_ms = e2e_time(h_res)
    e2e_all_ms = e2e_time(h_all)
    for r in replicas:
        r.check_device_errors()
    rotation = (f"not flushed: inputs larger than L2, {n_rep} independent copies of the step's "
                f"buffers replayed round-robin (their step inputs {n_rep * per_replica / 1e6:.0f} "
                f"MB = {n_rep * per_replica / l2_bytes:.1f}x L2)")
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    commit_ms = time_commit(st, stream, flush)
    sampled_ms = time_sampled(st, stream, flush, wl.vocab)
    sampled_topp_ms = time_sampled(st, stream, flush, wl.vocab, top_p=0.9)
    sampled_topk_ms = time_sampled(st, stream, flush, wl.vocab, top_k=20)
    degenerate = time_degenerate(dev, stream, flush)
    hbm, tf_burst, tf_sus, peak_kind = measured_peaks()
    ms_per_step = elapsed_max * 1e3 / args.steps
    value = flops_all / elapsed_max / 1e12
    attn_mean_ms = statistics.mean(attn_ms)
    achieved = flops / (attn_mean_ms / 1e3) / 1e12
    t_roof_ms = max(flops / (tf_burst * 1e12), kvb / (hbm * 1e9)) * 1e3
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; N(0,1) bf16 q and latent KV; drafter top-k from "
                "log-softmax of N(0,3) logits)",
        "config": dict(workload_config(wl), num_splits=st.launched_splits,
                       l2=rotation,
                       timing="CUDA graph replay of the 4-stage step, CUDA events per step",
                       parallelism=f"replicas x{world}"),
        "kv_gbs": round(kvb * args.steps * world / elapsed_max / 1e9, 2),
        "steps_per_s": round(args.steps * world / elapsed_max, 1),
        "attn_flops_per_step": flops,
        "kv_bytes_per_step": kvb,
        "algorithmic_bytes_per_step": algorithmic_bytes(wl.kv_indptr, wl.total_q, wl.H, st.total_words),
        "verify_attn_ms": round(attn_mean_ms, 5),
        "verify_attn_median_ms": round(statistics.median(attn_ms), 5),
        "l2_flushed": dict(flushed, timing="copy 0's step and ddt_verify_attn graphs, a 256 MiB "
                           "write before each replay (cold code and data), mean"),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": tf_burst,
                     "unit": "TFLOP/s", "frac": round(achieved / tf_burst, 4),
                     "traffic": profiled_traffic(), "peak_source": f"{peak_kind} bf16 burst",
                     "kernel": "ddt_verify_attn (partial + combine)",
                     "t_roof_ms": round(t_roof_ms, 5),
                     "frac_of_sustained": round(achieved / tf_sus, 4)},
        "e2e": {"value": round(flops / (e2e_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": int(st.results_bytes),
                "call": "ddt_step_graph_launch of a ddt_step_graph_create_io graph: pinned host "
                        "inputs (top-k, indptrs, kv_indices, q, target argmax) -> step -> the "
                        "accept results to pinned host memory, copies rotated as in the timed "
                        "loop",
                "with_attention_output": {
                    "value": round(flops / (e2e_all_ms / 1e3) / 1e12, 3),
                    "ms_per_step": round(e2e_all_ms, 5),
                    "d2h_bytes_per_step": int(h_all.numel()),
                    "call": "the same graph also copying the fp32 attention output and lse back"}},
        "gpu_launches": launches_per_step * args.steps,
        "accept_sampled": {"ms": round(sampled_ms, 5), "top_p_0.9_ms": round(sampled_topp_ms, 5),
                           "top_k_20_ms": round(sampled_topk_ms, 5),
                           "timing": "ddt_tree_links + "
                           "ddt_accept_sampled after the step (temperature 1, no top-k or top-p unless named, vocab "
                           f"{wl.vocab}, seeded N(0,1.5) logits); graph replay, L2 flushed, median"},
        "commit_kv": {"ms": round(commit_ms, 5), "timing": "ddt_commit_kv alone after the step, each "
                      "request committing its deepest root-to-leaf path; graph replay, L2 flushed, "
                      "median"},
        "degenerate": dict(degenerate, timing="each graph replayed on its own after the step, "
                           "L2 flushed, median; autoregressive = the whole step at budget 0, "
                           "prefill = ddt_prefill_step (causal chain + mask, attention) for "
                           "128 new tokens"),
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, seconds=args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return line


def replay_median(body, stream, flush, reps):
    """Median device time of `body(stream)` captured as one CUDA graph and
    replayed `reps` times after 5 untimed replays, L2 flushed before each."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            body(stream)
    ts = []
    for i in range(reps + 5):
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
            a.record(stream)
            g.replay()
            e.record(stream)
        torch.cuda.synchronize()
        if i >= 5:
            ts.append(a.elapsed_time(e))
    return statistics.median(ts)


def time_commit(st, stream, flush, reps=200):
    """Median time of ddt_commit_kv alone (the step after accept), every request
    committing the root-to-leaf path of its deepest node (lowest index among the
    deepest), so that up to max_depth rows move per request."""
    import torch
    qo = st.qo_indptr.cpu().numpy()
    par = st.parent.cpu().numpy()
    dep = st.depth.cpu().numpy()
    W = st.wl.max_depth + 1
    acc = np.full((st.B, W), -1, np.int32)
    alen = np.zeros(st.B, np.int32)
    for b in range(st.B):
        lo, hi = int(qo[b]), int(qo[b + 1])
        node = int(np.argmax(dep[lo:hi]))
        path = [node]
        while path[-1] != 0:
            path.append(int(par[lo + path[-1]]))
        path.reverse()
        alen[b] = len(path)
        acc[b, :len(path)] = path
    st.accept_len.copy_(torch.from_numpy(alen))
    st.accepted_nodes.copy_(torch.from_numpy(acc))
    ms = replay_median(lambda s: st.commit_kv(stream=s), stream, flush, reps)
    st.check_device_errors()
    return ms


def time_sampled(st, stream, flush, vocab, reps=200, top_p=None, top_k=0):
    """Median time of the sampling accept (links + rejection sampling) on the
    step's tree with seeded target logits, temperature 1, top-k `top_k` (0:
    none) and top-p `top_p` (None: none)."""
    import torch
    from tree_speculative_decoding_gb300 import ddt
    dev = st.node_token.device
    rows = st.node_token.numel()
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    logits = torch.randn((rows, vocab), generator=gen, device=dev) * 1.5
    coins = torch.rand((rows, st.wl.K + 1), generator=gen, device=dev)
    temp = torch.ones(st.B, dtype=torch.float32, device=dev)
    tk = torch.full((st.B,), top_k, dtype=torch.int32, device=dev)
    tp = None if top_p is None else torch.full((st.B,), top_p, dtype=torch.float32, device=dev)
    fc, ns, ri = (torch.empty(rows, dtype=torch.int32, device=dev) for _ in range(3))
    out = [torch.empty_like(t) for t in (st.accept_len, st.accepted_nodes, st.commit_tokens, st.bonus)]

    def body(s):
        ddt.ddt_tree_links(st.parent, st.qo_indptr, fc, ns, ri, stream=s)
        ddt.ddt_accept_sampled(st.node_token, fc, ns, st.qo_indptr, logits, temp, tk, coins,
                               st.wl.max_depth, *out, stream=s, top_p=tp)
    with torch.cuda.stream(stream):
        body(stream)
    ms = replay_median(body, stream, flush, reps)
    st.check_device_errors()
    return ms


def time_degenerate(dev, stream, flush, reps=200):
    """The path's degenerate shapes, one request after a prefix of 4096 at 64
    heads: the autoregressive step (budget 0; tree, mask, attention and
    accept) and a prefill chunk of 128 new tokens under a causal mask (the
    tree replaced by a chain: ddt_prefill_step, chain + mask and attention)."""
    import torch
    from tree_speculative_decoding_gb300 import workloads
    from tree_speculative_decoding_gb300.metrics import attn_flops, kv_bytes
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    res = {}
    for name in ("ar_p4096_b0_h64", "prefill_p4096_t128_h64"):
        wl = workloads.preset(name)
        st = VerifyStep(wl, dev)
        if name.startswith("prefill"):
            def body(s, st=st):
                st.run_prefill(stream=s)
        else:
            def body(s, st=st):
                st.run_one_call(stream=s)
        with torch.cuda.stream(stream):
            body(stream)
        torch.cuda.synchronize()
        st.check_device_errors()
        flops = attn_flops(wl.prefix_len, st.depth.cpu().numpy(), wl.qo_indptr, wl.H)
        ms = replay_median(body, stream, flush, reps)
        st.check_device_errors()
        res[name] = {"ms": round(ms, 5), "tflops": round(flops / ms / 1e9, 3),
                     "kv_gbs": round(kv_bytes(wl.kv_indptr) / ms / 1e6, 2),
                     "q_len": int(wl.q_len[0]), "num_splits": st.launched_splits}
    return res


def step_timeline(workload, reps=50):
    """Where the time goes inside one step: the step graph replayed `reps`
    times (L2 flushed before each) under the CUDA activity trace of
    torch.profiler; per kernel, the median start and end in µs from the first
    kernel of the step.  Diagnostic only: no reported figure comes from a
    traced run."""
    import re
    import torch
    from torch.profiler import ProfilerActivity, profile
    from tree_speculative_decoding_gb300 import workloads
    from tree_speculative_decoding_gb300.pipeline import VerifyStep
    wl = workloads.preset(workload)
    st = VerifyStep(wl, "cuda:0")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        st.run_one_call(stream=stream)
    torch.cuda.synchronize()
    st.check_device_errors()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            st.run_one_call(stream=stream)

    def replays(n):
        for _ in range(n):
            with torch.cuda.stream(stream):
                flush.zero_()
                g.replay()
        torch.cuda.synchronize()
    replays(10)
    with profile(activities=[ProfilerActivity.CUDA]):   # the tracer's own start-up
        replays(3)
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        replays(reps)
    kernels = sorted((e.time_range.start, e.time_range.end, e.name) for e in prof.events()
                     if e.device_type.name == "CUDA")
    steps, cur = [], None
    for t0, t1, name in kernels:
        if "FillFunctor" in name:      # the L2 flush opens each step
            cur = []
            steps.append(cur)
        elif cur is not None:
            m = re.search(r"(\w+_kernel)", name)
            cur.append((t0, t1, m.group(1) if m else name[:48]))
    rows = {}
    for k in steps[5:]:
        if not k:
            continue
        base = k[0][0]
        for t0, t1, name in k:
            rows.setdefault(name, []).append((t0 - base, t1 - base))
    st.check_device_errors()
    out = {name: {"start_us": round(statistics.median(a for a, _ in v), 2),
                  "end_us": round(statistics.median(b for _, b in v), 2), "steps": len(v)}
           for name, v in rows.items()}
    return {"workload": workload, "num_splits": st.launched_splits, "kernels": out}


def oracle_step(wl, rows=None, nthreads=0):
    """One verify step of the CPU oracle (attention on `nthreads` threads, 0 = all);
    returns attention FLOPs of the rows it computed."""
    import oracle
    from tree_speculative_decoding_gb300.metrics import attn_flops
    tok, par, dep = oracle.build_tree(wl.topk_logp, wl.topk_ids, wl.root_id, wl.budget,
                                      wl.qo_indptr, wl.max_depth, wl.K)
    mask, mip = oracle.compile_visibility(par, wl.qo_indptr, wl.prefix_len)
    oracle.verify_attn(wl.q, wl.kv_pool, wl.kv_indices, wl.kv_indptr, wl.qo_indptr, mask, mip,
                       wl.H, wl.scale, rows=rows, nthreads=nthreads)
    oracle.accept(tok, par, wl.qo_indptr, wl.argmax_random, wl.max_depth)
    full = attn_flops(wl.prefix_len, dep, wl.qo_indptr, wl.H)
    if rows is None:
        return full
    return full * len(rows) / (wl.total_q * wl.H)


def cpu_baseline(wl, seconds=10.0):
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    total, t0, reps = 0.0, time.perf_counter(), 0
    while True:
        total += oracle_step(wl)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    # the same on one thread, over a bounded sample of rows
    rows = np.arange(min(256, wl.total_q * wl.H), dtype=np.int64)
    t1 = time.perf_counter()
    f1 = oracle_step(wl, rows, nthreads=1)
    d1 = time.perf_counter() - t1
    return {"value": round(total / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} full oracle verify steps of {wl.name} (tree, mask, fp64 attention "
                      f"over all {wl.total_q * wl.H} rows, accept) in {dt:.1f} s",
            "single_thread": {"value": round(f1 / d1 / 1e12, 6), "cores": 1,
                              "sample": f"one oracle step with fp64 attention for {len(rows)} of "
                                        f"{wl.total_q * wl.H} rows in {d1:.2f} s"}}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, on this workload."""
    if rank != 0:
        return None
    import oracle
    from tree_speculative_decoding_gb300 import workloads
    oracle.build()
    wl = workloads.preset(args.workload)
    H = wl.H
    # bounded sample per step: the first 256 rows (4 nodes x 64 heads) of the step
    rows = np.arange(min(256, wl.total_q * H), dtype=np.int64)
    for _ in range(args.warmup):
        oracle_step(wl, rows)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_step(wl, rows)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"per step: oracle tree + mask + accept and fp64 attention for {len(rows)} of "
              f"{wl.total_q * H} rows of {args.workload}")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(wl), timing="host wall clock per oracle step",
                           parallelism="rank 0 only"),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                             "cores": oracle.num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def launch_ranks(n, argv):
    """Runs this script as n ranks (RANK / LOCAL_RANK / WORLD_SIZE / MASTER_* set
    as torchrun sets them) and returns the first non-zero exit code, else 0.
    Rank 0's JSON line reaches stdout unchanged; the other ranks print none."""
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()),
               WORLD_SIZE=str(n), LOCAL_WORLD_SIZE=str(n))
    procs = [subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv],
                              env=dict(env, RANK=str(r), LOCAL_RANK=str(r)))
             for r in range(n)]
    codes = [p.wait() for p in procs]
    return next((c for c in codes if c != 0), 0)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timeline", action="store_true",
                    help="print per-kernel start/end offsets inside one step (diagnostic)")
    ap.add_argument("--source-digests", action="store_true",
                    help="print the digests of the profiled attention sources and exit")
    args = ap.parse_args(argv)
    if args.source_digests:
        print(json.dumps({rel: source_digest(rel) for rel in PROFILE_TRAFFIC["sources"]}, indent=1))
        return
    if args.timeline:
        print(json.dumps(step_timeline(args.workload)), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv)))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_device(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
