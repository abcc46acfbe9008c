"""Benchmark of the tree-attention + greedy-verification hot path on GB300.

One step = one jf_tree_attention call plus one jf_tree_verify call over one
batch of seeded synthetic inputs: the Qwen3-8B attention shape (32 query
heads, 8 KV heads, head_dim 128), prefix 4096, a 256-node draft tree, and
256 x 151936 bf16 logits with a planted accepted path of length 10.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica on its own GPU (the path has no exchange step). Timing is the max
over ranks between barriers.

Timed region: the K steps are captured once into CUDA graphs and replayed,
with events on the launch stream before and after. The inputs rotate over
enough device copies that each step's data (105 MB) was evicted from the
126 MB L2 by the steps in between. The rooflines divide by the per-call
time of K back-to-back jf_tree_attention calls (tree_attention and
split_combine kernels) and of K jf_tree_verify calls (argmax_chunk and
accept_walk), timed the same way in the same clock window. Events the
library records around each kernel, in a traced copy of the step graph,
give per-kernel figures that include each launch gap. e2e times the
public calls eagerly on inputs in pinned host memory: each step's inputs
are copied to the device (on a second stream, into the other of two input
sets, while the previous step computes) and its results read back.
`--impl reference` times the fp64 CPU oracle on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "qwen3_8b_tree256"
METRIC = "tree-attn µs/step & % roofline (TFLOP/s | HBM GB/s); verify nodes/s"
L2_BYTES = 126 * 2 ** 20
MAX_DEPTH = 16
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def max_over_ranks(values, world: int, device):
    """Element-wise maximum of the floats `values` over all ranks (the values
    themselves on one rank): every timing is the slowest rank's."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], swp=f[8]))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 0.25 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded)}


def kernel_source_hash() -> str:
    """Hash of the sources that define the attention kernel, to tie a stored
    ncu traffic figure to the exact code it was measured on."""
    h = hashlib.sha256()
    for f in ("jf_attn.cu", "jf_common.cuh"):
        h.update(open(os.path.join(ROOT, "tree_masked_attention_causal_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def stored_traffic():
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get("tree_attention")
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent


# ------------------------------------------------------------ CPU oracle leg

def time_oracle(inp, target_s: float = 8.0):
    """Time the oracle on a bounded sample of one step and scale it to a full
    step. Returns (us_per_step, sample_description, threads)."""
    import numpy as np
    import oracle
    B, N = inp["parents"].shape
    # calibrate on 2 nodes, then take as many as fit the budget
    t0 = time.perf_counter()
    oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["prefix_lens"], inp["tree_k"],
                          inp["tree_v"], inp["parents"], inp["n_nodes"], sel=[(0, 0), (0, N - 1)])
    per_node = (time.perf_counter() - t0) / 2
    n_attn = int(max(2, min(N, 0.7 * target_s / max(per_node, 1e-6))))
    sel = [(0, int(i)) for i in np.linspace(0, N - 1, n_attn).round().astype(int)]
    t0 = time.perf_counter()
    oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["prefix_lens"], inp["tree_k"],
                          inp["tree_v"], inp["parents"], inp["n_nodes"], sel=sel)
    t_attn = time.perf_counter() - t0
    n_rows = min(B * N, 64)
    lg = inp["logits"].reshape(B * N, -1)[:n_rows]
    t0 = time.perf_counter()
    oracle.argmax_rows(lg)
    t_arg = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.tree_verify(inp["logits"][:1, :1], inp["tokens"][:1, :1], inp["parents"][:1, :1],
                       inp["n_nodes"][:1].clamp(max=1), MAX_DEPTH)
    t_walk_fixed = time.perf_counter() - t0
    total_nodes = int(inp["n_nodes"].sum())
    us = 1e6 * (t_attn * total_nodes / len(sel) + t_arg * total_nodes / n_rows + t_walk_fixed)
    desc = (f"attention for {len(sel)} of {total_nodes} nodes (all heads) and argmax of {n_rows} of "
            f"{total_nodes} logits rows, scaled to a full step")
    return us, desc, oracle.num_threads(), t_attn + t_arg


def run_reference(args, rank, world):
    if rank != 0:
        return
    from tree_masked_attention_causal_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w)
    times = []
    desc, threads = "", 0
    n = max(1, min(args.steps, 3))
    for _ in range(n):
        us, desc, threads, _ = time_oracle(inp, target_s=min(20.0, 60.0 / n))
        times.append(us)
    us = statistics.median(times)
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": world,
            "steps": n, "warmup": 0, "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, None),
            "cpu_baseline": {"value": us, "unit": "us/step", "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, extra):
    c = {"workload": f"{w.name}: batch {w.batch}, {w.n_q_heads}q/{w.n_kv_heads}kv heads, head_dim {w.head_dim}, "
                     f"prefix {w.prefix_min}" + (f"-{w.prefix_max}" if w.prefix_max != w.prefix_min else "") +
                     f", tree {w.max_nodes} nodes, vocab {w.vocab}",
         "batch": w.batch, "tree_nodes": w.max_nodes, "prefix": w.prefix_max, "vocab": w.vocab}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- GPU leg

def run_gpu(args, rank, world, local):
    import torch
    import torch.distributed as dist
    from tree_masked_attention_causal_gb300 import _build, binding as jb, synth

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    jb.load()

    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w)
    B, N, Hq, d = inp["q"].shape
    Hkv, Pcap, V = inp["k_cache"].shape[1], inp["k_cache"].shape[2], inp["logits"].shape[-1]
    shape = jb.make_shape(B, Hq, Hkv, d, N, Pcap, V)
    names = ["q", "k_cache", "v_cache", "prefix_lens", "tree_k", "tree_v", "parents", "n_nodes", "tokens", "logits"]
    step_bytes = sum(inp[k].numel() * inp[k].element_size() for k in names)
    R = max(2, math.ceil(3 * L2_BYTES / step_bytes))
    copies = [{k: inp[k].to(dev) for k in names} for _ in range(R)]
    ws = torch.empty(jb.jf_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    out = torch.empty_like(copies[0]["q"])
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty(B, MAX_DEPTH + 1, dtype=torch.int32, device=dev)
    am = torch.empty(B, N, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(c):
        jb.jf_tree_attention(c["q"], c["k_cache"], c["v_cache"], c["prefix_lens"], c["tree_k"], c["tree_v"],
                             c["parents"], c["n_nodes"], out, shape, ws, status=status)
        jb.jf_tree_verify(c["logits"], c["tokens"], c["parents"], c["n_nodes"], alen, path, am, shape, MAX_DEPTH, ws,
                          status=status)

    # warm-up (eager) and a correctness check of the planted path
    for i in range(max(3, args.warmup)):
        step(copies[i % R])
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status flag raised"
    assert int(alen[0].item()) == int(inp["planted_len"][0]), "planted accept length not recovered"

    # graphs of G steps each; K = G * M. Graph A (timed) holds only the
    # library's kernels, so the prep -> attention programmatic launch edge
    # stays intact; graph B is the same steps with an event pair around every
    # kernel, replayed right after A for the per-kernel durations.
    K = args.steps
    G = max(g for g in range(1, min(K, 250) + 1) if K % g == 0)
    M = K // G
    graph = torch.cuda.CUDAGraph()
    launches0 = jb.jf_kernel_launch_count()
    with torch.cuda.graph(graph):
        for i in range(G):
            step(copies[i % R])
    launches_per_step = (jb.jf_kernel_launch_count() - launches0) / G
    # The two calls alone, G back-to-back calls per graph, each on inputs that
    # left L2 since their last use: the attention inputs (21 MB a copy)
    # rotate over more copies than the whole steps do.
    attn_names = ["q", "k_cache", "v_cache", "prefix_lens", "tree_k", "tree_v", "parents", "n_nodes"]
    attn_bytes_in = sum(inp[k].numel() * inp[k].element_size() for k in attn_names)
    RA = max(R, math.ceil(3 * L2_BYTES / attn_bytes_in))
    acopies = copies + [{k: inp[k].to(dev) for k in attn_names} for _ in range(RA - R)]

    def attn_call(c):
        jb.jf_tree_attention(c["q"], c["k_cache"], c["v_cache"], c["prefix_lens"], c["tree_k"], c["tree_v"],
                             c["parents"], c["n_nodes"], out, shape, ws, status=status)

    def verify_call(c):
        jb.jf_tree_verify(c["logits"], c["tokens"], c["parents"], c["n_nodes"], alen, path, am, shape, MAX_DEPTH, ws,
                          status=status)

    for i in range(3):
        attn_call(acopies[i % RA])
        verify_call(copies[i % R])
    torch.cuda.synchronize()
    g_attn, g_verify = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_attn):
        for i in range(G):
            attn_call(acopies[i % RA])
    with torch.cuda.graph(g_verify):
        for i in range(G):
            verify_call(copies[i % R])
    max_kernels = 8
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_kernels * G)]
    traced = torch.cuda.CUDAGraph()
    jb.jf_trace_kernels(events, max_kernels * G)
    with torch.cuda.graph(traced):
        for i in range(G):
            step(copies[i % R])
    n_traced = jb.jf_trace_count()
    trace_names = [jb.jf_trace_name(k) for k in range(n_traced)]
    jb.jf_trace_kernels(None, 0)
    for g in (graph, g_attn, g_verify, traced):      # untimed
        g.replay()
    torch.cuda.synchronize()

    ev = lambda: torch.cuda.Event(enable_timing=True)
    start, end, a0, a1, v0, v1 = ev(), ev(), ev(), ev(), ev(), ev()
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(M):
            graph.replay()
        end.record()
        a0.record()
        for _ in range(M):
            g_attn.replay()
        a1.record()
        v0.record()
        for _ in range(M):
            g_verify.replay()
        v1.record()
        traced.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    clocks = clk.summary()
    total_ms, attn_call_ms, verify_call_ms = max_over_ranks(
        [start.elapsed_time(end), a0.elapsed_time(a1) / K, v0.elapsed_time(v1) / K], world, dev)

    # per-kernel durations of the traced replay: each includes its launch
    # gap after the previous event, without programmatic overlap
    per = {}
    for k, name in enumerate(trace_names):
        per.setdefault(name, []).append(events[2 * k].elapsed_time(events[2 * k + 1]))
    avg = {n: statistics.mean(v) for n, v in per.items()}

    # e2e through the public calls: pinned host inputs, an H2D copy of every
    # step's inputs and a D2H read of every step's results. The copy of step
    # i + 1's inputs runs on a second stream, into the other of two device
    # input sets, while step i computes.
    host = {k: inp[k].pin_memory() for k in names}
    dev_in = [{k: torch.empty_like(copies[0][k]) for k in names} for _ in range(2)]
    h_alen = torch.empty(B, dtype=torch.int32).pin_memory()
    h_path = torch.empty(B, MAX_DEPTH + 1, dtype=torch.int32).pin_memory()
    h_am = torch.empty(B, N, dtype=torch.int32).pin_memory()
    K_e2e = max(3, min(K, 50))
    compute = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        j = i % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[j])          # step i - 2 is done with set j
            for k in names:
                dev_in[j][k].copy_(host[k], non_blocking=True)
            copied[j].record(copy_stream)

    def run(i):
        j = i % 2
        compute.wait_event(copied[j])
        step(dev_in[j])
        consumed[j].record(compute)
        h_alen.copy_(alen, non_blocking=True)
        h_path.copy_(path, non_blocking=True)
        h_am.copy_(am, non_blocking=True)

    def e2e_steps(n):
        copy_stream.wait_stream(compute)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            run(i)

    e2e_steps(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(K_e2e)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1)], world, dev)[0]
    assert int(h_alen[0]) == int(inp["planted_len"][0])

    flops = synth.attention_flops(inp["parents"], inp["n_nodes"], inp["prefix_lens"], Hq, d)
    abytes = synth.attention_bytes(inp["prefix_lens"], inp["n_nodes"], Hq, Hkv, d)
    vbytes = synth.verify_bytes(inp["n_nodes"], V)
    pk, pk_src = peaks()
    achieved = flops / (attn_call_ms * 1e-3) / 1e12
    argmax_gbs = vbytes / (verify_call_ms * 1e-3) / 1e9
    traffic = stored_traffic()
    nodes = int(inp["n_nodes"].sum())

    if rank == 0:
        us_step = total_ms * 1e3 / (K * world)
        cpu_us, cpu_desc, cpu_threads, _ = time_oracle(inp, target_s=args.cpu_seconds)
        line = {
            "metric": METRIC, "value": us_step, "unit": "us/step", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": total_ms / K, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, {"l2": f"inputs rotate over {R} device copies ({R * step_bytes / 2**20:.0f} MB "
                                          f"> L2); attention-only calls over {RA} copies of their inputs",
                                    "graph_steps": G, "parallelism": f"replicas x{world}"}),
            "attn_us": attn_call_ms * 1e3, "verify_us": verify_call_ms * 1e3,
            "call_timing": "graphs of back-to-back jf_tree_attention calls and of jf_tree_verify calls, K each, "
                           "events on the launch stream, same clock window as the steps",
            "kernel_us": {n: v * 1e3 for n, v in avg.items()},
            "kernel_timing": "event pair around each kernel in a traced copy of the step graph; each figure "
                             "includes the kernel's launch gap and loses the programmatic overlap",
            "attn_tflops": achieved,
            "attn_roofline_frac": max(flops / (pk["bf16_tflops"] * 1e12), abytes / (pk["hbm_gbs"] * 1e9))
            / (attn_call_ms * 1e-3),
            "verify_gbs": argmax_gbs,
            "verify_nodes_per_s": nodes / (verify_call_ms * 1e-3),
            "roofline": {"bound": "tensor", "kernel": "tree_attention (+ split_combine: one jf_tree_attention call)",
                         "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / pk["bf16_tflops"], "peak_source": f"{pk_src} bf16 burst",
                         "traffic": None if traffic is None else traffic["bytes_per_launch"],
                         "algorithmic": flops},
            "argmax_roofline": {"bound": "hbm", "kernel": "argmax_chunk (+ accept_walk: one jf_tree_verify call)",
                                "achieved": argmax_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": argmax_gbs / pk["hbm_gbs"], "algorithmic": vbytes},
            "cpu_baseline": {"value": cpu_us, "unit": "us/step", "cores": cpu_threads, "kind": "oracle",
                             "sample": cpu_desc},
            "e2e": {"value": e2e_ms * 1e3 / (K_e2e * world), "unit": "us/step",
                    "h2d_bytes_per_step": step_bytes, "d2h_bytes_per_step": 4 * (B + B * (MAX_DEPTH + 1) + B * N)},
            "gpu_launches": int(round(launches_per_step * K)),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local)


if __name__ == "__main__":
    main()
