"""Benchmark of the tree-attention + greedy-verification hot path on GB300.

One step = one jf_tree_attention call plus one jf_tree_verify call over one
batch of seeded synthetic inputs. The headline workload is the Qwen3-8B
attention shape (32 query heads, 8 KV heads, head_dim 128), prefix 4096, a
256-node draft tree, and 256 x 151936 bf16 logits with a planted accepted
path of length 10.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--configs 0|1] [--config-steps KC]

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica on its own GPU (the path has no exchange step). Timing is the max
over ranks between barriers; `value` and `e2e` are per step of one replica
at every N, and `aggregate` sums the replicas' throughput.

Timed region: the K steps are captured once into CUDA graphs and replayed,
with events on the launch stream before and after. The inputs rotate over
enough device copies that each step's data (105 MB) was evicted from the
126 MB L2 by the steps in between. The rooflines divide by the per-call
time of K back-to-back jf_tree_attention calls (tree_attention and
split_combine kernels) and of K jf_tree_verify calls (argmax_chunk and
accept_walk), timed the same way in the same clock window, as are K
jf_tree_commit_kv calls (commit_kv) that append the accepted path to a
cache with room for it. Events the library records around each kernel, in
a traced copy of the step graph, give per-kernel figures that include each
launch gap. e2e times the public calls eagerly on inputs in pinned host
memory: each step's inputs are copied to the device (on a second stream,
into the other of two input sets, while the previous step computes) and
its results read back. The `configs` record repeats the call timings,
rooflines and an oracle sample for each of the five workloads.
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
    step. The attention sample is spread over every sequence's nodes and
    scaled by the keys each node attends to (prefix + depth + 1), so that
    ragged prefixes are weighted right. Returns (us_per_step, sample
    description, threads, seconds spent)."""
    import numpy as np
    import oracle
    from tree_masked_attention_causal_gb300 import synth
    B, N = inp["parents"].shape
    nodes, weight = [], []
    for b in range(B):
        n = int(inp["n_nodes"][b])
        depth = synth.node_depths(inp["parents"][b, :n].tolist())
        for i in range(n):
            nodes.append((b, i))
            weight.append(int(inp["prefix_lens"][b]) + depth[i] + 1)
    total_w = sum(weight)
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["prefix_lens"], inp["tree_k"], inp["tree_v"],
            inp["parents"], inp["n_nodes"])
    # calibrate on the two heaviest nodes, then take as many as fit the budget
    heavy = sorted(range(len(nodes)), key=lambda k: -weight[k])[:2]
    t0 = time.perf_counter()
    oracle.tree_attention(*args, sel=[nodes[k] for k in heavy])
    per_key = (time.perf_counter() - t0) / sum(weight[k] for k in heavy)
    mean_w = total_w / len(nodes)
    n_attn = int(max(2, min(len(nodes), 0.7 * target_s / max(per_key * mean_w, 1e-9))))
    pick = sorted(set(np.linspace(0, len(nodes) - 1, n_attn).round().astype(int).tolist()))
    t0 = time.perf_counter()
    oracle.tree_attention(*args, sel=[nodes[k] for k in pick])
    t_attn = time.perf_counter() - t0
    sample_w = sum(weight[k] for k in pick)
    n_rows = min(len(nodes), 64)
    lg = inp["logits"].reshape(B * N, -1)[:n_rows]
    t0 = time.perf_counter()
    oracle.argmax_rows(lg)
    t_arg = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.tree_verify(inp["logits"][:1, :1], inp["tokens"][:1, :1], inp["parents"][:1, :1],
                       inp["n_nodes"][:1].clamp(max=1), MAX_DEPTH)
    t_walk_fixed = time.perf_counter() - t0
    us = 1e6 * (t_attn * total_w / sample_w + t_arg * len(nodes) / n_rows + t_walk_fixed)
    desc = (f"attention for {len(pick)} of {len(nodes)} nodes (all heads; scaled by keys attended) and argmax "
            f"of {n_rows} of {len(nodes)} logits rows, scaled to a full step")
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


def graph_size(K: int) -> int:
    """Calls per captured graph: the largest divisor of K up to 250."""
    return max(g for g in range(1, min(K, 250) + 1) if K % g == 0)


# ---------------------------------------------------------------- GPU leg

class Calls:
    """One workload's inputs, resident on the device in enough copies that a
    call's inputs have left L2 since their last use, and the public calls on
    them: attention, verify, the step (both), and the KV commit of the
    accepted path."""

    STEP = ["q", "k_cache", "v_cache", "prefix_lens", "tree_k", "tree_v", "parents", "n_nodes", "tokens", "logits"]
    ATTN = ["q", "k_cache", "v_cache", "prefix_lens", "tree_k", "tree_v", "parents", "n_nodes"]

    def __init__(self, w, dev, G, torch, jb, synth):
        self.w, self.torch, self.jb, self.G = w, torch, jb, G
        inp = self.inp = synth.make_inputs(w)
        B, N, Hq, d = inp["q"].shape
        Hkv, Pcap, V = inp["k_cache"].shape[1], inp["k_cache"].shape[2], inp["logits"].shape[-1]
        self.B, self.N = B, N
        self.shape = jb.make_shape(B, Hq, Hkv, d, N, Pcap, V)
        self.step_bytes = sum(inp[k].numel() * inp[k].element_size() for k in self.STEP)
        self.R = max(2, math.ceil(3 * L2_BYTES / self.step_bytes))
        self.copies = [{k: inp[k].to(dev) for k in self.STEP} for _ in range(self.R)]
        attn_in = sum(inp[k].numel() * inp[k].element_size() for k in self.ATTN)
        self.RA = max(self.R, math.ceil(3 * L2_BYTES / attn_in))
        self.acopies = self.copies + [{k: inp[k].to(dev) for k in self.ATTN} for _ in range(self.RA - self.R)]
        self.ws = torch.empty(jb.jf_workspace_bytes(self.shape), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(self.copies[0]["q"])
        self.alen = torch.empty(B, dtype=torch.int32, device=dev)
        self.path = torch.empty(B, MAX_DEPTH + 1, dtype=torch.int32, device=dev)
        self.am = torch.empty(B, N, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # The commit appends up to MAX_DEPTH + 1 rows: it writes into caches
        # of its own with that much room above the longest prefix. Each of
        # the G commits of one graph takes its own copy of prefix_lens, all
        # restored by one copy at the head of the graph.
        self.shape_c = jb.make_shape(B, Hq, Hkv, d, N, Pcap + MAX_DEPTH + 1, V)
        self.kc = torch.zeros(B, Hkv, Pcap + MAX_DEPTH + 1, d, dtype=torch.bfloat16, device=dev)
        self.vc = torch.zeros_like(self.kc)
        self.pl_saved = inp["prefix_lens"].to(dev).repeat(G, 1)
        self.pl_slots = self.pl_saved.clone()
        self.c_alen = torch.empty_like(self.alen)
        self.c_path = torch.empty_like(self.path)
        # the same prefix caches as 16-row pages of a shuffled pool
        pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], 16, seed=w.seed)
        pool_bytes = 2 * pg["k_pages"].numel() * 2
        self.RP = min(G, max(2, math.ceil(3 * L2_BYTES / pool_bytes)))
        self.pages = [dict(k=pg["k_pages"].to(dev), v=pg["v_pages"].to(dev)) for _ in range(self.RP)]
        self.block_table = pg["block_table"].to(dev)
        self.num_pages = pg["num_pages"]
        # stochastic verification: target and draft logits with trees whose
        # tokens a sampling draft proposed, rotated like the other inputs
        sinp = synth.make_sample_inputs(w)
        snames = ["target_logits", "draft_logits", "tokens", "parents", "n_nodes"]
        self.sample_bytes = sum(sinp[k].numel() * sinp[k].element_size() for k in snames)
        self.RS = min(G, max(2, math.ceil(3 * L2_BYTES / self.sample_bytes)))
        self.scopies = [{k: sinp[k].to(dev) for k in snames} for _ in range(self.RS)]
        self.s_next = torch.empty(B, dtype=torch.int32, device=dev)
        # path scoring on the same draft logits and trees: top 8 per node, 64 candidates
        self.sc_k, self.sc_budget = 8, min(64, N * 8)
        f32 = dict(dtype=torch.float32, device=dev)
        self.sc_node, self.sc_path = torch.empty(B, N, **f32), torch.empty(B, N, **f32)
        self.sc_ttok = torch.empty(B, N, self.sc_k, dtype=torch.int32, device=dev)
        self.sc_tlp = torch.empty(B, N, self.sc_k, **f32)
        self.sc_cpar = torch.empty(B, self.sc_budget, dtype=torch.int32, device=dev)
        self.sc_ctok = torch.empty_like(self.sc_cpar)
        self.sc_cscore = torch.empty(B, self.sc_budget, **f32)
        self.s_alen = torch.empty_like(self.alen)
        self.s_path = torch.empty_like(self.path)

    def attn(self, i):
        c = self.acopies[i % self.RA]
        self.jb.jf_tree_attention(c["q"], c["k_cache"], c["v_cache"], c["prefix_lens"], c["tree_k"], c["tree_v"],
                                  c["parents"], c["n_nodes"], self.out, self.shape, self.ws, status=self.status)

    def verify(self, i, c=None):
        c = c or self.copies[i % self.R]
        self.jb.jf_tree_verify(c["logits"], c["tokens"], c["parents"], c["n_nodes"], self.alen, self.path, self.am,
                               self.shape, MAX_DEPTH, self.ws, status=self.status)

    def step(self, i, c=None):
        c = c or self.copies[i % self.R]
        self.jb.jf_tree_attention(c["q"], c["k_cache"], c["v_cache"], c["prefix_lens"], c["tree_k"], c["tree_v"],
                                  c["parents"], c["n_nodes"], self.out, self.shape, self.ws, status=self.status)
        self.verify(i, c)

    def commit(self, i):
        if i % self.G == 0:
            self.pl_slots.copy_(self.pl_saved)
        c = self.copies[i % self.R]
        self.jb.jf_tree_commit_kv(c["tree_k"], c["tree_v"], c["n_nodes"], self.c_alen, self.c_path, self.kc, self.vc,
                                  self.pl_slots[i % self.G], self.shape_c, MAX_DEPTH, status=self.status)

    def attn_paged(self, i):
        c, pg = self.acopies[i % self.RA], self.pages[i % self.RP]
        self.jb.jf_tree_attention_paged(c["q"], pg["k"], pg["v"], self.block_table, 16, self.num_pages,
                                        c["prefix_lens"], c["tree_k"], c["tree_v"], c["parents"], c["n_nodes"],
                                        self.out, self.shape, self.ws, status=self.status)

    def sample(self, i):
        c = self.scopies[i % self.RS]
        self.jb.jf_tree_verify_sample(c["target_logits"], c["draft_logits"], c["tokens"], c["parents"], c["n_nodes"],
                                      1.0, 1234, i, self.s_alen, self.s_path, self.s_next, self.shape, MAX_DEPTH,
                                      self.ws, status=self.status)

    def score(self, i):
        c = self.scopies[i % self.RS]
        self.jb.jf_tree_score(c["draft_logits"], c["tokens"], c["parents"], c["n_nodes"], 1.0, self.sc_k,
                              self.sc_budget, self.sc_node, self.sc_path, self.sc_ttok, self.sc_tlp, self.sc_cpar,
                              self.sc_ctok, self.sc_cscore, self.shape, self.ws, status=self.status)

    def warm(self, n):
        for i in range(n):
            self.step(i)
        self.torch.cuda.synchronize()
        assert int(self.status.item()) == 0, f"{self.w.name}: device status flag raised"
        want = self.inp["planted_len"].tolist()
        assert self.alen.tolist() == want, f"{self.w.name}: planted accept lengths not recovered"
        self.c_alen.copy_(self.alen)
        self.c_path.copy_(self.path)
        for i in range(min(n, self.G)):
            self.attn(i)
            self.commit(i)
            self.sample(i)
            self.score(i)
            self.attn_paged(i)
        self.torch.cuda.synchronize()
        assert int(self.status.item()) == 0, f"{self.w.name}: device status flag raised by the commit"

    def graph(self, fn):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g):
            for i in range(self.G):
                fn(i)
        return g

    def commit_bytes(self):
        """Algorithmic bytes of one commit: each accepted node's K and V rows
        (all KV heads) read from the tree and written to the cache."""
        Hkv, d = self.kc.shape[1], self.kc.shape[3]
        rows = int(self.inp["planted_len"].sum())
        return 2 * 2 * rows * Hkv * d * 2 + 4 * self.B * (MAX_DEPTH + 4)

    def rooflines(self, attn_ms, verify_ms, commit_ms, pk, synth, sample_ms=None, score_ms=None, paged_ms=None):
        inp, w = self.inp, self.w
        flops = synth.attention_flops(inp["parents"], inp["n_nodes"], inp["prefix_lens"], w.n_q_heads, w.head_dim)
        abytes = synth.attention_bytes(inp["prefix_lens"], inp["n_nodes"], w.n_q_heads, w.n_kv_heads, w.head_dim)
        vbytes = synth.verify_bytes(inp["n_nodes"], w.vocab)
        cbytes = self.commit_bytes()
        t_flop = flops / (pk["bf16_tflops"] * 1e12)
        t_byte = abytes / (pk["hbm_gbs"] * 1e9)
        nodes = int(inp["n_nodes"].sum())
        return {
            "attn_us": attn_ms * 1e3, "attn_tflops": flops / (attn_ms * 1e-3) / 1e12,
            "attn_gbs": abytes / (attn_ms * 1e-3) / 1e9, "attn_bound": "tensor" if t_flop >= t_byte else "hbm",
            "attn_roofline_frac": max(t_flop, t_byte) / (attn_ms * 1e-3),
            "attn_flop": flops, "attn_bytes": abytes,
            "verify_us": verify_ms * 1e3, "verify_gbs": vbytes / (verify_ms * 1e-3) / 1e9,
            "verify_hbm_frac": vbytes / (verify_ms * 1e-3) / (pk["hbm_gbs"] * 1e9),
            "verify_nodes_per_s": nodes / (verify_ms * 1e-3), "verify_bytes": vbytes,
            "commit_us": commit_ms * 1e3, "commit_gbs": cbytes / (commit_ms * 1e-3) / 1e9, "commit_bytes": cbytes,
            **({} if sample_ms is None else {
                "sample_us": sample_ms * 1e3, "sample_bytes": 2 * vbytes,
                "sample_gbs": 2 * vbytes / (sample_ms * 1e-3) / 1e9,
                "sample_hbm_frac": 2 * vbytes / (sample_ms * 1e-3) / (pk["hbm_gbs"] * 1e9)}),
            **({} if paged_ms is None else {
                "attn_paged_us": paged_ms * 1e3,
                "attn_paged_roofline_frac": max(t_flop, t_byte) / (paged_ms * 1e-3)}),
            **({} if score_ms is None else {
                "score_us": score_ms * 1e3, "score_bytes": vbytes,
                "score_gbs": vbytes / (score_ms * 1e-3) / 1e9,
                "score_hbm_frac": vbytes / (score_ms * 1e-3) / (pk["hbm_gbs"] * 1e9)}),
        }


def time_graphs(graphs, M, torch):
    """Replay each graph M times back to back; events on the launch stream
    around each run. Returns the milliseconds of each."""
    out = []
    for g in graphs:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(M):
            g.replay()
        b.record()
        out.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in out]


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
    pk, pk_src = peaks()

    # graphs of G calls each; K = G * M. Graph `graph` (timed) holds only the
    # library's kernels, so the programmatic launch edges stay intact;
    # `traced` is the same steps with an event pair around every kernel,
    # replayed right after for the per-kernel durations.
    K = args.steps
    G = graph_size(K)
    M = K // G
    w = synth.WORKLOADS[args.workload]
    H = Calls(w, dev, G, torch, jb, synth)
    H.warm(max(3, args.warmup))
    B, N = H.B, H.N
    launches0 = jb.jf_kernel_launch_count()
    graph = H.graph(H.step)
    launches_per_step = (jb.jf_kernel_launch_count() - launches0) / G
    g_attn, g_verify, g_commit, g_sample = H.graph(H.attn), H.graph(H.verify), H.graph(H.commit), H.graph(H.sample)
    g_score, g_paged = H.graph(H.score), H.graph(H.attn_paged)
    max_kernels = 8
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_kernels * G)]
    jb.jf_trace_kernels(events, max_kernels * G)
    traced = H.graph(H.step)
    n_traced = jb.jf_trace_count()
    trace_names = [jb.jf_trace_name(k) for k in range(n_traced)]
    jb.jf_trace_kernels(None, 0)
    for g in (graph, g_attn, g_verify, g_commit, g_sample, g_score, g_paged, traced):      # untimed
        g.replay()
    torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_step, t_attn, t_verify, t_commit, t_sample, t_score, t_paged = time_graphs(
            [graph, g_attn, g_verify, g_commit, g_sample, g_score, g_paged], M, torch)
        traced.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    clocks = clk.summary()
    assert int(H.status.item()) == 0, "device status flag raised in the timed region"
    total_ms, attn_ms, verify_ms, commit_ms, sample_ms, score_ms, paged_ms = max_over_ranks(
        [t_step, t_attn / K, t_verify / K, t_commit / K, t_sample / K, t_score / K, t_paged / K], world, dev)

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
    names = Calls.STEP
    host = {k: H.inp[k].pin_memory() for k in names}
    dev_in = [{k: torch.empty_like(H.copies[0][k]) for k in names} for _ in range(2)]
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
        H.step(i, dev_in[j])
        consumed[j].record(compute)
        h_alen.copy_(H.alen, non_blocking=True)
        h_path.copy_(H.path, non_blocking=True)
        h_am.copy_(H.am, non_blocking=True)

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
    assert h_alen.tolist() == H.inp["planted_len"].tolist()

    head = H.rooflines(attn_ms, verify_ms, commit_ms, pk, synth, sample_ms, score_ms, paged_ms)
    head["step_us"] = total_ms * 1e3 / K
    traffic = stored_traffic()
    cpu = time_oracle(H.inp, target_s=args.cpu_seconds) if rank == 0 else None
    head_desc = {"l2": f"inputs rotate over {H.R} device copies ({H.R * H.step_bytes / 2**20:.0f} MB > L2); "
                       f"attention-only calls over {H.RA} copies of their inputs", "graph_steps": G}

    # every workload: the three calls and the step, fewer steps each
    configs = {}
    cfg_clocks = None
    if args.configs:
        Kc = min(K, args.config_steps)
        Gc = graph_size(Kc)
        del graph, g_attn, g_verify, g_commit, g_sample, g_score, g_paged, traced
        with ClockSampler(local) as clk2:
            for name, wc in synth.WORKLOADS.items():
                if name == args.workload:
                    rec = dict(head)
                    rec.update({"steps": K, "l2": head_desc["l2"]})
                else:
                    Hc = Calls(wc, dev, Gc, torch, jb, synth)
                    Hc.warm(3)
                    gs = [Hc.graph(f) for f in (Hc.step, Hc.attn, Hc.verify, Hc.commit, Hc.sample, Hc.score,
                                                Hc.attn_paged)]
                    for g in gs:
                        g.replay()
                    torch.cuda.synchronize()
                    if world > 1:
                        dist.barrier()
                    ts = time_graphs(gs, Kc // Gc, torch)
                    assert int(Hc.status.item()) == 0, f"{name}: device status flag raised"
                    ts = max_over_ranks([t / Kc for t in ts], world, dev)
                    rec = Hc.rooflines(ts[1], ts[2], ts[3], pk, synth, ts[4], ts[5], ts[6])
                    rec.update({"step_us": ts[0] * 1e3, "steps": Kc,
                                "l2": f"inputs rotate over {Hc.R} device copies "
                                      f"({Hc.R * Hc.step_bytes / 2**20:.0f} MB); attention-only calls over "
                                      f"{Hc.RA} copies"})
                    if rank == 0:
                        o = time_oracle(Hc.inp, target_s=args.cpu_seconds / 3)
                        rec.update({"oracle_us_per_step": o[0], "oracle_cores": o[2], "oracle_sample": o[1]})
                    del gs, Hc
                    torch.cuda.empty_cache()
                if name == args.workload and cpu is not None:
                    rec.update({"oracle_us_per_step": cpu[0], "oracle_cores": cpu[2], "oracle_sample": cpu[1]})
                configs[name] = rec
        cfg_clocks = clk2.summary()

    if rank == 0:
        us_step = total_ms * 1e3 / K
        line = {
            "metric": METRIC, "value": us_step, "unit": "us/step", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": total_ms / K, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, dict(head_desc, parallelism=f"replicas x{world}")),
            "aggregate": {"steps_per_s": world * K / (total_ms * 1e-3),
                          "nodes_per_s": world * K * int(H.inp["n_nodes"].sum()) / (total_ms * 1e-3),
                          "note": "all replicas together; value and e2e are per step of one replica "
                                  "(the slowest rank)"},
            "attn_us": head["attn_us"], "verify_us": head["verify_us"], "commit_us": head["commit_us"],
            "sample_us": head["sample_us"], "score_us": head["score_us"], "attn_paged_us": head["attn_paged_us"],
            "call_timing": "graphs of back-to-back jf_tree_attention calls, of jf_tree_verify calls, of "
                           "jf_tree_commit_kv calls, of jf_tree_verify_sample calls (T = 1, a new Philox "
                           "offset each), of jf_tree_score calls (top 8, 64 candidates) and of "
                           "jf_tree_attention_paged calls (16-row pages of a shuffled pool), K each, events on the "
                           "launch stream, same clock window as the steps",
            "kernel_us": {n: v * 1e3 for n, v in avg.items()},
            "kernel_timing": "event pair around each kernel in a traced copy of the step graph; each figure "
                             "includes the kernel's launch gap and loses the programmatic overlap",
            "attn_tflops": head["attn_tflops"], "attn_roofline_frac": head["attn_roofline_frac"],
            "verify_gbs": head["verify_gbs"], "verify_nodes_per_s": head["verify_nodes_per_s"],
            "roofline": {"bound": "tensor", "kernel": "tree_attention (+ split_combine: one jf_tree_attention call)",
                         "achieved": head["attn_tflops"], "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": head["attn_tflops"] / pk["bf16_tflops"], "peak_source": f"{pk_src} bf16 burst",
                         "traffic": None if traffic is None else traffic["bytes_per_launch"],
                         "algorithmic": head["attn_flop"]},
            "argmax_roofline": {"bound": "hbm", "kernel": "argmax_chunk (+ accept_walk: one jf_tree_verify call)",
                                "achieved": head["verify_gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": head["verify_hbm_frac"], "peak_source": f"{pk_src} copy",
                                "algorithmic": head["verify_bytes"]},
            "cpu_baseline": {"value": cpu[0], "unit": "us/step", "cores": cpu[2], "kind": "oracle",
                             "sample": cpu[1]},
            "e2e": {"value": e2e_ms * 1e3 / K_e2e, "unit": "us/step",
                    "h2d_bytes_per_step": H.step_bytes,
                    "d2h_bytes_per_step": 4 * (B + B * (MAX_DEPTH + 1) + B * N)},
            "gpu_launches": int(round(launches_per_step * K)),
            "clocks": clocks,
        }
        if configs:
            line["configs"] = configs
            line["configs_timing"] = (f"per workload: graphs of {min(K, args.config_steps)} calls of each kind "
                                      f"(the headline workload: its K above); oracle on a bounded sample")
            line["configs_clocks"] = cfg_clocks
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
    ap.add_argument("--configs", type=int, default=1, help="1: also time every workload (the configs record)")
    ap.add_argument("--config-steps", type=int, default=1000)
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local)


if __name__ == "__main__":
    main()
