"""Seeded synthetic inputs for tree attention and greedy tree verification.

This module draws trees, tensors, token ids and logits. It holds none of the
method's arithmetic: it never evaluates attention, never takes an argmax and
never walks a tree to decide acceptance. The accepted path is planted *by
construction*. Every node u gets a token ``top[u]`` that is written into its
logits row at +16.0. Every other entry is a N(0, 1) draw clamped to [-8, 8],
so ``top[u]`` is that row's unique maximum. The path's tokens copy the
``top`` of their parent. Every other child of a path node gets a token that
differs from its parent's ``top``.

The workloads follow the method's setting: Qwen3-8B / Qwen3-30B-A3B
attention shapes, vocabulary 151936, and draft-tree budgets of 16 and 256
nodes. Sources: "JetFlow: Scaling Speculative Decoding with Parallel Tree
Drafting" (blog), section "Empirical Results"; the paper's section 1
Introduction, on tree budgets 16 and 256.

Both the CUDA path's tests and the fp64 oracle's tests draw from this module.
Neither side imports the other.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch

# Planted logit for a node's chosen top token. N(0,1) draws are clamped to
# [-CLAMP, CLAMP], so no other entry can tie with or exceed it.
PLANT_VALUE = 16.0
CLAMP = 8.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes plus the rules used to draw the trees."""

    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    max_nodes: int
    prefix_min: int          # prefix length is uniform in [prefix_min, prefix_max]
    prefix_max: int
    prefix_cap: int          # rows reserved per (sequence, kv-head) in the KV cache
    vocab: int
    depth_limit: int         # every node has depth <= depth_limit (root depth 0)
    branch_limit: Optional[int]  # max children per node, None = unlimited
    accept_min: int          # planted accept length (path nodes incl. root),
    accept_max: int          # uniform in [accept_min, accept_max]
    seed: int


# The five workloads. Seeds are 20260 + index.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 4, 1, 64, 16, 64, 64, 64, 1024, 4, None, 3, 3, 20260),
    "qwen3_8b_tree16": Workload("qwen3_8b_tree16", 1, 32, 8, 128, 16, 2048, 2048, 2048,
                                151936, 8, None, 5, 5, 20261),
    "qwen3_8b_tree256": Workload("qwen3_8b_tree256", 1, 32, 8, 128, 256, 4096, 4096, 4096,
                                 151936, 16, 8, 10, 10, 20262),
    "qwen3_30b_a3b_tree256": Workload("qwen3_30b_a3b_tree256", 1, 32, 4, 128, 256, 8192, 8192,
                                      8192, 151936, 16, 8, 8, 8, 20263),
    "serving_16x64": Workload("serving_16x64", 16, 32, 8, 128, 64, 512, 16384, 16384, 151936,
                              10, None, 1, 8, 20264),
}


def _randint(gen: torch.Generator, lo: int, hi: int) -> int:
    """Uniform integer in [lo, hi] (inclusive)."""
    return int(torch.randint(lo, hi + 1, (1,), generator=gen).item())


def random_tree(gen: torch.Generator, n: int, depth_limit: int,
                branch_limit: Optional[int]) -> List[int]:
    """Random topological tree: parents[0] = -1; node i > 0 takes a parent
    uniformly among earlier nodes whose depth is < depth_limit and whose child
    count is < branch_limit."""
    parents = [-1]
    depth = [0]
    kids = [0]
    for i in range(1, n):
        cand = [u for u in range(i) if depth[u] < depth_limit
                and (branch_limit is None or kids[u] < branch_limit)]
        if not cand:
            raise ValueError("tree rule leaves no admissible parent")
        u = cand[_randint(gen, 0, len(cand) - 1)]
        parents.append(u)
        depth.append(depth[u] + 1)
        kids.append(0)
        kids[u] += 1
    return parents


def node_depths(parents: List[int]) -> List[int]:
    """Depth of every node of a topological parents list (root depth 0)."""
    d = [0] * len(parents)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def chain_to_root(parents: List[int], i: int) -> List[int]:
    """Nodes from the root down to i (inclusive)."""
    out = []
    while i >= 0:
        out.append(i)
        i = parents[i]
    return out[::-1]


def _bf16_randn(gen: torch.Generator, shape, clamp: Optional[float] = None) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if clamp is not None:
        x.clamp_(-clamp, clamp)
    return x.to(torch.bfloat16)


def _token_other_than(gen: torch.Generator, vocab: int, avoid: int) -> int:
    t = _randint(gen, 0, vocab - 2)
    return t + 1 if t >= avoid else t


def plant_path(gen: torch.Generator, parents: List[int], n: int, vocab: int,
               accept_len: int):
    """Choose per-node top tokens and tree tokens so that the accepted path
    (root included) has exactly ``accept_len`` nodes.

    Returns (tokens, top, path) or None if no node has depth accept_len - 1.
    """
    depth = node_depths(parents[:n])
    ends = [i for i in range(n) if depth[i] == accept_len - 1]
    if not ends:
        return None
    end = ends[_randint(gen, 0, len(ends) - 1)]
    path = chain_to_root(parents, end)
    on_path = set(path)
    top = [_randint(gen, 0, vocab - 1) for _ in range(n)]
    tokens = [_randint(gen, 0, vocab - 1)]          # root token is never checked
    for c in range(1, n):
        u = parents[c]
        if c in on_path:
            tokens.append(top[u])
        elif u in on_path:
            tokens.append(_token_other_than(gen, vocab, top[u]))
        else:
            tokens.append(_randint(gen, 0, vocab - 1))
    return tokens, top, path


def make_inputs(w: Workload, seed: Optional[int] = None, kv_fill: float = 0.0,
                with_logits: bool = True) -> Dict[str, object]:
    """Draw every input of one call of each entry point, as CPU tensors.

    Layouts (row-major):
      q, out          bf16 [B, Nmax, Hq, d]
      k_cache/v_cache bf16 [B, Hkv, Pcap, d]; rows >= prefix_lens[b] hold kv_fill
      tree_k/tree_v   bf16 [B, Nmax, Hkv, d]
      prefix_lens     int32 [B]
      parents, tokens int32 [B, Nmax]
      n_nodes         int32 [B]
      logits          bf16 [B, Nmax, V]
    """
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, N = w.batch, w.max_nodes
    prefix_lens = [_randint(gen, w.prefix_min, w.prefix_max) for _ in range(B)]
    parents_all, tokens_all, top_all, paths, accept = [], [], [], [], []
    for b in range(B):
        L = _randint(gen, w.accept_min, w.accept_max)
        for _attempt in range(1000):
            par = random_tree(gen, N, w.depth_limit, w.branch_limit)
            planted = plant_path(gen, par, N, w.vocab, L)
            if planted is not None:
                break
        else:
            raise RuntimeError("could not draw a tree with the planted depth")
        tok, top, path = planted
        parents_all.append(par)
        tokens_all.append(tok)
        top_all.append(top)
        paths.append(path)
        accept.append(L)

    q = _bf16_randn(gen, (B, N, w.n_q_heads, w.head_dim))
    tree_k = _bf16_randn(gen, (B, N, w.n_kv_heads, w.head_dim))
    tree_v = _bf16_randn(gen, (B, N, w.n_kv_heads, w.head_dim))
    k_cache = torch.full((B, w.n_kv_heads, w.prefix_cap, w.head_dim), kv_fill,
                         dtype=torch.bfloat16)
    v_cache = torch.full_like(k_cache, kv_fill)
    for b in range(B):
        P = prefix_lens[b]
        k_cache[b, :, :P] = _bf16_randn(gen, (w.n_kv_heads, P, w.head_dim))
        v_cache[b, :, :P] = _bf16_randn(gen, (w.n_kv_heads, P, w.head_dim))

    out: Dict[str, object] = dict(
        workload=w,
        q=q, k_cache=k_cache, v_cache=v_cache, tree_k=tree_k, tree_v=tree_v,
        prefix_lens=torch.tensor(prefix_lens, dtype=torch.int32),
        parents=torch.tensor(parents_all, dtype=torch.int32),
        n_nodes=torch.full((B,), N, dtype=torch.int32),
        tokens=torch.tensor(tokens_all, dtype=torch.int32),
        top_tokens=torch.tensor(top_all, dtype=torch.int32),
        planted_len=torch.tensor(accept, dtype=torch.int32),
        planted_path=paths,
    )
    if with_logits:
        out["logits"] = make_logits(gen, B, N, w.vocab, out["top_tokens"])
    return out


def make_logits(gen: torch.Generator, B: int, N: int, vocab: int,
                top_tokens: torch.Tensor) -> torch.Tensor:
    """N(0,1) logits clamped to [-8, 8] in bf16, with +16 at each row's top token."""
    logits = _bf16_randn(gen, (B, N, vocab), clamp=CLAMP)
    flat = logits.view(B * N, vocab)
    rows = torch.arange(B * N)
    flat[rows, top_tokens.reshape(-1).long()] = PLANT_VALUE
    return logits


def paged_layout(k_cache: torch.Tensor, v_cache: torch.Tensor, prefix_lens: torch.Tensor, page_size: int,
                 seed: int = 0, spare: int = 3, spare_fill: float = float("nan")) -> Dict[str, object]:
    """The same prefix caches as pages of a shared pool, in a shuffled order.

      k_pages, v_pages  bf16 [num_pages, page_size, Hkv, d]: page j of
                        sequence b holds rows j*page_size .. of its cache
      block_table       int32 [B, Pcap / page_size]: the physical page of each
                        used logical page; -1 past the prefix
      num_pages         the used pages plus `spare` pages filled with
                        spare_fill (never referenced)
    """
    B, Hkv, Pcap, d = k_cache.shape
    assert Pcap % page_size == 0
    per_seq = Pcap // page_size
    used = [-(-int(prefix_lens[b]) // page_size) for b in range(B)]
    num_pages = sum(used) + spare
    gen = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=gen).tolist()
    k_pages = torch.full((num_pages, page_size, Hkv, d), spare_fill, dtype=torch.bfloat16)
    v_pages = torch.full_like(k_pages, spare_fill)
    table = torch.full((B, per_seq), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for j in range(used[b]):
            phys = perm[nxt]
            nxt += 1
            table[b, j] = phys
            rows = slice(j * page_size, (j + 1) * page_size)
            k_pages[phys] = k_cache[b, :, rows].transpose(0, 1)
            v_pages[phys] = v_cache[b, :, rows].transpose(0, 1)
    return dict(k_pages=k_pages, v_pages=v_pages, block_table=table, num_pages=num_pages, page_size=page_size)


# Draft logits of the sampling inputs are N(0, SAMPLE_SCALE^2); the
# target's are the draft's plus SAMPLE_NOISE * N(0, 1), so that the target
# agrees with the draft often but not always.
SAMPLE_SCALE = 2.0
SAMPLE_NOISE = 0.5


def make_sample_inputs(w: Workload, seed: Optional[int] = None, temperature: float = 1.0,
                       noise: float = SAMPLE_NOISE) -> Dict[str, torch.Tensor]:
    """Inputs of one stochastic verification call on workload w's shapes.

      draft_logits   bf16 [B, Nmax, V]: N(0, SAMPLE_SCALE^2) clamped to [-8, 8]
      target_logits  bf16 [B, Nmax, V]: draft + noise * N(0,1), clamped alike
      parents        int32 [B, Nmax]: trees drawn like make_inputs' trees
      tokens         int32 [B, Nmax]: node c's token is a draw from the
                     draft's distribution at its parent, softmax(draft_logits
                     [b, parent(c)] / temperature), as a sampling draft
                     proposes it; node 0's token is 0
      n_nodes        int32 [B] = Nmax
    """
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 7919)
    B, N, V = w.batch, w.max_nodes, w.vocab
    parents = torch.tensor([random_tree(gen, N, w.depth_limit, w.branch_limit) for _ in range(B)],
                           dtype=torch.int32)
    draft = (SAMPLE_SCALE * torch.randn((B, N, V), generator=gen)).clamp(-CLAMP, CLAMP).to(torch.bfloat16)
    target = (draft.float() + noise * torch.randn((B, N, V), generator=gen)).clamp(-CLAMP, CLAMP)
    target = target.to(torch.bfloat16)
    tokens = torch.zeros((B, N), dtype=torch.int32)
    for b in range(B):
        probs = torch.softmax(draft[b].float() / temperature, dim=-1)
        rows = probs[parents[b, 1:].long()]
        tokens[b, 1:] = torch.multinomial(rows, 1, generator=gen).reshape(-1).to(torch.int32)
    return dict(target_logits=target, draft_logits=draft, parents=parents, tokens=tokens,
                n_nodes=torch.full((B,), N, dtype=torch.int32))


def attention_flops(parents: torch.Tensor, n_nodes: torch.Tensor, prefix_lens: torch.Tensor,
                    n_q_heads: int, head_dim: int) -> int:
    """Algorithmic FLOP of one tree-attention call: only the (node, key) pairs
    the mask allows, 2 multiply-adds (QK^T and PV) of head_dim each."""
    total = 0
    for b in range(parents.shape[0]):
        n = int(n_nodes[b])
        depth = node_depths(parents[b, :n].tolist())
        total += sum(int(prefix_lens[b]) + d + 1 for d in depth)
    return 4 * head_dim * n_q_heads * total


def attention_bytes(prefix_lens: torch.Tensor, n_nodes: torch.Tensor, n_q_heads: int,
                    n_kv_heads: int, head_dim: int) -> int:
    """Algorithmic HBM bytes of one tree-attention call: each prefix K/V row
    and tree K/V row read once, q read once, out written once, plus the
    parents/lengths arrays."""
    P = int(prefix_lens.sum())
    N = int(n_nodes.sum())
    kv = 2 * 2 * n_kv_heads * head_dim * (P + N)
    qo = 2 * 2 * n_q_heads * head_dim * N
    return kv + qo + 4 * N + 8 * int(prefix_lens.numel())


def verify_bytes(n_nodes: torch.Tensor, vocab: int) -> int:
    """Algorithmic HBM bytes of one verify call: each valid logits row read
    once, plus tokens/parents (4 B each per node)."""
    N = int(n_nodes.sum())
    return 2 * N * vocab + 8 * N
