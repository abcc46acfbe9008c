"""Pins of the oracle's draft-side path scoring (CPU only).

The rule ("JetFlow: Scaling Speculative Decoding with Parallel Tree
Drafting", section "What JetFlow Does Differently"): a path's draft
probability is the product of conditionals, each on the concrete ancestor
tokens of its branch. The pins: node log-probabilities against
torch.log_softmax gathered at the tokens; path log-probabilities against
an ancestor-indicator matrix (built by transitive closure, not by the
oracle's chain walk) times the node values; exp(path log-prob) against the
frequency with which sampling the draft level by level reproduces a path;
uniform logits give -depth ln V in closed form; the top-k against a stable
descending torch.sort; the budgeted expansion against a brute-force sort of
every candidate.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from tree_masked_attention_causal_gb300 import synth


def bf16(x):
    return torch.tensor(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def ancestors_incl(parents, n):
    """A[c, j] = 1 iff j is c or an ancestor of c, by repeated squaring."""
    A = torch.eye(n, dtype=torch.float64)
    for c in range(1, n):
        A[c, parents[c]] = 1.0
    for _ in range(9):
        A = ((A @ A) > 0).double()
    return A


def case(seed, B=3, N=20, V=64, scale=2.0, branch=3):
    gen = torch.Generator().manual_seed(seed)
    parents = torch.tensor([synth.random_tree(gen, N, 10, branch) for _ in range(B)], dtype=torch.int32)
    draft = bf16(torch.randn((B, N, V), generator=gen).numpy() * scale)
    tokens = torch.randint(0, V, (B, N), generator=gen, dtype=torch.int32)
    return draft, tokens, parents, torch.full((B,), N, dtype=torch.int32)


@pytest.mark.parametrize("seed,T", [(0, 1.0), (1, 0.7), (2, 2.5)])
def test_node_and_path_logprobs_match_torch(seed, T):
    draft, tokens, parents, n = case(seed)
    B, N, V = draft.shape
    r = oracle.tree_score(draft, tokens, parents, n, T)
    lsm = torch.log_softmax(draft.double() / T, dim=-1)
    for b in range(B):
        par = parents[b].tolist()
        node = torch.zeros(N, dtype=torch.float64)
        for c in range(1, N):
            node[c] = lsm[b, par[c], tokens[b, c]]
        np.testing.assert_allclose(r["node_lp"][b], node.numpy(), rtol=0, atol=1e-12)
        path = ancestors_incl(par, N) @ node
        np.testing.assert_allclose(r["path_lp"][b], path.numpy(), rtol=0, atol=1e-11)


def test_uniform_logits_give_minus_depth_log_v():
    B, N, V = 2, 30, 128
    gen = torch.Generator().manual_seed(9)
    parents = torch.tensor([synth.random_tree(gen, N, 12, None) for _ in range(B)], dtype=torch.int32)
    tokens = torch.randint(0, V, (B, N), generator=gen, dtype=torch.int32)
    draft = bf16(np.full((B, N, V), 0.75))
    r = oracle.tree_score(draft, tokens, parents, torch.full((B,), N, dtype=torch.int32), 0.9)
    for b in range(B):
        depth = synth.node_depths(parents[b].tolist())
        np.testing.assert_allclose(r["path_lp"][b], -np.array(depth) * math.log(V), rtol=0, atol=1e-12)


def test_path_probability_is_the_frequency_of_sampling_it():
    """exp(path_lp) of the deepest node of a chain equals the frequency
    with which drawing each level from the draft reproduces the chain."""
    V, N, T = 4, 4, 1.0
    rng = np.random.default_rng(3)
    lg = rng.normal(size=(1, N, V)) * 1.0
    draft = bf16(lg)
    parents = torch.tensor([[-1, 0, 1, 2]], dtype=torch.int32)
    tokens = torch.tensor([[0, 1, 3, 2]], dtype=torch.int32)
    r = oracle.tree_score(draft, tokens, parents, torch.tensor([N], dtype=torch.int32), T)
    q = torch.softmax(draft.double() / T, -1).numpy()[0]
    trials = 200000
    hit = np.ones(trials, dtype=bool)
    for lvl in range(1, N):
        draw = rng.choice(V, size=trials, p=q[lvl - 1])
        hit &= draw == int(tokens[0, lvl])
    freq = hit.mean()
    prob = math.exp(r["path_lp"][0, N - 1])
    assert abs(freq - prob) < 5 * math.sqrt(prob * (1 - prob) / trials)


@pytest.mark.parametrize("k", [1, 4, 16])
def test_topk_matches_stable_sort(k):
    draft, tokens, parents, n = case(4, V=200, scale=1.0)
    # plant ties: copy some values within rows
    d = draft.clone()
    d[:, :, 10] = d[:, :, 3]
    d[:, :, 150] = d[:, :, 3]
    r = oracle.tree_score(d, tokens, parents, n, 1.3, top_k=k)
    vals, idx = torch.sort(d.float(), dim=-1, descending=True, stable=True)
    np.testing.assert_array_equal(r["topk_tok"], idx[:, :, :k].numpy())
    lsm = torch.log_softmax(d.double() / 1.3, dim=-1)
    np.testing.assert_allclose(r["topk_lp"], torch.gather(lsm, 2, idx[:, :, :k]).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("budget", [1, 7, 40])
def test_budget_expansion_matches_brute_force(budget):
    draft, tokens, parents, n = case(5, B=2, N=12, V=50, scale=3.0)
    k = 4
    r = oracle.tree_score(draft, tokens, parents, n, 1.0, top_k=k, budget=budget)
    lsm = torch.log_softmax(draft.double(), dim=-1)
    for b in range(draft.shape[0]):
        cands = []
        for u in range(draft.shape[1]):
            vals, idx = torch.sort(draft[b, u].float(), descending=True, stable=True)
            for j in range(k):
                v = int(idx[j])
                cands.append((-(r["path_lp"][b, u] + float(lsm[b, u, v])), u, j, v))
        cands.sort()
        want = cands[:budget]
        assert r["cand_parent"][b].tolist() == [c[1] for c in want]
        assert r["cand_token"][b].tolist() == [c[3] for c in want]
        np.testing.assert_allclose(r["cand_score"][b], [-c[0] for c in want], rtol=0, atol=1e-12)
        assert r["gaps"][b] > 0                  # the smallest nonzero gap


def test_malformed_and_out_of_range():
    draft, tokens, parents, n = case(6, B=3, N=6, V=16)
    parents = parents.clone()
    parents[1, 4] = 5
    tokens = tokens.clone()
    tokens[2, 3] = 99
    r = oracle.tree_score(draft, tokens, parents, n, 1.0, top_k=2, budget=3)
    assert np.isnan(r["node_lp"][1]).all() and np.isnan(r["path_lp"][1]).all()
    assert (r["topk_tok"][1] == -1).all() and (r["cand_parent"][1] == -1).all()
    assert r["node_lp"][2, 3] == -np.inf
    assert np.isfinite(r["node_lp"][0]).all() and r["node_lp"][0, 0] == 0.0
