"""Pins of the oracle's stochastic tree verification (CPU only).

The random numbers: the oracle's Philox4x64-10 is checked word for word
against numpy's Philox bit generator, an independent implementation of the
same published generator (Salmon et al., "Parallel random numbers: as easy
as 1, 2, 3", SC 2011), and the acceptance and sampling uniforms against
numpy's words at the documented counters.

The method: speculative sampling (the paper's section 2.1 cites Leviathan
et al. 2023 for the draft-then-verify rule) must leave the target's
distribution unchanged. When a node's children are drawn independently
from the draft distribution q, the token emitted after that node (the
accepted child's token, or the sample drawn when every child is rejected)
follows the target distribution p exactly, whatever q is. These tests draw
the children from q many times and compare the emitted tokens with p by a
chi-square test, at the root and one level down. A dropped residual, a
missing normalisation or a wrong sibling order each moves that
distribution. Two limits reduce to deterministic rules: draft equal to
target accepts every first child, and a near-zero temperature gives the
greedy walk's path and the greedy argmax as the next token.
"""

import numpy as np
import pytest
import torch

import oracle


def bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def softmax64(z_bf16, T):
    z = z_bf16.to(torch.float64).numpy() / T
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def chi2_stat(counts, probs):
    n = counts.sum()
    exp = n * probs
    keep = exp > 0
    assert counts[~keep].sum() == 0, "a token of zero probability was emitted"
    return float((((counts - exp) ** 2)[keep] / exp[keep]).sum()), int(keep.sum()) - 1


# Upper 0.1% points of chi-square for the degrees of freedom used here.
CHI2_999 = {3: 16.27, 4: 18.47, 5: 20.52, 6: 22.46, 7: 24.32}


# ----------------------------------------------------------------- Philox

@pytest.mark.parametrize("counter,key", [
    ([1, 0, 0, 0], [0, 0]),
    ([6, 0, 0, 0], [0x0123456789ABCDEF, 0xFEDCBA9876543210]),
    ([0, 1, 0, 0], [7, 11]),                       # the counter below it carries across words
    ([2 ** 63, 5, 2 ** 64 - 1, 3], [2 ** 64 - 1, 2 ** 64 - 1]),
    ([123456789, 987654321, 42, 0], [0x9E3779B97F4A7C15, 1]),
])
def test_philox_matches_numpy(counter, key):
    # numpy's generator increments its 256-bit counter before each block
    c = sum(int(w) << (64 * i) for i, w in enumerate(counter)) - 1
    prev = np.array([(c >> (64 * i)) & (2 ** 64 - 1) for i in range(4)], dtype=np.uint64)
    ref = np.random.Philox(counter=prev, key=np.array(key, dtype=np.uint64)).random_raw(8)
    got = oracle.philox4x64_10(counter, key)
    np.testing.assert_array_equal(got, ref[:4])
    nxt = list(counter)
    nxt[0] = (nxt[0] + 1) % 2 ** 64
    if nxt[0] == 0:
        nxt[1] += 1
    np.testing.assert_array_equal(oracle.philox4x64_10(nxt, key), ref[4:])


@pytest.mark.parametrize("purpose,b,index", [(0, 0, 0), (0, 3, 5), (1, 0, 151935), (1, 15, 7)])
def test_uniform_is_top_23_bits_of_the_documented_word(purpose, b, index):
    seed, offset = 0x5EED, 17
    ctr = np.array([index // 4, b, purpose, 0], dtype=np.uint64)
    c = sum(int(w) << (64 * i) for i, w in enumerate(ctr)) - 1
    prev = np.array([(c >> (64 * i)) & (2 ** 64 - 1) for i in range(4)], dtype=np.uint64)
    w = int(np.random.Philox(counter=prev, key=np.array([seed, offset], dtype=np.uint64)).random_raw(4)[index % 4])
    assert oracle.uniform(seed, offset, purpose, b, index) == ((w >> 41) + 0.5) / 2 ** 23


def test_uniforms_are_uniform():
    u = np.array([oracle.uniform(3, 0, 0, 0, i) for i in range(20000)])
    assert u.min() > 0 and u.max() < 1
    counts = np.histogram(u, bins=10, range=(0, 1))[0]
    stat = ((counts - 2000) ** 2 / 2000).sum()
    assert stat < 27.9                            # chi-square, 9 dof, 0.1%


# ------------------------------------------------------- the distribution

def star_batch(p_logits, q_logits, k, trials, rng, V, T):
    """`trials` sequences, each a root with k children whose tokens are
    drawn independently from q = softmax(q_logits / T). Every node row holds
    the same target and draft logits."""
    N = k + 1
    tgt = np.broadcast_to(p_logits, (trials, N, V)).copy()
    drf = np.broadcast_to(q_logits, (trials, N, V)).copy()
    q = softmax64(bf16(q_logits), T)
    tokens = np.zeros((trials, N), dtype=np.int32)
    tokens[:, 1:] = rng.choice(V, size=(trials, k), p=q)
    parents = np.zeros((trials, N), dtype=np.int32)
    parents[:, 0] = -1
    return bf16(tgt), bf16(drf), tokens, parents, np.full(trials, N, dtype=np.int32)


@pytest.mark.parametrize("k,T", [(1, 1.0), (3, 1.0), (4, 0.7)])
def test_first_emitted_token_follows_the_target(k, T):
    rng = np.random.default_rng(100 + k)
    V = 6
    p_logits = rng.normal(size=V) * 1.5
    q_logits = rng.normal(size=V) * 1.5
    trials = 20000
    tgt, drf, tokens, parents, n = star_batch(p_logits, q_logits, k, trials, rng, V, T)
    alen, path, nxt, _ = oracle.tree_verify_sample(tgt, drf, tokens, parents, n, 4, T, seed=77, offset=k)
    first = np.where(alen >= 2, tokens[np.arange(trials), np.maximum(path[:, 1], 0)], nxt)
    p = softmax64(bf16(p_logits), T)
    stat, dof = chi2_stat(np.bincount(first, minlength=V).astype(float), p)
    assert stat < CHI2_999[dof], (stat, dof)
    # the draft is not the target here, so both outcomes occur
    assert 0 < (alen >= 2).mean() < 1


def test_second_emitted_token_follows_the_accepted_childs_target():
    """Depth two: a root with 2 children drawn from q_root, each child with
    2 children drawn from q_child. The target row of a child depends on its
    token only, so after accepting a child with token x the next emitted
    token must follow p_x."""
    rng = np.random.default_rng(7)
    V, trials = 5, 30000
    pl = rng.normal(size=(V + 1, V)) * 1.2          # row V: the root's target; row x: a child with token x
    ql = rng.normal(size=(V + 1, V)) * 1.2
    N = 7                                           # root; children 1, 2; grandchildren 3, 4 (of 1), 5, 6 (of 2)
    parents = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2], dtype=np.int32), (trials, 1))
    qs = softmax64(bf16(ql), 1.0)
    tokens = np.zeros((trials, N), dtype=np.int32)
    tokens[:, 1:3] = rng.choice(V, size=(trials, 2), p=qs[V])
    tgt = np.zeros((trials, N, V), dtype=np.float32)
    drf = np.zeros((trials, N, V), dtype=np.float32)
    tgt[:, 0] = pl[V]
    drf[:, 0] = ql[V]
    for c, kids in ((1, (3, 4)), (2, (5, 6))):
        x = tokens[:, c]
        tgt[:, c] = pl[x]
        drf[:, c] = ql[x]
        for g in kids:
            u = rng.random(trials)
            tokens[:, g] = (u[:, None] > np.cumsum(qs[x], axis=1)).sum(axis=1)
            tgt[:, g] = 0.0
            drf[:, g] = 0.0
    alen, path, nxt, _ = oracle.tree_verify_sample(bf16(tgt), bf16(drf), tokens, parents,
                                                   np.full(trials, N, dtype=np.int32), 4, 1.0, seed=5, offset=0)
    ps = softmax64(bf16(pl), 1.0)
    went = alen >= 2
    x1 = tokens[np.arange(trials), np.maximum(path[:, 1], 0)]
    second = np.where(alen >= 3, tokens[np.arange(trials), np.maximum(path[:, 2], 0)], nxt)
    for x in range(V):
        sel = went & (x1 == x)
        if sel.sum() < 500:
            continue
        stat, dof = chi2_stat(np.bincount(second[sel], minlength=V).astype(float), ps[x])
        assert stat < CHI2_999[dof], (x, stat, dof)


def test_leaf_root_samples_the_target():
    rng = np.random.default_rng(3)
    V, trials = 7, 20000
    pl = rng.normal(size=V) * 2.0
    tgt = bf16(np.broadcast_to(pl, (trials, 1, V)).copy())
    drf = bf16(np.zeros((trials, 1, V)))
    alen, path, nxt, _ = oracle.tree_verify_sample(tgt, drf, np.zeros((trials, 1), np.int32),
                                                   np.full((trials, 1), -1, np.int32), np.ones(trials, np.int32),
                                                   4, 1.3, seed=9, offset=2)
    assert (alen == 1).all() and (path[:, 0] == 0).all() and (path[:, 1:] == -1).all()
    stat, dof = chi2_stat(np.bincount(nxt, minlength=V).astype(float), softmax64(bf16(pl), 1.3))
    assert stat < CHI2_999[dof]


# --------------------------------------------------- deterministic limits

def random_tree(rng, n, max_children=3):
    parents = [-1]
    kids = {0: 0}
    for i in range(1, n):
        while True:
            p = int(rng.integers(0, i))
            if kids[p] < max_children:
                break
        parents.append(p)
        kids[p] += 1
        kids[i] = 0
    return parents


def test_equal_draft_and_target_accept_every_first_child():
    rng = np.random.default_rng(11)
    B, N, V = 8, 24, 50
    parents = np.array([random_tree(rng, N) for _ in range(B)], dtype=np.int32)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    lg = bf16(rng.normal(size=(B, N, V)))
    for max_depth in (16, 2):
        alen, path, nxt, _ = oracle.tree_verify_sample(lg, lg, tokens, parents, np.full(B, N, np.int32),
                                                       max_depth, 0.9, seed=1, offset=0)
        for b in range(B):
            want = [0]
            while len(want) <= max_depth:
                kids = [c for c in range(N) if parents[b, c] == want[-1]]
                if not kids:
                    break
                want.append(kids[0])
            assert alen[b] == len(want)
            assert path[b, :len(want)].tolist() == want
            assert (path[b, len(want):] == -1).all()
            assert 0 <= nxt[b] < V


def test_near_zero_temperature_is_the_greedy_walk():
    rng = np.random.default_rng(21)
    B, N, V = 12, 20, 64
    parents = np.array([random_tree(rng, N) for _ in range(B)], dtype=np.int32)
    # well-separated integer logits: the argmax beats the rest by >= 1
    lg = rng.permutation(np.tile(np.arange(V, dtype=np.float32), (B * N, 1)).T).T.reshape(B, N, V)
    for b in range(B):
        for i in range(N):
            lg[b, i] = rng.permutation(V).astype(np.float32)
    am = lg.argmax(-1)
    tokens = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        for c in range(1, N):
            # siblings get distinct tokens; about half of them match the parent's argmax
            sib = [s for s in range(1, c) if parents[b, s] == parents[b, c]]
            used = {int(tokens[b, s]) for s in sib}
            want = int(am[b, parents[b, c]])
            if want not in used and rng.random() < 0.6:
                tokens[b, c] = want
            else:
                tokens[b, c] = next(t for t in rng.permutation(V) if t not in used and t != want)
    # a flat draft: q is uniform at every temperature, so the ratio p(x) / q(x)
    # is V p(x): above 1 for the argmax, below 2^-24 for any other token
    draft = bf16(np.zeros((B, N, V)))
    alen, path, nxt, _ = oracle.tree_verify_sample(bf16(lg), draft, tokens, parents, np.full(B, N, np.int32),
                                                   16, 0.01, seed=4, offset=1)
    g_alen, g_path, g_am = oracle.tree_verify(bf16(lg), tokens, parents, np.full(B, N, np.int32), 16)
    np.testing.assert_array_equal(alen, g_alen)
    np.testing.assert_array_equal(path, g_path)
    last = path[np.arange(B), alen - 1]
    np.testing.assert_array_equal(nxt, g_am[np.arange(B), last])


def test_malformed_trees():
    V = 8
    lg = bf16(np.zeros((3, 4, V)))
    parents = np.array([[-1, 0, 0, 1], [0, 0, 0, 1], [-1, 0, 2, 1]], dtype=np.int32)
    tokens = np.zeros((3, 4), dtype=np.int32)
    alen, path, nxt, _ = oracle.tree_verify_sample(lg, lg, tokens, parents, np.array([4, 4, 4], np.int32),
                                                   3, 1.0, seed=0, offset=0)
    assert alen.tolist()[1:] == [0, 0] and nxt.tolist()[1:] == [-1, -1]
    assert (path[1:] == -1).all()
    assert alen[0] >= 1 and nxt[0] >= 0
