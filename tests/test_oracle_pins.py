"""Pins of the fp64 oracle against sources other than itself (CPU only).

Attention is checked against torch's fp64 scaled_dot_product_attention. The
boolean mask is built here by transitive closure of the parent relation,
not by the oracle's chain walk. A chain tree must equal textbook causal
attention. N=1 must equal single-token decode. With q = 0 the softmax
weights are uniform, so every output is the plain mean of the visible
value rows. Deleting or relabelling non-ancestors must leave a node's
output bit-identical. Argmax is checked against torch.argmax. The tree
walk is checked against brute-force enumeration of every root path, and
against the hand-worked cases in golden/walk_cases.txt.

Rule sources: "JetFlow: Scaling Speculative Decoding with Parallel Tree
Drafting" (blog), section "What JetFlow Does Differently", for the mask;
the paper's section 2.1 "Background", for greedy acceptance.
"""

import itertools
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tree_masked_attention_causal_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "walk_cases.txt")


# ----------------------------------------------------------------- helpers

def ancestor_matrix(parents, n):
    """Boolean [n, n]: A[i, j] iff j is i or an ancestor of i. Built as the
    reflexive-transitive closure of the child->parent relation by repeated
    squaring of a boolean matrix, independent of any chain walk."""
    A = torch.eye(n, dtype=torch.bool)
    for i in range(1, n):
        A[i, parents[i]] = True
    for _ in range(max(1, math.ceil(math.log2(max(n, 2))))):
        A = (A.to(torch.float64) @ A.to(torch.float64)) > 0
    return A


def random_case(seed, B=2, N=12, Hq=4, Hkv=2, d=16, Pcap=24, prefix=None, parents=None):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    if parents is None:
        parents = torch.tensor([synth.random_tree(g, N, 6, None) for _ in range(B)], dtype=torch.int32)
    if prefix is None:
        prefix = torch.randint(0, Pcap + 1, (B,), generator=g, dtype=torch.int32)
    return dict(q=bf(B, N, Hq, d), k_cache=bf(B, Hkv, Pcap, d), v_cache=bf(B, Hkv, Pcap, d),
                tree_k=bf(B, N, Hkv, d), tree_v=bf(B, N, Hkv, d), prefix_lens=prefix,
                parents=parents, n_nodes=torch.full((B,), N, dtype=torch.int32))


def sdpa_reference(c, scale=None):
    """fp64 SDPA over keys = prefix ++ all tree nodes with an explicit mask."""
    q, kc, vc, tk, tv = (c[k].to(torch.float64) for k in ("q", "k_cache", "v_cache", "tree_k", "tree_v"))
    B, N, Hq, d = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = torch.empty(B, N, Hq, d, dtype=torch.float64)
    for b in range(B):
        P = int(c["prefix_lens"][b])
        K = torch.cat([kc[b, :, :P], tk[b].transpose(0, 1)], dim=1)      # [Hkv, P+N, d]
        V = torch.cat([vc[b, :, :P], tv[b].transpose(0, 1)], dim=1)
        K = K.repeat_interleave(G, dim=0)                                 # query head h -> kv h // G
        V = V.repeat_interleave(G, dim=0)
        anc = ancestor_matrix(c["parents"][b].tolist(), N)
        mask = torch.cat([torch.ones(N, P, dtype=torch.bool), anc], dim=1)
        o = F.scaled_dot_product_attention(q[b].transpose(0, 1), K, V, attn_mask=mask, scale=scale)
        out[b] = o.transpose(0, 1)
    return out


def run_oracle(c, **kw):
    return oracle.tree_attention(c["q"], c["k_cache"], c["v_cache"], c["prefix_lens"], c["tree_k"],
                                 c["tree_v"], c["parents"], c["n_nodes"], **kw)


# --------------------------------------------------------------- attention

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attention_equals_sdpa_with_ancestor_mask(seed):
    c = random_case(seed)
    np.testing.assert_allclose(run_oracle(c), sdpa_reference(c).numpy(), rtol=0, atol=1e-12)


def test_attention_custom_scale():
    c = random_case(7)
    np.testing.assert_allclose(run_oracle(c, scale=0.37), sdpa_reference(c, scale=0.37).numpy(),
                               rtol=0, atol=1e-12)


def test_chain_tree_is_causal_attention():
    """parents[i] = i - 1: the tree is a plain continuation of the prefix, so
    node outputs are the last N rows of causal attention over P + N tokens."""
    B, N, Hq, Hkv, d, P = 1, 9, 4, 1, 32, 13
    chain = torch.tensor([[-1] + list(range(N - 1))], dtype=torch.int32)
    c = random_case(11, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, Pcap=P,
                    prefix=torch.tensor([P], dtype=torch.int32), parents=chain)
    got = run_oracle(c)[0]                                                # [N, Hq, d]
    f = lambda t: t.to(torch.float64)
    K = torch.cat([f(c["k_cache"][0, 0]), f(c["tree_k"][0, :, 0])], 0)    # [P+N, d]
    V = torch.cat([f(c["v_cache"][0, 0]), f(c["tree_v"][0, :, 0])], 0)
    for h in range(Hq):
        Q = torch.cat([torch.zeros(P, d, dtype=torch.float64), f(c["q"][0, :, h])], 0)
        ref = F.scaled_dot_product_attention(Q[None], K[None], V[None], is_causal=True)[0, P:]
        np.testing.assert_allclose(got[:, h], ref.numpy(), rtol=0, atol=1e-12)


def test_single_node_is_decode_attention():
    c = random_case(5, B=3, N=1, Pcap=40, parents=torch.full((3, 1), -1, dtype=torch.int32))
    got = run_oracle(c)
    f = lambda t: t.to(torch.float64)
    for b in range(3):
        P = int(c["prefix_lens"][b])
        for h in range(4):
            kh = h // 2
            K = torch.cat([f(c["k_cache"][b, kh, :P]), f(c["tree_k"][b, 0, kh])[None]], 0)
            V = torch.cat([f(c["v_cache"][b, kh, :P]), f(c["tree_v"][b, 0, kh])[None]], 0)
            ref = F.scaled_dot_product_attention(f(c["q"][b, 0, h])[None, None], K[None], V[None])
            np.testing.assert_allclose(got[b, 0, h], ref[0, 0].numpy(), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    """q = 0 makes every score 0, so each output is the unweighted mean of
    the value rows the node may see: the prefix, its ancestors and itself."""
    N = 10
    star_and_chain = torch.tensor([[-1, 0, 0, 1, 3, 3, 2, 0, 7, 8]], dtype=torch.int32)
    c = random_case(3, B=1, N=N, Hq=4, Hkv=2, d=8, Pcap=6,
                    prefix=torch.tensor([5], dtype=torch.int32), parents=star_and_chain)
    c["q"] = torch.zeros_like(c["q"])
    got = run_oracle(c)
    visible = {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3], 4: [0, 1, 3, 4], 5: [0, 1, 3, 5],
               6: [0, 2, 6], 7: [0, 7], 8: [0, 7, 8], 9: [0, 7, 8, 9]}   # worked by hand
    for i, nodes in visible.items():
        for h in range(4):
            kh = h // 2
            rows = [c["v_cache"][0, kh, j] for j in range(5)] + [c["tree_v"][0, j, kh] for j in nodes]
            mean = torch.stack(rows).to(torch.float64).mean(0)
            np.testing.assert_allclose(got[0, i, h], mean.numpy(), rtol=0, atol=1e-14)


def test_star_tree_sees_prefix_root_and_self():
    N = 7
    star = torch.tensor([[-1] + [0] * (N - 1)], dtype=torch.int32)
    c = random_case(9, B=1, N=N, parents=star, prefix=torch.tensor([17], dtype=torch.int32))
    got = run_oracle(c)
    f = lambda t: t.to(torch.float64)
    for i in range(N):
        for h in range(4):
            kh = h // 2
            keys = [0] if i == 0 else [0, i]
            K = torch.cat([f(c["k_cache"][0, kh, :17])] + [f(c["tree_k"][0, j, kh])[None] for j in keys])
            V = torch.cat([f(c["v_cache"][0, kh, :17])] + [f(c["tree_v"][0, j, kh])[None] for j in keys])
            ref = F.scaled_dot_product_attention(f(c["q"][0, i, h])[None, None], K[None], V[None])
            np.testing.assert_allclose(got[0, i, h], ref[0, 0].numpy(), rtol=0, atol=1e-12)


def test_deleting_non_ancestors_is_bit_identical():
    c = random_case(21, B=1, N=14)
    full = run_oracle(c)
    par = c["parents"][0].tolist()
    for i in [5, 9, 13]:
        chain = synth.chain_to_root(par, i)
        sub = dict(c)
        idx = torch.tensor(chain)
        sub["parents"] = torch.tensor([[-1] + list(range(len(chain) - 1))], dtype=torch.int32)
        sub["n_nodes"] = torch.tensor([len(chain)], dtype=torch.int32)
        for k in ("q", "tree_k", "tree_v"):
            sub[k] = c[k][:, idx].contiguous()
        got = run_oracle(sub)
        assert np.array_equal(got[0, -1], full[0, i])


def test_relabelling_non_ancestors_is_bit_identical():
    """Give every non-ancestor of node i new parents and new q/k/v values:
    node i's output must not change at all."""
    c = random_case(33, B=1, N=16)
    i = 12
    full = run_oracle(c)
    par = c["parents"][0].tolist()
    anc = set(synth.chain_to_root(par, i))
    g = torch.Generator().manual_seed(99)
    new_par = list(par)
    for j in range(1, 16):
        if j not in anc:
            new_par[j] = int(torch.randint(0, j, (1,), generator=g))
    alt = dict(c)
    alt["parents"] = torch.tensor([new_par], dtype=torch.int32)
    # keep i's chain intact in the relabelled tree
    assert synth.chain_to_root(new_par, i) == synth.chain_to_root(par, i)
    for k in ("tree_k", "tree_v", "q"):
        t = c[k].clone()
        for j in range(16):
            if j not in anc:
                t[0, j] = torch.randn(t.shape[2:], generator=g).to(torch.bfloat16)
        alt[k] = t
    got = run_oracle(alt)
    assert np.array_equal(got[0, i], full[0, i])


def test_malformed_tree_gives_nan_rows():
    c = random_case(4, B=2, N=6)
    c["parents"][1, 3] = 3                          # not topological
    got = run_oracle(c)
    assert np.isnan(got[1]).all()
    assert not np.isnan(got[0]).any()


def test_row_selection_matches_full():
    c = random_case(8, B=2, N=10)
    full = run_oracle(c)
    sel = [(0, 3), (1, 9), (1, 0)]
    part = run_oracle(c, sel=sel)
    for b, i in sel:
        assert np.array_equal(part[b, i], full[b, i])
    assert np.isnan(part[0, 0]).all()


# ------------------------------------------------------------------ argmax

def test_argmax_matches_torch_first_occurrence():
    g = torch.Generator().manual_seed(1)
    x = torch.randint(-3, 4, (64, 333), generator=g).to(torch.bfloat16)   # many ties
    x[5] = 0.0
    x[6, ::2] = -0.0
    x[7, 100] = float("nan")
    x[7, 200] = float("nan")
    x[8, 50] = float("inf")
    x[8, 60] = float("inf")
    x[9, -1] = float("nan")
    x[10] = float("-inf")
    np.testing.assert_array_equal(oracle.argmax_rows(x), torch.argmax(x, dim=-1).numpy())


def test_argmax_random_rows_match_torch():
    x = torch.randn(16, 151936, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.argmax_rows(x), torch.argmax(x, dim=-1).numpy())


# -------------------------------------------------------------- tree walk

def brute_force_accept(parents, tokens, am, n, max_depth):
    """Enumerate every root-to-node path, keep those whose every edge
    agrees, take the longest (lowest end index on ties)."""
    best_len, best_end = 0, None
    for end in range(n):
        path = synth.chain_to_root(parents, end)
        if all(tokens[path[k]] == am[path[k - 1]] for k in range(1, len(path))):
            if len(path) > best_len:
                best_len, best_end = len(path), end
    path = synth.chain_to_root(parents, best_end)[: max_depth + 1]
    return len(path), path + [-1] * (max_depth + 1 - len(path))


def onehot_logits(am_rows, V, Nmax, seed=0):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn(1, Nmax, V, generator=g).clamp(-1, 1).to(torch.bfloat16)
    for u, a in enumerate(am_rows):
        lg[0, u, a] = 4.0
    return lg


def all_parent_arrays(n):
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield [-1] + list(choice)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_walk_equals_brute_force_on_every_small_tree(n):
    g = torch.Generator().manual_seed(n)
    V = 3
    for parents in all_parent_arrays(n):
        for trial in range(3):
            lg = torch.randint(0, 3, (1, n, V), generator=g).to(torch.bfloat16)   # ties on purpose
            tokens = torch.randint(0, V, (1, n), generator=g, dtype=torch.int32)
            am = torch.argmax(lg[0], dim=-1).tolist()
            for max_depth in (n - 1, 1):
                alen, path, am_o = oracle.tree_verify(lg, tokens, torch.tensor([parents], dtype=torch.int32),
                                                      torch.tensor([n], dtype=torch.int32), max_depth)
                assert am_o[0].tolist() == am
                L, p = brute_force_accept(parents, tokens[0].tolist(), am, n, max_depth)
                assert alen[0] == L and path[0].tolist() == p, (parents, tokens, am)


def test_walk_equals_brute_force_random_trees():
    g = torch.Generator().manual_seed(77)
    for trial in range(200):
        n = int(torch.randint(1, 13, (1,), generator=g))
        parents = synth.random_tree(g, n, 12, None)
        V = 2
        lg = torch.randint(0, 4, (1, n, V), generator=g).to(torch.bfloat16)
        tokens = torch.randint(0, V, (1, n), generator=g, dtype=torch.int32)
        am = torch.argmax(lg[0], dim=-1).tolist()
        alen, path, _ = oracle.tree_verify(lg, tokens, torch.tensor([parents], dtype=torch.int32),
                                           torch.tensor([n], dtype=torch.int32), 11)
        L, p = brute_force_accept(parents, tokens[0].tolist(), am, n, 11)
        assert alen[0] == L and path[0].tolist() == p


def load_golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0]}
            cases.append(cur)
        else:
            cur[key] = [int(v) for v in vals]
    return cases


@pytest.mark.parametrize("case", load_golden_cases(), ids=lambda c: c["name"])
def test_walk_golden_cases(case):
    Nmax = len(case["parents"])
    n = case["n"][0]
    md = case["max_depth"][0]
    lg = onehot_logits(case["argmax"], 10, Nmax)
    alen, path, am = oracle.tree_verify(lg, torch.tensor([case["tokens"]], dtype=torch.int32),
                                        torch.tensor([case["parents"]], dtype=torch.int32),
                                        torch.tensor([n], dtype=torch.int32), md)
    assert alen[0] == case["accept_len"][0]
    assert path[0].tolist() == case["path"]
    valid = 1 <= n <= Nmax
    assert am[0].tolist() == [case["argmax"][i] if valid and i < n else -1 for i in range(Nmax)]


def test_planted_path_is_recovered_tiny():
    inp = synth.make_inputs(synth.WORKLOADS["tiny"])
    alen, path, am = oracle.tree_verify(inp["logits"], inp["tokens"], inp["parents"], inp["n_nodes"], 16)
    assert alen[0] == int(inp["planted_len"][0]) == 3
    assert path[0, :3].tolist() == inp["planted_path"][0]
    np.testing.assert_array_equal(am, inp["top_tokens"].numpy())


@pytest.mark.parametrize("seed", range(5))
def test_planted_lengths_recovered_small_batch(seed):
    w = synth.Workload("small_batch", 6, 4, 2, 16, 24, 4, 12, 12, 97, 6, 3, 1, 6, 500 + seed)
    inp = synth.make_inputs(w)
    alen, path, _ = oracle.tree_verify(inp["logits"], inp["tokens"], inp["parents"], inp["n_nodes"], 8)
    np.testing.assert_array_equal(alen, inp["planted_len"].numpy())
    for b in range(6):
        L = int(inp["planted_len"][b])
        assert path[b, :L].tolist() == inp["planted_path"][b]


def test_tree_validity_rule():
    assert oracle.tree_is_valid([-1, 0, 1, 0], 4, 4)
    assert not oracle.tree_is_valid([-1, 0, 2, 0], 4, 4)
    assert not oracle.tree_is_valid([0, 0], 2, 2)
    assert not oracle.tree_is_valid([-1, -1], 2, 2)
    assert not oracle.tree_is_valid([-1], 0, 1)
    assert not oracle.tree_is_valid([-1, 0], 3, 2)
    assert oracle.tree_is_valid([-1, 0, 77], 2, 3)          # padding is not checked


# ----------------------------------------------------------- KV commit


def _commit_cases():
    path = os.path.join(os.path.dirname(__file__), "golden", "commit_cases.txt")
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "rows": []}
            cases.append(cur)
        elif key == "row":
            cur["rows"].append((int(vals[0]), int(vals[3])))
        elif key == "path":
            cur["path"] = [int(v) for v in vals]
        else:
            cur[key] = int(vals[0])
    return cases


@pytest.mark.parametrize("case", _commit_cases(), ids=lambda c: c["name"])
def test_commit_kv_golden_cases(case):
    """Hand-worked commits (tests/golden/commit_cases.txt): which cache rows
    change, from which node, the new prefix length and the flag."""
    Hkv, d, Pcap, Nmax = case["Hkv"], 2, 6, 4
    val = np.zeros((1, Nmax, Hkv, d), dtype=np.float32)
    for i in range(Nmax):
        for h in range(Hkv):
            for e in range(d):
                val[0, i, h, e] = i + h / 4 + e / 8
    tk = torch.from_numpy(val).to(torch.bfloat16)
    tv = torch.from_numpy(-val).to(torch.bfloat16)
    kc = torch.full((1, Hkv, Pcap, d), 0.5, dtype=torch.bfloat16)
    vc = torch.full((1, Hkv, Pcap, d), 0.5, dtype=torch.bfloat16)
    k2, v2, pl, flags = oracle.commit_kv(tk, tv, torch.tensor([case["n"]], dtype=torch.int32),
                                         torch.tensor([case["a"]], dtype=torch.int32),
                                         torch.tensor([case["path"]], dtype=torch.int32), kc, vc,
                                         torch.tensor([case["P"]], dtype=torch.int32), case["max_depth"])
    assert int(flags[0]) == case["flag"]
    assert int(pl[0]) == case["new_P"]
    half = np.uint16(0x3F00)                      # bf16 0.5
    want_k = np.full((1, Hkv, Pcap, d), half, dtype=np.uint16)
    want_v = want_k.copy()
    tkb = tk.view(torch.int16).numpy().view(np.uint16)
    tvb = tv.view(torch.int16).numpy().view(np.uint16)
    for r, i in case["rows"]:
        want_k[0, :, r] = tkb[0, i]
        want_v[0, :, r] = tvb[0, i]
    np.testing.assert_array_equal(k2, want_k)
    np.testing.assert_array_equal(v2, want_v)


def test_commit_then_attention_equals_chain_attention():
    """Composition with the attention's definition: commit a whole chain
    (path 0..N-1) and node i's tree attention over the original prefix
    equals attention over the committed cache cut at P + i (rows of nodes
    0..i-1) with a one-node tree holding node i. A wrong row order, offset
    or head in the commit changes the key sequence and fails this."""
    g = torch.Generator().manual_seed(77)
    B, N, Hq, Hkv, d, P, Pcap = 2, 6, 4, 2, 64, 5, 16
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    q, tk, tv = bf(B, N, Hq, d), bf(B, N, Hkv, d), bf(B, N, Hkv, d)
    kc, vc = bf(B, Hkv, Pcap, d), bf(B, Hkv, Pcap, d)
    chain = torch.tensor([[-1] + list(range(N - 1))] * B, dtype=torch.int32)
    pl = torch.full((B,), P, dtype=torch.int32)
    nn = torch.full((B,), N, dtype=torch.int32)
    ref = oracle.tree_attention(q, kc, vc, pl, tk, tv, chain, nn)
    k2, v2, pl2, flags = oracle.commit_kv(tk, tv, nn, nn, torch.arange(N, dtype=torch.int32).repeat(B, 1), kc, vc,
                                          pl, N - 1)
    assert (flags == 0).all() and (pl2 == P + N).all()
    k2 = torch.from_numpy(k2.view(np.int16)).view(torch.bfloat16)
    v2 = torch.from_numpy(v2.view(np.int16)).view(torch.bfloat16)
    one = torch.full((B, 1), -1, dtype=torch.int32)
    for i in range(N):
        got = oracle.tree_attention(q[:, i:i + 1], k2, v2, torch.full((B,), P + i, dtype=torch.int32),
                                    tk[:, i:i + 1], tv[:, i:i + 1], one, torch.ones(B, dtype=torch.int32))
        np.testing.assert_allclose(got[:, 0], ref[:, i], rtol=0, atol=1e-12)


def test_gather_pages_picks_the_documented_element():
    """Row p of sequence b, head h is pages[table[b, p // ps], p % ps, h]:
    checked on a pool whose every element encodes its own coordinates."""
    num_pages, ps, Hkv, d = 6, 4, 2, 3
    pages = np.zeros((num_pages, ps, Hkv, d), dtype=np.uint16)
    for ph in range(num_pages):
        for r in range(ps):
            for h in range(Hkv):
                for c in range(d):
                    pages[ph, r, h, c] = ph * 1000 + r * 100 + h * 10 + c
    table = np.array([[4, 1, 5], [0, 3, -1]], dtype=np.int32)
    lens = np.array([11, 6], dtype=np.int32)
    out = oracle.gather_pages(pages, table, lens, ps, 12)
    for b in range(2):
        for p in range(12):
            for h in range(Hkv):
                want = [table[b, p // ps] * 1000 + (p % ps) * 100 + h * 10 + c for c in range(d)] if p < lens[b] \
                    else [0] * d
                assert out[b, h, p].tolist() == want


def test_paged_layout_round_trip_and_attention():
    c = random_case(11, B=3, N=9, Pcap=48, prefix=torch.tensor([48, 5, 0], dtype=torch.int32))
    pg = synth.paged_layout(c["k_cache"], c["v_cache"], c["prefix_lens"], 8, seed=2)
    kc = oracle.gather_pages(pg["k_pages"], pg["block_table"], c["prefix_lens"], 8, 48)
    ref_k = c["k_cache"].view(torch.int16).numpy().view(np.uint16)
    for b in range(3):
        P = int(c["prefix_lens"][b])
        np.testing.assert_array_equal(kc[b, :, :P], ref_k[b, :, :P])
    a = oracle.tree_attention_paged(c["q"], pg["k_pages"], pg["v_pages"], pg["block_table"], 8, 48,
                                    c["prefix_lens"], c["tree_k"], c["tree_v"], c["parents"], c["n_nodes"])
    b_ = run_oracle(c)
    np.testing.assert_array_equal(a, b_)


def test_paged_commit_equals_contiguous_commit():
    """Committing into pages and gathering them back gives the cache the
    contiguous commit gives, for the golden requests' flags as well."""
    c = random_case(12, B=4, N=9, Pcap=48, prefix=torch.tensor([40, 5, 47, 0], dtype=torch.int32))
    pg = synth.paged_layout(c["k_cache"], c["v_cache"], c["prefix_lens"], 8, seed=4, spare=2, spare_fill=0.0)
    # give every sequence all its pages (the commit may grow into unused ones)
    table = pg["block_table"].clone()
    nxt = pg["num_pages"]
    for b in range(4):
        for j in range(6):
            if table[b, j] < 0:
                table[b, j] = nxt
                nxt += 1
    kp = torch.cat([pg["k_pages"], torch.zeros(nxt - pg["num_pages"], *pg["k_pages"].shape[1:], dtype=torch.bfloat16)])
    vp = torch.cat([pg["v_pages"], torch.zeros_like(kp[pg["num_pages"]:])])
    alen = torch.tensor([3, 2, 2, 1], dtype=torch.int32)
    path = torch.tensor([[0, 1, 4, -1], [0, 2, -1, -1], [0, 3, -1, -1], [0, -1, -1, -1]], dtype=torch.int32)
    path = torch.cat([path, torch.full((4, 13), -1, dtype=torch.int32)], 1)
    kc, vc, pl, fl = oracle.commit_kv(c["tree_k"], c["tree_v"], c["n_nodes"], alen, path, c["k_cache"],
                                      c["v_cache"], c["prefix_lens"], 16)
    kp2, vp2, pl2, fl2 = oracle.commit_kv_paged(c["tree_k"], c["tree_v"], c["n_nodes"], alen, path, kp, vp, table, 8,
                                                c["prefix_lens"], 16)
    np.testing.assert_array_equal(pl2, pl)
    np.testing.assert_array_equal(fl2, fl)
    assert fl.tolist() == [0, 0, 2, 0]                   # 47 + 2 > 48: no room
    kg = oracle.gather_pages(kp2, table, pl2, 8, 48)
    vg = oracle.gather_pages(vp2, table, pl2, 8, 48)
    for b in range(4):
        P = int(pl2[b])
        np.testing.assert_array_equal(kg[b, :, :P], kc[b, :, :P])
        np.testing.assert_array_equal(vg[b, :, :P], vc[b, :, :P])
    # a used page outside the pool makes the request malformed
    bad = table.clone()
    bad[0, 5] = nxt + 3
    _, _, pl3, fl3 = oracle.commit_kv_paged(c["tree_k"], c["tree_v"], c["n_nodes"], alen, path, kp, vp, bad, 8,
                                            c["prefix_lens"], 16)
    assert fl3[0] == 1 and pl3[0] == 40
