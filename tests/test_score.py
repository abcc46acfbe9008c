"""GPU parity of draft-side path scoring (jf_tree_score) against the oracle.

Top-k tokens are compared bit for bit: they are chosen by comparing bf16
logits, exactly, on both sides. Log-probabilities are fp32 on the GPU:
(z - max) is exact, the row's log-sum comes from chunked fp32 sums
(relative error ~1e-6 of a sum of up to 151936 terms, a few 1e-5 at worst
in the log), so a node's value is held to 5e-5 + 1e-5 |ref| and a path's
to 5e-5 per path node + 1e-5 |ref|. The budgeted expansion orders
candidates by fp32 scores: its parents and tokens are compared in order
when the oracle's smallest nonzero score gap is above 1e-3 (else the
GPU's selection is checked to be valid: non-increasing scores, each equal
to its node's path score plus its token's log-probability).
"""

import numpy as np
import pytest
import torch

import oracle
from tree_masked_attention_causal_gb300 import binding as jb, synth
from helpers import lib, new_workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib()


def run(draft, tokens, parents, n_nodes, T, k, budget):
    B, N, V = draft.shape
    shape = jb.make_shape(B, 1, 1, 64, N, 1, V)
    dev = lambda t: torch.as_tensor(t).contiguous().cuda()
    o = dict(node=torch.full((B, N), 7.0, device="cuda"), path=torch.full((B, N), 7.0, device="cuda"),
             ttok=torch.full((B, N, max(k, 1)), -7, dtype=torch.int32, device="cuda"),
             tlp=torch.full((B, N, max(k, 1)), 7.0, device="cuda"),
             cpar=torch.full((B, max(budget, 1)), -7, dtype=torch.int32, device="cuda"),
             ctok=torch.full((B, max(budget, 1)), -7, dtype=torch.int32, device="cuda"),
             cscore=torch.full((B, max(budget, 1)), 7.0, device="cuda"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    jb.jf_tree_score(dev(draft), dev(tokens), dev(parents), dev(n_nodes), T, k, budget, o["node"], o["path"],
                     o["ttok"] if k else None, o["tlp"] if k else None, o["cpar"] if budget else None,
                     o["ctok"] if budget else None, o["cscore"] if budget else None, shape, new_workspace(shape),
                     status=st)
    torch.cuda.synchronize()
    out = {key: v.cpu().numpy() for key, v in o.items()}
    out["ttok"], out["tlp"] = out["ttok"][:, :, :k], out["tlp"][:, :, :k]
    for key in ("cpar", "ctok", "cscore"):
        out[key] = out[key][:, :budget]
    return out, int(st.item())


def depths_of(parents, n):
    d = np.zeros(len(parents), dtype=np.int64)
    for i in range(1, n):
        d[i] = d[parents[i]] + 1
    return d


def compare(draft, tokens, parents, n_nodes, T, k, budget):
    g, st = run(draft, tokens, parents, n_nodes, T, k, budget)
    r = oracle.tree_score(draft, tokens, parents, n_nodes, T, top_k=k, budget=budget)
    par = np.asarray(parents)
    B = par.shape[0]
    for b in range(B):
        n = int(n_nodes[b])
        ok = r["path_lp"][b, 0] == r["path_lp"][b, 0]
        if not ok:
            assert np.isnan(g["node"][b]).all() and np.isnan(g["path"][b]).all()
            continue
        depth = depths_of(par[b], n)
        ref_n, got_n = r["node_lp"][b, :n], g["node"][b, :n]
        fin = np.isfinite(ref_n)
        assert (np.isneginf(got_n) == np.isneginf(ref_n)).all()
        assert (np.abs(got_n[fin] - ref_n[fin]) <= 5e-5 + 1e-5 * np.abs(ref_n[fin])).all(), b
        ref_p, got_p = r["path_lp"][b, :n], g["path"][b, :n]
        fin = np.isfinite(ref_p)
        assert (np.isneginf(got_p) == np.isneginf(ref_p)).all()
        tol = 5e-5 * (depth[:n][fin] + 1) + 1e-5 * np.abs(ref_p[fin])
        assert (np.abs(got_p[fin] - ref_p[fin]) <= tol).all(), b
        assert np.isnan(g["node"][b, n:]).all() and np.isnan(g["path"][b, n:]).all()
        if k:
            np.testing.assert_array_equal(g["ttok"][b], r["topk_tok"][b])
            rl, gl = r["topk_lp"][b, :n], g["tlp"][b, :n]
            assert (np.abs(gl - rl) <= 5e-5 + 1e-5 * np.abs(rl)).all()
        if budget:
            if r["gaps"][b] > 1e-3:
                np.testing.assert_array_equal(g["cpar"][b], r["cand_parent"][b])
                np.testing.assert_array_equal(g["ctok"][b], r["cand_token"][b])
            sel = g["cpar"][b] >= 0
            s = g["cscore"][b][sel]
            assert (np.diff(s) <= 0).all()
            for j in np.nonzero(sel)[0]:
                u, v = g["cpar"][b, j], g["ctok"][b, j]
                rank = list(g["ttok"][b, u]).index(v)
                assert abs(g["cscore"][b, j] - (g["path"][b, u] + g["tlp"][b, u, rank])) <= 1e-5 * (1 + abs(s[0]))
            np.testing.assert_allclose(g["cscore"][b][sel], r["cand_score"][b][sel], rtol=1e-5, atol=5e-4)
    return g, r, st


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workloads_match_oracle(name):
    inp = synth.make_sample_inputs(synth.WORKLOADS[name])
    N = inp["parents"].shape[1]
    k = 8
    budget = min(64, N * k)
    _, _, st = compare(inp["draft_logits"], inp["tokens"], inp["parents"], inp["n_nodes"], 1.0, k, budget)
    assert st == 0


@pytest.mark.parametrize("T,k,budget", [(0.6, 1, 1), (1.7, 16, 0), (1.0, 0, 0), (1.0, 16, 16 * 20)])
def test_options(T, k, budget):
    gen = torch.Generator().manual_seed(31)
    B, N, V = 3, 20, 4096
    parents = torch.tensor([synth.random_tree(gen, N, 8, 4) for _ in range(B)], dtype=torch.int32)
    draft = (2 * torch.randn((B, N, V), generator=gen)).to(torch.bfloat16)
    tokens = torch.randint(0, V, (B, N), generator=gen, dtype=torch.int32)
    compare(draft, tokens, parents, torch.full((B,), N, dtype=torch.int32), T, k, budget)


def test_ties_padding_malformed_and_out_of_range():
    """Equal logits within and across chunks (the lower index first), ragged
    n_nodes, a malformed tree and tokens outside the vocabulary."""
    gen = torch.Generator().manual_seed(32)
    B, N, V = 4, 24, 151936
    parents = torch.tensor([synth.random_tree(gen, N, 8, 4) for _ in range(B)], dtype=torch.int32)
    draft = torch.randn((B, N, V), generator=gen).to(torch.bfloat16)
    for pos in (5, 77824 - 1, 77824, 77824 + 5, V - 1, 40000, 120000):     # ties on both sides of chunk cuts
        draft[:, :, pos] = 9.0
    n_nodes = torch.tensor([N, 17, 1, N], dtype=torch.int32)
    parents[3, 10] = 11                                                     # malformed
    tokens = torch.randint(0, V, (B, N), generator=gen, dtype=torch.int32)
    tokens[0, 3], tokens[0, 4] = V + 2, -1                                  # out of range: -inf
    g, r, st = compare(draft, tokens, parents, n_nodes, 1.0, 8, 40)
    assert st == jb.JF_STATUS_BAD_TREE
    assert np.isneginf(g["node"][0, 3]) and np.isneginf(g["node"][0, 4])
    assert g["ttok"][0, 0, :7].tolist() == [5, 40000, 77823, 77824, 77829, 120000, V - 1]


def test_topk_where_the_best_entries_crowd():
    """Layouts that defeat a bound taken from per-thread maxima: one thread
    holding 20 of a row's best entries in separate vectors, eight tied best
    entries in one vector, a constant row, and a row of equal values with a
    few larger ones (every entry then reaches the bound)."""
    B, N, V = 1, 5, 151936
    gen = torch.Generator().manual_seed(33)
    z = torch.randn((B, N, V), generator=gen)
    for j in range(20):                          # the vectors of one thread of the first chunk
        z[0, 0, 8 * (37 + 256 * j) + (j % 8)] = 20.0 + 0.25 * j
    z[0, 1, 8 * 1000: 8 * 1000 + 8] = 30.0       # one vector, eight ties
    z[0, 1, [3, 90001, 150000, 77830, 12345, 54321, 111111, 8 * 1000 + 9]] = 29.0
    z[0, 2] = 1.0                                # constant: the lowest indices
    z[0, 3] = -60.0
    z[0, 3, [17, 40000, 77824, 100000, V - 1]] = 3.0
    z[0, 4, 8 * (200 + 256 * 3)] = 50.0          # one entry far above the rest
    draft = z.to(torch.bfloat16)
    parents = torch.tensor([[-1, 0, 1, 1, 0]], dtype=torch.int32)
    tokens = torch.tensor([[0, 5, 7, V - 1, 77824]], dtype=torch.int32)
    for k, budget in ((16, 0), (16, 30), (3, 7)):
        g, r, st = compare(draft, tokens, parents, torch.tensor([N], dtype=torch.int32), 1.0, k, budget)
        assert st == 0
    g, r, st = compare(draft, tokens, parents, torch.tensor([N], dtype=torch.int32), 1.0, 16, 0)
    assert g["ttok"][0, 0].tolist() == [8 * (37 + 256 * j) + (j % 8) for j in range(19, 3, -1)]
    assert g["ttok"][0, 1, :8].tolist() == list(range(8000, 8008))
    assert g["ttok"][0, 2].tolist() == list(range(16))
    assert g["ttok"][0, 3].tolist() == [17, 40000, 77824, 100000, V - 1] + list(range(11))


def test_budget_when_thousands_of_candidates_tie():
    """Constant draft rows on a 256-node star: the root's candidates lead
    and the other 2040 are exactly equal, so the selection (ties to the
    lower (node, rank)) takes more than a short list can hold."""
    B, N, V = 1, 256, 4096
    draft = torch.zeros((B, N, V), dtype=torch.bfloat16)
    parents = torch.tensor([[-1] + [0] * (N - 1)], dtype=torch.int32)
    tokens = torch.arange(N, dtype=torch.int32).reshape(1, N)
    for k, budget in ((8, 64), (8, 256), (2, 100)):
        g, r, st = compare(draft, tokens, parents, torch.tensor([N], dtype=torch.int32), 1.0, k, budget)
        assert st == 0
        np.testing.assert_array_equal(g["cpar"][0], r["cand_parent"][0])
        np.testing.assert_array_equal(g["ctok"][0], r["cand_token"][0])


def test_largest_direct_budget_and_top16_at_tree256():
    """Top 16 and a budget of 128 (the largest the bucket selection takes)
    on the Qwen3-8B tree-256 shape: 4096 candidates a sequence."""
    inp = synth.make_sample_inputs(synth.WORKLOADS["qwen3_8b_tree256"])
    _, _, st = compare(inp["draft_logits"], inp["tokens"], inp["parents"], inp["n_nodes"], 1.0, 16, 128)
    assert st == 0
