"""GPU parity of stochastic tree verification (jf_tree_verify_sample)
against the oracle.

Accept lengths, paths and next tokens must be equal. Both sides draw the
same Philox4x64-10 numbers; the oracle decides in fp64, the kernels in
fp32 from chunked sums, so a decision whose margin is within fp32 rounding
could go either way. The oracle reports each sequence's smallest margins
(acceptance test |U - ratio|, residual mass, Gumbel top-2 gap); sequences
with a margin under SAFE are not compared, and every test requires that
almost all of its sequences are compared.
"""

import numpy as np
import pytest
import torch

import oracle
from tree_masked_attention_causal_gb300 import binding as jb, synth
from helpers import lib, new_workspace

pytestmark = pytest.mark.gpu

# fp32 relative error of a ratio or a mass here is ~1e-6, of a Gumbel key
# ~1e-5 absolute: these margins leave two orders of magnitude
SAFE = (1e-4, 1e-4, 1e-3)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib()


def shape_for(target, B, N):
    return jb.make_shape(B, 1, 1, 64, N, 1, target.shape[-1])


def run(inp, T, seed, offset, max_depth=16, status=None, ws=None):
    tg, dr = inp["target_logits"], inp["draft_logits"]
    B, N, V = tg.shape
    shape = shape_for(tg, B, N)
    dev = {k: inp[k].cuda() for k in ("target_logits", "draft_logits", "tokens", "parents", "n_nodes")}
    alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, max_depth + 1), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    jb.jf_tree_verify_sample(dev["target_logits"], dev["draft_logits"], dev["tokens"], dev["parents"],
                             dev["n_nodes"], T, seed, offset, alen, path, nxt, shape, max_depth,
                             new_workspace(shape) if ws is None else ws, status=st)
    torch.cuda.synchronize()
    return alen.cpu().numpy(), path.cpu().numpy(), nxt.cpu().numpy(), int(st.item())


def compare(inp, T, seed, offset, max_depth=16, min_safe=0.9):
    alen, path, nxt, st = run(inp, T, seed, offset, max_depth)
    r_alen, r_path, r_nxt, m = oracle.tree_verify_sample(inp["target_logits"], inp["draft_logits"], inp["tokens"],
                                                         inp["parents"], inp["n_nodes"], max_depth, T, seed, offset)
    safe = (m[:, 0] > SAFE[0]) & (m[:, 1] > SAFE[1]) & (m[:, 2] > SAFE[2])
    assert safe.mean() >= min_safe, f"only {safe.sum()} of {len(safe)} sequences have safe margins"
    np.testing.assert_array_equal(alen[safe], r_alen[safe])
    np.testing.assert_array_equal(path[safe], r_path[safe])
    np.testing.assert_array_equal(nxt[safe], r_nxt[safe])
    assert st == 0
    return alen, path, nxt, r_alen, safe


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workloads_match_oracle(name):
    inp = synth.make_sample_inputs(synth.WORKLOADS[name])
    lens = []
    for offset in range(3):
        alen, *_ = compare(inp, 1.0, 1234, offset, min_safe=1.0 if inp["parents"].shape[0] == 1 else 0.9)
        lens.extend(alen.tolist())
    assert max(lens) >= 2                        # paths are accepted, not only the root


@pytest.mark.parametrize("T", [0.5, 2.0])
def test_other_temperatures(T):
    w = synth.WORKLOADS["qwen3_8b_tree16"]
    inp = synth.make_sample_inputs(w, temperature=T)
    compare(inp, T, 99, 5, min_safe=1.0)


def test_batch_of_star_trees_matches_oracle_and_target_distribution():
    """8000 roots with 3 children drawn from q, V = 8: equal to the oracle
    sequence by sequence, and the first emitted token follows p."""
    rng = np.random.default_rng(5)
    B, k, V, T = 8000, 3, 8, 1.0
    pl = rng.normal(size=V) * 1.5
    ql = rng.normal(size=V) * 1.5
    N = k + 1
    to_bf = lambda x: torch.tensor(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    q = torch.softmax(to_bf(ql).double() / T, -1).numpy()
    p = torch.softmax(to_bf(pl).double() / T, -1).numpy()
    tokens = np.zeros((B, N), dtype=np.int32)
    tokens[:, 1:] = rng.choice(V, size=(B, k), p=q)
    parents = np.zeros((B, N), dtype=np.int32)
    parents[:, 0] = -1
    inp = dict(target_logits=to_bf(np.broadcast_to(pl, (B, N, V))), draft_logits=to_bf(np.broadcast_to(ql, (B, N, V))),
               tokens=torch.tensor(tokens), parents=torch.tensor(parents),
               n_nodes=torch.full((B,), N, dtype=torch.int32))
    alen, path, nxt, _, _ = compare(inp, T, 2024, 0, max_depth=4, min_safe=0.99)
    first = np.where(alen >= 2, tokens[np.arange(B), np.maximum(path[:, 1], 0)], nxt)
    counts = np.bincount(first, minlength=V)
    stat = (((counts - B * p) ** 2) / (B * p)).sum()
    assert stat < 24.32                          # chi-square, 7 dof, 0.1%


def test_edge_cases():
    """Malformed trees, out-of-range tokens, a single node, max_depth 0 and
    a cut path, in one batch; the malformed ones raise BAD_TREE."""
    rng = np.random.default_rng(8)
    B, N, V = 6, 12, 1024
    tg = torch.tensor(rng.normal(size=(B, N, V)).astype(np.float32) * 2).to(torch.bfloat16)
    dr = torch.tensor(rng.normal(size=(B, N, V)).astype(np.float32) * 2).to(torch.bfloat16)
    parents = np.array([[-1] + list(range(N - 1))] * B, dtype=np.int32)     # chains
    parents[1, 3] = 5                                                       # malformed (forward edge)
    n_nodes = np.full(B, N, dtype=np.int32)
    n_nodes[2] = 1                                                          # a single node
    n_nodes[3] = 0                                                          # malformed (no root)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    tokens[4, 1:] = [V + 5, -3] + [0] * (N - 3)                             # out of range: rejected
    # sequence 5: draft = target along the chain: every node is accepted, cut by max_depth
    dr[5] = tg[5]
    inp = dict(target_logits=tg, draft_logits=dr, tokens=torch.tensor(tokens), parents=torch.tensor(parents),
               n_nodes=torch.tensor(n_nodes))
    for max_depth in (0, 3, 16):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        alen, path, nxt, s = run(inp, 1.0, 7, 3, max_depth=max_depth, status=st)
        r_alen, r_path, r_nxt, m = oracle.tree_verify_sample(tg, dr, tokens, parents, n_nodes, max_depth, 1.0, 7, 3)
        np.testing.assert_array_equal(alen, r_alen)
        np.testing.assert_array_equal(path, r_path)
        np.testing.assert_array_equal(nxt, r_nxt)
        assert s == jb.JF_STATUS_BAD_TREE
        assert alen[1] == 0 and alen[3] == 0 and nxt[1] == -1 and (path[1] == -1).all()
        assert alen[2] == 1 and alen[4] == 1
        assert alen[5] == min(max_depth, N - 1) + 1


def test_flat_draft_near_zero_temperature_is_greedy():
    """A flat draft at T = 0.01 with well-separated target logits: the
    path and next token of jf_tree_verify's greedy rule."""
    rng = np.random.default_rng(12)
    B, N, V = 4, 32, 256                         # integer logits 0..255: exact in bf16, gaps >= 1
    lg = np.stack([np.stack([rng.permutation(V) for _ in range(N)]) for _ in range(B)]).astype(np.float32)
    am = lg.argmax(-1)
    parents = np.zeros((B, N), dtype=np.int32)
    tokens = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        parents[b, 0] = -1
        used = {}
        for c in range(1, N):
            p = int(rng.integers(0, c))
            parents[b, c] = p
            taken = used.setdefault(p, set())
            t = int(am[b, p]) if (int(am[b, p]) not in taken and rng.random() < 0.6) else \
                int(next(x for x in rng.permutation(V) if x not in taken and x != am[b, p]))
            taken.add(t)
            tokens[b, c] = t
    tg = torch.tensor(lg).to(torch.bfloat16)
    inp = dict(target_logits=tg, draft_logits=torch.zeros_like(tg), tokens=torch.tensor(tokens),
               parents=torch.tensor(parents), n_nodes=torch.full((B,), N, dtype=torch.int32))
    alen, path, nxt, st = run(inp, 0.01, 3, 0)
    g_alen, g_path, g_am = oracle.tree_verify(tg, tokens, parents, np.full(B, N, np.int32), 16)
    np.testing.assert_array_equal(alen, g_alen)
    np.testing.assert_array_equal(path, g_path)
    last = path[np.arange(B), alen - 1]
    np.testing.assert_array_equal(nxt, g_am[np.arange(B), last])
    assert st == 0


def test_repeatable_and_offset_changes_the_draws():
    w = synth.WORKLOADS["serving_16x64"]
    inp = synth.make_sample_inputs(w)
    a1 = run(inp, 1.0, 11, 0)
    a2 = run(inp, 1.0, 11, 0)
    for x, y in zip(a1[:3], a2[:3]):
        np.testing.assert_array_equal(x, y)
    a3 = run(inp, 1.0, 11, 1)
    assert (a3[2] != a1[2]).mean() > 0.5
