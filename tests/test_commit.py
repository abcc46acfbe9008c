"""GPU parity of the accepted-path KV commit (jf_tree_commit_kv) against the
oracle: the whole KV caches, the prefix lengths and the status flags must
match bit for bit.

The accepted paths come from the GPU's own jf_tree_verify on the same
inputs (itself bit-exact against the oracle, tests/test_parity.py), so the
test runs the step the way a caller does: verify, then commit.
"""

import numpy as np
import pytest
import torch

import oracle
from tree_masked_attention_causal_gb300 import binding as jb, synth
from helpers import lib, new_workspace, shape_of, small_inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def verify_then_commit(inp, max_depth=16, alen=None, path=None, prefix_lens=None):
    """Run the GPU verify (unless alen/path are given), then the GPU commit
    and the oracle commit on the same requests; compare everything."""
    dev = to_dev(inp)
    shape = shape_of(inp)
    B, N = inp["parents"].shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if alen is None:
        a = torch.empty(B, dtype=torch.int32, device="cuda")
        p = torch.empty(B, max_depth + 1, dtype=torch.int32, device="cuda")
        jb.jf_tree_verify(dev["logits"], dev["tokens"], dev["parents"], dev["n_nodes"], a, p, None, shape,
                          max_depth, new_workspace(shape), status=status)
        status.zero_()
    else:
        a, p = alen.to(torch.int32).cuda(), path.to(torch.int32).cuda()
    pl = (inp["prefix_lens"] if prefix_lens is None else prefix_lens).to(torch.int32)
    kc, vc, pld = dev["k_cache"].clone(), dev["v_cache"].clone(), pl.cuda()
    jb.jf_tree_commit_kv(dev["tree_k"], dev["tree_v"], dev["n_nodes"], a, p, kc, vc, pld, shape, max_depth,
                         status=status)
    torch.cuda.synchronize()
    r_k, r_v, r_pl, r_flags = oracle.commit_kv(inp["tree_k"], inp["tree_v"], inp["n_nodes"], a.cpu(), p.cpu(),
                                               inp["k_cache"], inp["v_cache"], pl, max_depth)
    np.testing.assert_array_equal(pld.cpu().numpy(), r_pl)
    np.testing.assert_array_equal(_bits(kc), r_k)
    np.testing.assert_array_equal(_bits(vc), r_v)
    st = int(status.item())
    assert bool(st & jb.JF_STATUS_BAD_TREE) == bool((r_flags == 1).any())
    assert bool(st & jb.JF_STATUS_CACHE_FULL) == bool((r_flags == 2).any())
    return a.cpu(), pld.cpu(), r_flags


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_commit(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    # room for the accepted path: the caches of these workloads are exactly
    # as long as their longest prefix, so commit onto shorter prefixes
    pl = (inp["prefix_lens"] - 16).clamp(min=0)
    a, pld, flags = verify_then_commit(inp, prefix_lens=pl)
    np.testing.assert_array_equal(a.numpy(), inp["planted_len"].numpy())
    assert (flags == 0).all()
    np.testing.assert_array_equal(pld.numpy(), (pl + a).numpy())


def test_commit_cut_paths_and_full_cache():
    """Paths cut by max_depth 0 and 3; one sequence whose cache is nearly
    full (no room) and one that fills it exactly; one with no prefix."""
    inp = small_inputs(60, B=4, N=40, Hq=8, Hkv=2, d=128, Pcap=50, vocab=8,
                       prefixes=torch.tensor([49, 0, 20, 45], dtype=torch.int32))
    for md in (0, 3, 16):
        verify_then_commit(inp, max_depth=md)


def test_commit_malformed_requests_and_nan_rows():
    """Malformed trees (verify reports 0: nothing changes), paths through
    nodes outside the tree, lengths above the tree or the slots, prefix
    lengths out of range, and NaN in the copied rows (copied bit for bit)."""
    inp = small_inputs(61, B=6, N=16, Hq=4, Hkv=1, d=64, Pcap=64, vocab=8,
                       n_nodes=torch.tensor([16, 16, 16, 5, 16, 16], dtype=torch.int32))
    inp["tree_k"][0, 3] = float("nan")
    inp["tree_v"][0, 3] = float("nan")
    md = 4
    alen = torch.tensor([3, 0, 2, 4, 3, 6], dtype=torch.int32)
    path = torch.full((6, md + 1), -1, dtype=torch.int32)
    path[0, :3] = torch.tensor([0, 3, 7])
    path[2, :2] = torch.tensor([0, 16])             # node 16 is padding
    path[3, :4] = torch.tensor([0, 1, 2, 3])        # a = 4 <= n = 5: fine
    path[4, :3] = torch.tensor([0, 1, 2])
    path[5, :5] = torch.tensor([0, 1, 2, 3, 4])     # a = 6 > max_depth + 1
    pl = torch.tensor([10, 10, 10, 10, 65, 10], dtype=torch.int32)   # sequence 4: prefix beyond the cache
    _, pld, flags = verify_then_commit(inp, max_depth=md, alen=alen, path=path, prefix_lens=pl)
    np.testing.assert_array_equal(flags, [0, 0, 1, 0, 1, 1])


def test_commit_then_attention_sees_the_committed_rows():
    """After a commit of a whole chain, the next attention call over the
    longer prefix computes what the tree attention over the chain computed
    (the GPU path end to end: attention, commit, attention)."""
    from helpers import assert_attention_close, oracle_attention, out_f64, run_attention
    B, N, Hq, Hkv, d, P = 2, 24, 8, 2, 128, 100
    chain = torch.tensor([[-1] + list(range(N - 1))] * B, dtype=torch.int32)
    inp = small_inputs(62, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, Pcap=P + N, parents=chain,
                       prefixes=torch.full((B,), P, dtype=torch.int32))
    ref = oracle_attention(inp)
    alen = torch.full((B,), N, dtype=torch.int32)
    path = torch.arange(N, dtype=torch.int32).repeat(B, 1)
    dev = to_dev(inp)
    shape = shape_of(inp)
    pld = dev["prefix_lens"].clone()
    jb.jf_tree_commit_kv(dev["tree_k"], dev["tree_v"], dev["n_nodes"], alen.cuda(), path.cuda(), dev["k_cache"],
                         dev["v_cache"], pld, shape, N - 1)
    torch.cuda.synchronize()
    assert (pld.cpu() == P + N).all()
    # node i alone, over the committed prefix cut at P + i
    for i in (0, 7, N - 1):
        one = dict(inp)
        one.update(q=inp["q"][:, i:i + 1].contiguous(), tree_k=inp["tree_k"][:, i:i + 1].contiguous(),
                   tree_v=inp["tree_v"][:, i:i + 1].contiguous(), parents=torch.full((B, 1), -1, dtype=torch.int32),
                   n_nodes=torch.ones(B, dtype=torch.int32), prefix_lens=torch.full((B,), P + i, dtype=torch.int32))
        dev1 = to_dev(one)
        dev1["k_cache"], dev1["v_cache"] = dev["k_cache"], dev["v_cache"]
        out, st = run_attention(dev1, shape_of(one))
        assert st == 0
        assert_attention_close(out_f64(out), ref[:, i:i + 1], [(b, 0) for b in range(B)], f"node {i}", strict=True)


def full_tables(pg, prefix_cap):
    """Give every sequence a page for every row it may hold (its unused
    entries get fresh pages at the end of the pool), as a serving engine
    would before a commit."""
    table = pg["block_table"].clone()
    nxt = pg["num_pages"]
    per_seq = table.shape[1]
    for b in range(table.shape[0]):
        for j in range(per_seq):
            if table[b, j] < 0:
                table[b, j] = nxt
                nxt += 1
    shp = pg["k_pages"].shape[1:]
    kp = torch.cat([pg["k_pages"], torch.zeros((nxt - pg["num_pages"],) + tuple(shp), dtype=torch.bfloat16)])
    vp = torch.cat([pg["v_pages"], torch.zeros((nxt - pg["num_pages"],) + tuple(shp), dtype=torch.bfloat16)])
    return kp, vp, table, nxt


@pytest.mark.parametrize("page_size", [8, 64])
def test_paged_commit_matches_oracle(page_size):
    """Verify, then commit into a paged pool: every page, the prefix lengths
    and the flags against the oracle; one sequence without room."""
    inp = small_inputs(63, B=5, N=40, Hq=8, Hkv=2, d=128, Pcap=128, vocab=8,
                       prefixes=torch.tensor([100, 0, 125, 64, 128], dtype=torch.int32))
    dev = to_dev(inp)
    shape = shape_of(inp)
    md = 16
    a = torch.empty(5, dtype=torch.int32, device="cuda")
    p = torch.empty(5, md + 1, dtype=torch.int32, device="cuda")
    jb.jf_tree_verify(dev["logits"], dev["tokens"], dev["parents"], dev["n_nodes"], a, p, None, shape, md,
                      new_workspace(shape))
    pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], page_size, seed=9, spare_fill=0.0)
    kp, vp, table, num_pages = full_tables(pg, 128)
    kpd, vpd, pld = kp.cuda(), vp.cuda(), inp["prefix_lens"].cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    jb.jf_tree_commit_kv_paged(dev["tree_k"], dev["tree_v"], dev["n_nodes"], a, p, kpd, vpd, table.cuda(), page_size,
                               num_pages, pld, shape, md, status=st)
    torch.cuda.synchronize()
    rk, rv, rpl, rfl = oracle.commit_kv_paged(inp["tree_k"], inp["tree_v"], inp["n_nodes"], a.cpu(), p.cpu(), kp, vp,
                                              table, page_size, inp["prefix_lens"], md)
    np.testing.assert_array_equal(pld.cpu().numpy(), rpl)
    np.testing.assert_array_equal(_bits(kpd), rk)
    np.testing.assert_array_equal(_bits(vpd), rv)
    assert bool(int(st.item()) & jb.JF_STATUS_CACHE_FULL) == bool((rfl == 2).any())
    assert (rfl == 2).any() and (rfl == 0).sum() >= 3


def test_paged_chain_equals_contiguous_chain():
    """Paged attention, commit into pages, paged attention again: bit for
    bit what the contiguous calls give; a bad page flags its sequence."""
    B, N, Hq, Hkv, d, Pcap = 3, 24, 8, 2, 128, 256
    inp = small_inputs(64, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, Pcap=Pcap,
                       prefixes=torch.tensor([100, 17, 200], dtype=torch.int32))
    from helpers import run_attention
    shape = shape_of(inp)
    dev = to_dev(inp)
    alen = torch.tensor([5, 3, 4], dtype=torch.int32)
    path = torch.full((B, 17), -1, dtype=torch.int32)
    for b in range(B):
        node, chain = 0, [0]
        while len(chain) < int(alen[b]):
            kids = [c for c in range(N) if int(inp["parents"][b, c]) == node]
            if not kids:
                break
            node = kids[0]
            chain.append(node)
        alen[b] = len(chain)
        path[b, :len(chain)] = torch.tensor(chain)
    # contiguous chain
    kc, vc, plc = dev["k_cache"].clone(), dev["v_cache"].clone(), dev["prefix_lens"].clone()
    jb.jf_tree_commit_kv(dev["tree_k"], dev["tree_v"], dev["n_nodes"], alen.cuda(), path.cuda(), kc, vc, plc, shape, 16)
    dev2 = dict(dev)
    dev2.update(k_cache=kc, v_cache=vc, prefix_lens=plc)
    ref, _ = run_attention(dev2, shape)
    # paged chain
    pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], 16, seed=10)
    kp, vp, table, num_pages = full_tables(pg, Pcap)
    kpd, vpd, tabd, pld = kp.cuda(), vp.cuda(), table.cuda(), dev["prefix_lens"].clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    jb.jf_tree_commit_kv_paged(dev["tree_k"], dev["tree_v"], dev["n_nodes"], alen.cuda(), path.cuda(), kpd, vpd, tabd,
                               16, num_pages, pld, shape, 16, status=st)
    out = torch.empty_like(dev["q"])
    jb.jf_tree_attention_paged(dev["q"], kpd, vpd, tabd, 16, num_pages, pld, dev["tree_k"], dev["tree_v"],
                               dev["parents"], dev["n_nodes"], out, shape, new_workspace(shape), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(pld.cpu().numpy(), plc.cpu().numpy())
    np.testing.assert_array_equal(_bits(out), _bits(ref))
    # a page outside the pool where sequence 1's rows would go
    bad = tabd.clone()
    bad[1, int(pld[1]) // 16] = num_pages + 7
    pl_before = pld.clone()
    st.zero_()
    jb.jf_tree_commit_kv_paged(dev["tree_k"], dev["tree_v"], dev["n_nodes"], alen.cuda(), path.cuda(), kpd, vpd, bad,
                               16, num_pages, pld, shape, 16, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & jb.JF_STATUS_BAD_TREE
    assert int(pld[1]) == int(pl_before[1])
