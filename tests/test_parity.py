"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Accept lengths, paths and argmax must match bit for bit. Attention outputs
must be within max-abs 1e-2 and mean-abs 1e-3 of the fp64 oracle, on
unit-variance bf16 inputs. Every call runs with guard zones around `out`,
and padding rows must still hold the sentinel.
"""

import numpy as np
import pytest
import torch

from tree_masked_attention_causal_gb300 import synth
import oracle
from helpers import (assert_attention_close, lib, oracle_attention, out_bits, out_f64, padding_untouched,
                     run_attention, run_verify, shape_of, small_inputs, to_dev, valid_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib()


# The five workloads, every row of every one.
FULL = ["tiny", "qwen3_8b_tree16", "qwen3_8b_tree256", "qwen3_30b_a3b_tree256"]


@pytest.mark.parametrize("name", FULL + ["serving_16x64"])
def test_workload_attention(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    dev = to_dev(inp)
    shape = shape_of(inp)
    out, status = run_attention(dev, shape)
    assert status == 0
    got = out_f64(out)
    rows = valid_rows(inp)                          # every node of every sequence (1024 for the serving batch)
    ref = oracle_attention(inp)
    assert_attention_close(got, ref, rows, name, strict=True)


@pytest.mark.parametrize("name", FULL + ["serving_16x64"])
def test_workload_verify(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    dev = to_dev(inp)
    alen, path, am, status = run_verify(dev, shape_of(inp), max_depth=16)
    assert status == 0
    r_len, r_path, r_am = oracle.tree_verify(inp["logits"], inp["tokens"], inp["parents"], inp["n_nodes"], 16)
    np.testing.assert_array_equal(am, r_am)
    np.testing.assert_array_equal(alen, r_len)
    np.testing.assert_array_equal(path, r_path)
    np.testing.assert_array_equal(alen, inp["planted_len"].numpy())


def check_attention(inp, scale=0.0, rows=None, what=None):
    import inspect
    dev = to_dev(inp)
    shape = shape_of(inp, scale)
    out, status = run_attention(dev, shape)
    ref = oracle_attention(inp, scale=scale)
    rows = rows if rows is not None else valid_rows(inp)
    assert_attention_close(out_f64(out), ref, rows, what or inspect.stack()[1].function)
    assert padding_untouched(out_bits(out), inp)
    return out, status


@pytest.mark.parametrize("G,d", [(1, 64), (2, 128), (4, 64), (8, 128), (16, 64), (32, 128), (64, 64), (128, 128)])
def test_gqa_groups_and_head_dims(G, d):
    Hkv = 2
    inp = small_inputs(10 + G, B=2, N=40, Hq=G * Hkv, Hkv=Hkv, d=d, Pcap=300)
    check_attention(inp)


def test_many_sequences_mixed_lengths():
    """Many small and large work units: the stream-K split cuts some units
    into several pieces, leaves others whole, and CTAs cross unit
    boundaries; prefixes of 0, 1, 127, 128, 129 tokens and ragged trees."""
    B = 12
    prefixes = torch.tensor([0, 1, 127, 128, 129, 700, 5, 640, 0, 300, 64, 1000], dtype=torch.int32)
    n_nodes = torch.tensor([40, 1, 17, 33, 40, 2, 39, 40, 8, 31, 40, 25], dtype=torch.int32)
    inp = small_inputs(50, B=B, N=40, Hq=8, Hkv=2, d=128, Pcap=1024, prefixes=prefixes, n_nodes=n_nodes)
    check_attention(inp)


def test_single_node_tree():
    inp = small_inputs(1, B=3, N=1, parents=torch.full((3, 1), -1, dtype=torch.int32), Pcap=333)
    check_attention(inp)


def test_chain_of_256():
    chain = torch.tensor([[-1] + list(range(255))], dtype=torch.int32)
    inp = small_inputs(2, B=1, N=256, Hq=4, Hkv=1, d=128, Pcap=129, parents=chain,
                       prefixes=torch.tensor([129], dtype=torch.int32))
    check_attention(inp)


def test_star_tree_256():
    star = torch.tensor([[-1] + [0] * 255], dtype=torch.int32)
    inp = small_inputs(3, B=1, N=256, Hq=8, Hkv=8, d=64, Pcap=64, parents=star)
    check_attention(inp)


def test_prefix_zero_and_full():
    inp = small_inputs(4, B=3, N=33, Pcap=256, prefixes=torch.tensor([0, 256, 128], dtype=torch.int32))
    check_attention(inp)


def test_ragged_n_nodes_leaves_padding_untouched():
    inp = small_inputs(5, B=4, N=96, Hq=8, Hkv=2, d=128, Pcap=700,
                       n_nodes=torch.tensor([96, 1, 37, 65], dtype=torch.int32))
    for b in range(4):                                  # padding parents: anything
        inp["parents"][b, int(inp["n_nodes"][b]):] = 12345
    check_attention(inp)


def test_nan_in_unused_cache_rows_and_padding_nodes():
    inp = small_inputs(6, B=2, N=50, Pcap=390, prefixes=torch.tensor([77, 389], dtype=torch.int32),
                       n_nodes=torch.tensor([50, 23], dtype=torch.int32), kv_fill=float("nan"))
    inp["tree_k"][1, 23:] = float("nan")
    inp["tree_v"][1, 23:] = float("nan")
    inp["q"][1, 23:] = float("nan")
    check_attention(inp)


def test_custom_scale():
    inp = small_inputs(7, B=1, N=30, Pcap=150)
    check_attention(inp, scale=0.05)


def test_long_ragged_prefixes_split_kv():
    """Prefixes long enough that every query tile is split over CTAs."""
    inp = small_inputs(8, B=3, N=24, Hq=32, Hkv=8, d=128, Pcap=9000,
                       prefixes=torch.tensor([9000, 1, 4097], dtype=torch.int32))
    check_attention(inp)


def test_rotated_prefix_walk_ragged_with_nan_tails():
    """Prefix K/V beyond half the L2 (167 MB here), where each unit walks its
    prefix tiles from a rotated start: the ragged last tile of a prefix then
    falls inside a piece, and the cache rows past it hold NaN."""
    inp = small_inputs(10, B=3, N=24, Hq=32, Hkv=8, d=128, Pcap=24000,
                       prefixes=torch.tensor([23999, 130, 16385], dtype=torch.int32), kv_fill=float("nan"))
    check_attention(inp)


@pytest.mark.parametrize("vscale", [1e5, 1e30])
def test_values_beyond_fp16_in_split_units(vscale):
    """V far beyond fp16's largest value (65504), on prefixes long enough
    that every unit is split: the split pieces keep their rows in fp16
    scaled by a power of two per half row, so split and whole units alike
    must match the oracle (compared after dividing both by the scale)."""
    inp = small_inputs(8, B=3, N=24, Hq=32, Hkv=8, d=128, Pcap=9000,
                       prefixes=torch.tensor([9000, 1, 4097], dtype=torch.int32))
    inp["v_cache"] = (inp["v_cache"].float() * vscale).to(torch.bfloat16)
    inp["tree_v"] = (inp["tree_v"].float() * vscale).to(torch.bfloat16)
    out, status = run_attention(to_dev(inp), shape_of(inp))
    assert status == 0
    got = out_f64(out)
    assert np.isfinite(got[:, :24]).all()
    ref = oracle_attention(inp)
    assert_attention_close(got / vscale, ref / vscale, valid_rows(inp), f"V x {vscale:g}")


def test_malformed_tree_flags_and_nans():
    inp = small_inputs(9, B=3, N=16, Pcap=100)
    inp["parents"][1, 5] = 7                           # parent not earlier
    inp["n_nodes"][2] = 0                              # out of range
    dev = to_dev(inp)
    out, status = run_attention(dev, shape_of(inp))
    assert status & 1
    o = out.float().cpu()
    assert torch.isnan(o[1]).all() and torch.isnan(o[2]).all()
    ref = oracle_attention(inp)
    assert_attention_close(out_f64(out), ref, [(0, i) for i in range(16)])


def test_repeat_calls_are_deterministic_and_reuse_workspace():
    inp = small_inputs(11, B=2, N=64, Hq=32, Hkv=8, d=128, Pcap=3000)
    dev = to_dev(inp)
    shape = shape_of(inp)
    from helpers import new_workspace
    ws = new_workspace(shape)
    a, _ = run_attention(dev, shape, ws=ws)
    b, _ = run_attention(dev, shape, ws=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ verify

def check_verify(inp, max_depth=16):
    dev = to_dev(inp)
    alen, path, am, status = run_verify(dev, shape_of(inp), max_depth=max_depth)
    r_len, r_path, r_am = oracle.tree_verify(inp["logits"], inp["tokens"], inp["parents"], inp["n_nodes"], max_depth)
    np.testing.assert_array_equal(am, r_am)
    np.testing.assert_array_equal(alen, r_len)
    np.testing.assert_array_equal(path, r_path)
    return status


def test_verify_ties_nan_and_signed_zero():
    inp = small_inputs(20, B=2, N=8, vocab=110000)     # 16 rows: 4096-element argmax chunks
    lg = inp["logits"]
    lg[0, 0] = 0.0
    lg[0, 1, 20000] = 9.0
    lg[0, 1, 105000] = 9.0                             # tie across chunks: lowest index
    lg[0, 2, 5] = float("nan")
    lg[0, 2, 60000] = float("nan")                     # first NaN wins
    lg[0, 3] = -0.0
    lg[0, 3, 57000] = 0.0                              # +0 == -0: index 0 wins
    lg[0, 4] = float("-inf")
    lg[0, 5, 109999] = float("inf")
    lg[0, 6, 49151] = 10.0                             # chunk boundary
    lg[0, 6, 49152] = 10.0
    lg[0, 7, 51201] = float("nan")                     # NaN only in a later chunk
    lg[1, 0, 3] = 10.0
    lg[1, 0, 7] = 10.0                                 # tie inside one 8-element vector
    check_verify(inp)


def test_verify_duplicate_sibling_tokens_and_cut_path():
    N = 12
    par = torch.tensor([[-1, 0, 0, 1, 2, 3, 4, 5, 6, 7, 8, 9]], dtype=torch.int32)
    inp = small_inputs(21, B=1, N=N, parents=par, vocab=64)
    top = torch.arange(N) % 7 + 3
    lg = torch.zeros(1, N, 64)
    lg[0, torch.arange(N), top] = 5.0
    inp["logits"] = lg.to(torch.bfloat16)
    tok = torch.zeros(1, N, dtype=torch.int32)
    for c in range(1, N):
        tok[0, c] = top[par[0, c]]
    inp["tokens"] = tok
    check_verify(inp, max_depth=16)
    check_verify(inp, max_depth=3)
    check_verify(inp, max_depth=0)


def test_verify_ragged_and_malformed():
    inp = small_inputs(22, B=4, N=40, vocab=1000, n_nodes=torch.tensor([40, 1, 17, 0], dtype=torch.int32))
    inp["parents"][2, 17:] = 999
    inp["parents"][0, 9] = 9
    status = check_verify(inp)
    assert status & 1


def test_verify_chain_of_256_deep_paths():
    """A 256-node chain: every edge agrees up to node 200, then one breaks;
    paths deeper than max_depth are cut."""
    N = 256
    par = torch.tensor([[-1] + list(range(N - 1))], dtype=torch.int32)
    inp = small_inputs(24, B=1, N=N, parents=par, vocab=16)
    top = inp["logits"][0].float().argmax(-1)          # no ties: N(0,1) bf16 logits, 16 values a row
    tok = torch.zeros(1, N, dtype=torch.int32)
    for c in range(1, N):
        tok[0, c] = top[c - 1] if c <= 200 else (top[c - 1] + 1) % 16
    inp["tokens"] = tok
    for md in (255, 200, 64, 0):
        check_verify(inp, max_depth=md)


def test_verify_random_trees_many_matches():
    """Small vocabulary so that many edges agree and long paths form."""
    for seed in range(3):
        inp = small_inputs(30 + seed, B=8, N=64, vocab=8)
        check_verify(inp, max_depth=63)


@pytest.mark.parametrize("B,N", [(2, 8), (2, 256)])
def test_verify_ties_at_chunk_boundaries(B, N):
    """Equal maxima on both sides of 2048-element boundaries (every argmax
    chunk ends on one), ties just past them and NaN on both sides: with few
    rows (short chunks) and with many (two chunks per row of 151936)."""
    V = 151936
    inp = small_inputs(23, B=B, N=N, vocab=V)
    lg = inp["logits"]
    for r in range(B * N):
        b, i = divmod(r, N)
        e = ((r % 74) + 1) * 2048
        if r % 3 == 0:
            lg[b, i, e - 1] = 9.0
            lg[b, i, e] = 9.0
        elif r % 3 == 1:
            lg[b, i, e] = 9.0
            lg[b, i, e + 5] = 9.0
        else:
            lg[b, i, e - 2048] = float("nan")
            lg[b, i, e] = float("nan")
    check_verify(inp)


def test_verify_all_chunks_vocab_151936():
    inp = small_inputs(40, B=2, N=5, vocab=151936)
    check_verify(inp)
