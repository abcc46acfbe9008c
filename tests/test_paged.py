"""Tree attention over a paged prefix cache (jf_tree_attention_paged).

The pages of the shared pool are handed out in a shuffled order, and spare
pages full of NaN sit among them, so a row read from the wrong page shows.
The kernel runs the same tiles and arithmetic as over the contiguous cache,
so the outputs must be bit-identical to jf_tree_attention's on the same
cache; one page size is also compared with the oracle (the pages gathered
back into the cache they stand for, then the fp64 tree attention).
"""

import numpy as np
import pytest
import torch

import oracle
from tree_masked_attention_causal_gb300 import binding as jb, synth
from helpers import (assert_attention_close, lib, new_workspace, out_bits, out_f64, run_attention, shape_of,
                     small_inputs, to_dev, valid_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib()


def run_paged(inp, pg, shape, status=None):
    dev = to_dev(inp)
    B, N, Hq, d = inp["q"].shape
    out = torch.full((B, N, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    jb.jf_tree_attention_paged(dev["q"], pg["k_pages"].cuda(), pg["v_pages"].cuda(), pg["block_table"].cuda(),
                               pg["page_size"], pg["num_pages"], dev["prefix_lens"], dev["tree_k"], dev["tree_v"],
                               dev["parents"], dev["n_nodes"], out, shape, new_workspace(shape), status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def same_as_contiguous(inp, page_size, seed=0):
    shape = shape_of(inp)
    ref, st0 = run_attention(to_dev(inp), shape)
    pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], page_size, seed=seed)
    got, st = run_paged(inp, pg, shape)
    assert st == st0 == 0
    bi, ni = np.array(valid_rows(inp)).T
    np.testing.assert_array_equal(out_bits(got)[bi, ni].numpy(), out_bits(ref)[bi, ni].numpy())
    return got, pg


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128])
def test_serving_batch_bit_identical_to_contiguous(page_size):
    inp = synth.make_inputs(synth.WORKLOADS["serving_16x64"], with_logits=False)
    same_as_contiguous(inp, page_size, seed=page_size)


@pytest.mark.parametrize("name", ["qwen3_8b_tree256", "qwen3_30b_a3b_tree256", "tiny"])
def test_workloads_bit_identical_to_contiguous(name):
    inp = synth.make_inputs(synth.WORKLOADS[name], with_logits=False)
    same_as_contiguous(inp, 16 if name != "tiny" else 8)


def test_paged_matches_oracle():
    inp = small_inputs(41, B=6, N=40, Hq=16, Hkv=4, d=128, Pcap=512,
                       prefixes=torch.tensor([0, 1, 15, 16, 17, 512], dtype=torch.int32))
    shape = shape_of(inp)
    pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], 16, seed=3)
    got, st = run_paged(inp, pg, shape)
    assert st == 0
    ref = oracle.tree_attention_paged(inp["q"], pg["k_pages"], pg["v_pages"], pg["block_table"], 16, 512,
                                      inp["prefix_lens"], inp["tree_k"], inp["tree_v"], inp["parents"],
                                      inp["n_nodes"])
    assert_attention_close(out_f64(got), ref, valid_rows(inp), what="paged vs oracle")


def test_bad_block_table_entry_flags_only_its_sequence():
    inp = small_inputs(42, B=3, N=12, Hq=8, Hkv=2, d=64, Pcap=256,
                       prefixes=torch.tensor([200, 100, 64], dtype=torch.int32))
    shape = shape_of(inp)
    ref, _ = run_attention(to_dev(inp), shape)
    pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], 32, seed=5)
    pg["block_table"] = pg["block_table"].clone()
    pg["block_table"][1, 2] = pg["num_pages"]                    # used page 2 of sequence 1 (rows 64..95)
    got, st = run_paged(inp, pg, shape)
    assert st == jb.JF_STATUS_BAD_TREE
    g = got.float().cpu().numpy()
    assert np.isnan(g[1]).all()
    np.testing.assert_array_equal(out_bits(got)[0].numpy(), out_bits(ref)[0].numpy())
    np.testing.assert_array_equal(out_bits(got)[2].numpy(), out_bits(ref)[2].numpy())
    pg["block_table"][1, 2] = -1
    got, st = run_paged(inp, pg, shape)
    assert st == jb.JF_STATUS_BAD_TREE and np.isnan(got[1].float().cpu().numpy()).all()


def test_entries_past_the_prefix_are_not_read():
    inp = small_inputs(43, B=2, N=10, Hq=8, Hkv=2, d=128, Pcap=384,
                       prefixes=torch.tensor([130, 7], dtype=torch.int32))
    shape = shape_of(inp)
    ref, _ = run_attention(to_dev(inp), shape)
    pg = synth.paged_layout(inp["k_cache"], inp["v_cache"], inp["prefix_lens"], 64, seed=6)
    pg["block_table"] = pg["block_table"].clone()
    pg["block_table"][0, 3:] = 2 ** 30                           # unused entries: garbage
    pg["block_table"][1, 1:] = -5
    got, st = run_paged(inp, pg, shape)
    assert st == 0
    np.testing.assert_array_equal(out_bits(got).numpy(), out_bits(ref).numpy())
