"""The allocation-free verify entry point, jf_tree_verify_noalloc.

Some callers cannot allocate device memory, so they cannot give the library
a workspace. Examples: a CUDA graph being captured, an allocator that owns
the whole device, or an embedding that forbids cudaMalloc after start-up.
This entry point keeps its scratch in a fixed device array inside the
library.

The tests check that it returns exactly what jf_tree_verify (workspace
variant) returns, on two calls in a row with different inputs. The array
keeps the previous call's contents, so the second call also checks that
nothing stale leaks through. Problems larger than the array must be
refused before anything is launched. This file is named to be collected
last.
"""

import numpy as np
import pytest
import torch

import oracle
from tree_masked_attention_causal_gb300 import _build, binding as jb, synth

A16 = 1 << 20            # fake aligned address, never dereferenced


def test_noalloc_refuses_problems_beyond_the_array():
    _build.build()
    # 4 x 256 rows x 2 chunks x 8 B = 16 KB fits; 200 x 256 rows of vocab
    # 262144 (4 chunks of 65536) x 8 B = 1.6 MB does not
    ok = jb.make_shape(4, 0, 0, 0, 256, 0, 151936)
    too_big = jb.make_shape(200, 0, 0, 0, 256, 0, 262144)
    assert jb.jf_tree_verify_noalloc(A16, A16, A16, A16, A16, A16, None, too_big, 16, stream=0,
                                     check=False) == jb.JF_ERR_SHAPE
    assert jb.jf_tree_verify_noalloc(None, A16, A16, A16, A16, A16, None, ok, 16, stream=0,
                                     check=False) == jb.JF_ERR_NULL


def _run_both(name, max_depth=16):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    dev = {k: v.cuda() for k, v in inp.items() if isinstance(v, torch.Tensor)}
    B, N = inp["tokens"].shape
    shape = jb.make_shape(B, 0, 0, 0, N, 0, inp["logits"].shape[-1])
    outs = []
    for variant in ("workspace", "noalloc"):
        alen = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        path = torch.full((B, max_depth + 1), -9, dtype=torch.int32, device="cuda")
        am = torch.full((B, N), -9, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if variant == "workspace":
            ws = torch.empty(jb.jf_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
            jb.jf_tree_verify(dev["logits"], dev["tokens"], dev["parents"], dev["n_nodes"], alen, path, am, shape,
                              max_depth, ws, status=status)
        else:
            jb.jf_tree_verify_noalloc(dev["logits"], dev["tokens"], dev["parents"], dev["n_nodes"], alen, path, am,
                                      shape, max_depth, status=status)
        torch.cuda.synchronize()
        outs.append((alen.cpu(), path.cpu(), am.cpu(), int(status.item())))
    return inp, outs


@pytest.mark.gpu
def test_noalloc_matches_workspace_variant_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _build.build()
    for name in ("serving_16x64", "qwen3_8b_tree256"):        # two different calls in a row
        inp, (ref, got) = _run_both(name)
        for r, g in zip(ref[:3], got[:3]):
            assert torch.equal(r, g), name
        assert ref[3] == got[3] == 0
        assert torch.equal(got[0], inp["planted_len"])
        # and directly against the fp64 oracle's argmax, lengths and paths
        r_len, r_path, r_am = oracle.tree_verify(inp["logits"], inp["tokens"], inp["parents"], inp["n_nodes"], 16)
        np.testing.assert_array_equal(got[0].numpy(), r_len)
        np.testing.assert_array_equal(got[1].numpy(), r_path)
        np.testing.assert_array_equal(got[2].numpy(), r_am)
