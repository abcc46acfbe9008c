"""Failure detection without a GPU fault: a bounded wait that runs out.

Every wait in the attention kernel is bounded; when one runs out the kernel
raises JF_STATUS_TIMEOUT in `status`, every warp leaves its loop, the copies
and MMAs in flight are waited for, TMEM is freed and the call returns. A
second build of the library (JF_STALL_TEST) leaves each CTA's first K tile
load un-issued, so its first QK^T waits on a barrier that nothing completes;
the build gives every wait a 20 ms limit. The test checks that the call ends
with the flag raised and that the context stays usable: the normal library
then computes a correct result in the same process.
"""

import time

import numpy as np
import pytest
import torch

from tree_masked_attention_causal_gb300 import _build, binding as jb, synth
from helpers import assert_attention_close, oracle_attention, out_f64, shape_of, to_dev, valid_rows

pytestmark = pytest.mark.gpu


def test_attention_wait_runs_out_sets_status_and_returns():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    stall = jb.open_library(_build.build_variant("stall", ["JF_STALL_TEST", "JF_WAIT_NS=20000000ull"]))
    _build.build()
    inp = synth.make_inputs(synth.WORKLOADS["qwen3_8b_tree16"])
    dev = to_dev(inp)
    shape = shape_of(inp)
    ws = torch.zeros(jb.jf_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(dev["q"])
    t0 = time.time()
    jb.jf_tree_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["prefix_lens"], dev["tree_k"],
                         dev["tree_v"], dev["parents"], dev["n_nodes"], out, shape, ws, status=status, lib=stall)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30.0
    assert int(status.item()) & jb.JF_STATUS_TIMEOUT
    # the context is still usable, and the normal build computes the right thing
    status.zero_()
    jb.jf_tree_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["prefix_lens"], dev["tree_k"],
                         dev["tree_v"], dev["parents"], dev["n_nodes"], out, shape, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = valid_rows(inp)
    assert_attention_close(out_f64(out), oracle_attention(inp), rows, "after a timed-out call", strict=True)
