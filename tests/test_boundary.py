"""The C ABI boundary without a GPU.

The library must load on a machine without a GPU and export every function
that include/jf_tree.h declares. Every argument error that the host can
detect is reported before the first CUDA call, so these tests pass fake
(never dereferenced) pointers and never reach a kernel.
"""

import ctypes

import pytest

from tree_masked_attention_causal_gb300 import _build, binding as jb


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return jb.load()


def test_exports_every_header_symbol(lib):
    names = jb.header_symbols()
    assert {"jf_tree_attention", "jf_tree_verify", "jf_workspace_bytes", "jf_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def good_shape(**kw):
    d = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, max_nodes=64, prefix_cap=1000, vocab=4096)
    d.update(kw)
    return jb.make_shape(**d)


def test_workspace_bytes(lib):
    assert jb.jf_workspace_bytes(good_shape()) > 0
    assert jb.jf_workspace_bytes(good_shape(batch=4)) > jb.jf_workspace_bytes(good_shape())
    for bad in (dict(batch=0), dict(max_nodes=0), dict(max_nodes=257)):
        assert jb.jf_workspace_bytes(good_shape(**bad)) == 0
    # a verify-only shape (attention fields unset) still gets a workspace
    assert jb.jf_workspace_bytes(jb.make_shape(3, 0, 0, 0, 16, 0, 1024)) > 0
    # an attention-only shape (vocab unset) too
    assert jb.jf_workspace_bytes(good_shape(vocab=0)) > 0
    assert lib.jf_workspace_bytes(None) == 0


def _argmax_chunks(rows, V, sms=256):
    """Chunks per logits row, as include/jf_tree.h and the layout state it:
    pieces of about 76800 elements, more of them for few rows (up to ~4
    CTAs per SM, within one wave of 4 per SM), multiples of 2048. A call
    cuts them for its device's SM count; the workspace is sized for 256."""
    cdiv = lambda a, b: -(-a // b)
    per = cdiv(V, 76800)
    want = min(cdiv(4 * sms, rows), 4 * sms // rows)
    if want > per:
        per = min(want, cdiv(V, 2048))
    chunk = cdiv(cdiv(V, per), 2048) * 2048
    return cdiv(V, chunk)


@pytest.mark.parametrize("rows,V,expect", [(256, 151936, 2), (16, 151936, 38), (10, 151936, 38), (152, 151936, 4)])
def test_argmax_chunks_on_152_sms(rows, V, expect):
    """The chunking a call on a 152-SM GB300 uses (the rule, restated)."""
    assert _argmax_chunks(rows, V, sms=152) == expect


@pytest.mark.parametrize("B,N,V,expect", [(1, 256, 151936, 4), (1, 16, 151936, 38), (16, 64, 151936, 2),
                                          (2, 5, 151936, 75), (1, 16, 1024, 1), (4, 200, 262144, 4),
                                          (1, 152, 151936, 6)])
def test_argmax_chunk_rule(lib, B, N, V, expect):
    """The verify region of the workspace holds one int2 per (row, chunk)
    and the sampling region two float2 (target and draft; the scoring
    shares it): their growth from a one-chunk vocabulary pins the chunk
    count they are sized for (256 SMs, the bound for any device's
    chunking)."""
    assert _argmax_chunks(B * N, V) == expect
    align = lambda x: -(-x // 256) * 256
    base = jb.jf_workspace_bytes(jb.make_shape(B, 0, 0, 0, N, 0, 8))
    ws = jb.jf_workspace_bytes(jb.make_shape(B, 0, 0, 0, N, 0, V))
    rows = B * N
    regions = lambda c: align(rows * c * 8) + align(2 * rows * c * 8)
    assert ws - base == regions(expect) - regions(1)


A16 = 1 << 20            # fake 16-byte-aligned addresses: never dereferenced


def attn(shape, ws_bytes=1 << 40, **over):
    args = dict(q=A16, k_cache=A16, v_cache=A16, prefix_lens=A16, tree_k=A16, tree_v=A16, parents=A16,
                n_nodes=A16, out=A16, workspace=A16)
    args.update(over)
    return jb.jf_tree_attention(args["q"], args["k_cache"], args["v_cache"], args["prefix_lens"], args["tree_k"],
                                args["tree_v"], args["parents"], args["n_nodes"], args["out"], shape,
                                args["workspace"], ws_bytes, status=None, stream=0, check=False)


def verify(shape, ws_bytes=1 << 40, max_depth=16, **over):
    args = dict(logits=A16, tokens=A16, parents=A16, n_nodes=A16, alen=A16, path=A16, workspace=A16)
    args.update(over)
    return jb.jf_tree_verify(args["logits"], args["tokens"], args["parents"], args["n_nodes"], args["alen"],
                             args["path"], None, shape, max_depth, args["workspace"], ws_bytes, status=None,
                             stream=0, check=False)


@pytest.mark.parametrize("name", ["q", "k_cache", "v_cache", "prefix_lens", "tree_k", "tree_v", "parents",
                                  "n_nodes", "out", "workspace"])
def test_attention_null_pointer(lib, name):
    assert attn(good_shape(), **{name: None}) == jb.JF_ERR_NULL


@pytest.mark.parametrize("bad", [dict(batch=0), dict(n_q_heads=6, n_kv_heads=4), dict(n_q_heads=12, n_kv_heads=4),
                                 dict(head_dim=96), dict(head_dim=256), dict(max_nodes=300), dict(prefix_cap=0),
                                 dict(n_kv_heads=0), dict(scale=-1.0), dict(scale=float("nan")),
                                 dict(n_q_heads=256, n_kv_heads=1)])
def test_attention_bad_shape(lib, bad):
    assert attn(good_shape(**bad)) == jb.JF_ERR_SHAPE


@pytest.mark.parametrize("name", ["q", "k_cache", "v_cache", "tree_k", "tree_v", "out"])
def test_attention_misaligned(lib, name):
    assert attn(good_shape(), **{name: A16 + 8}) == jb.JF_ERR_ALIGN


def test_attention_workspace(lib):
    s = good_shape()
    need = jb.jf_workspace_bytes(s)
    assert attn(s, ws_bytes=need - 1) == jb.JF_ERR_WORKSPACE
    assert attn(s, workspace=A16 + 128) == jb.JF_ERR_ALIGN


def test_attention_null_shape(lib):
    rc = lib.jf_tree_attention(A16, A16, A16, A16, A16, A16, A16, A16, A16, None, A16, 1 << 30, None, None)
    assert rc == jb.JF_ERR_NULL


@pytest.mark.parametrize("name", ["logits", "tokens", "parents", "n_nodes", "alen", "path", "workspace"])
def test_verify_null_pointer(lib, name):
    assert verify(good_shape(), **{name: None}) == jb.JF_ERR_NULL


@pytest.mark.parametrize("bad", [dict(vocab=0), dict(vocab=1001), dict(max_nodes=257), dict(batch=0)])
def test_verify_bad_shape(lib, bad):
    assert verify(good_shape(**bad)) == jb.JF_ERR_SHAPE


def test_verify_bad_depth_alignment_workspace(lib):
    s = good_shape()
    assert verify(s, max_depth=-1) == jb.JF_ERR_SHAPE
    assert verify(s, logits=A16 + 2) == jb.JF_ERR_ALIGN
    assert verify(s, ws_bytes=jb.jf_workspace_bytes(s) - 1) == jb.JF_ERR_WORKSPACE


def sample(shape, max_depth=16, temperature=1.0, ws_bytes=None, **over):
    args = dict(target=A16, draft=A16, tokens=A16, parents=A16, n_nodes=A16, alen=A16, path=A16, nxt=A16,
                workspace=A16 * 2)
    args.update(over)
    if ws_bytes is None:
        ws_bytes = jb.jf_workspace_bytes(shape)
    return jb.jf_tree_verify_sample(args["target"], args["draft"], args["tokens"], args["parents"], args["n_nodes"],
                                    temperature, 1, 0, args["alen"], args["path"], args["nxt"], shape, max_depth,
                                    args["workspace"], ws_bytes, stream=0, check=False)


@pytest.mark.parametrize("name", ["target", "draft", "tokens", "parents", "n_nodes", "alen", "path", "nxt",
                                  "workspace"])
def test_sample_null_pointer(lib, name):
    assert sample(good_shape(), **{name: None}) == jb.JF_ERR_NULL


@pytest.mark.parametrize("bad", [dict(vocab=0), dict(vocab=1001), dict(max_nodes=257), dict(batch=0)])
def test_sample_bad_shape(lib, bad):
    assert sample(good_shape(**bad)) == jb.JF_ERR_SHAPE


@pytest.mark.parametrize("T", [0.0, -1.0, float("nan"), float("inf")])
def test_sample_bad_temperature(lib, T):
    assert sample(good_shape(), temperature=T) == jb.JF_ERR_SHAPE


def test_sample_depth_alignment_workspace(lib):
    s = good_shape()
    assert sample(s, max_depth=-1) == jb.JF_ERR_SHAPE
    assert sample(s, target=A16 + 2) == jb.JF_ERR_ALIGN
    assert sample(s, draft=A16 + 8) == jb.JF_ERR_ALIGN
    assert sample(s, workspace=A16 + 16) == jb.JF_ERR_ALIGN
    assert sample(s, ws_bytes=jb.jf_workspace_bytes(s) - 1) == jb.JF_ERR_WORKSPACE


def commit(shape, max_depth=16, **over):
    args = dict(tree_k=A16, tree_v=A16, n_nodes=A16, alen=A16, path=A16, k_cache=A16, v_cache=A16,
                prefix_lens=A16)
    args.update(over)
    return jb.jf_tree_commit_kv(args["tree_k"], args["tree_v"], args["n_nodes"], args["alen"], args["path"],
                                args["k_cache"], args["v_cache"], args["prefix_lens"], shape, max_depth, stream=0,
                                check=False)


@pytest.mark.parametrize("name", ["tree_k", "tree_v", "n_nodes", "alen", "path", "k_cache", "v_cache",
                                  "prefix_lens"])
def test_commit_null_pointer(lib, name):
    assert commit(good_shape(), **{name: None}) == jb.JF_ERR_NULL


@pytest.mark.parametrize("bad", [dict(batch=0), dict(head_dim=96), dict(max_nodes=300), dict(prefix_cap=0),
                                 dict(n_kv_heads=0)])
def test_commit_bad_shape(lib, bad):
    assert commit(good_shape(**bad)) == jb.JF_ERR_SHAPE


@pytest.mark.parametrize("name", ["tree_k", "tree_v", "k_cache", "v_cache"])
def test_commit_misaligned_and_depth(lib, name):
    assert commit(good_shape(), **{name: A16 + 8}) == jb.JF_ERR_ALIGN
    assert commit(good_shape(), max_depth=-1) == jb.JF_ERR_SHAPE


def test_status_strings(lib):
    for code in range(6):
        assert jb.jf_status_string(code)
    assert "unknown" in jb.jf_status_string(99)


def test_trace_arm_disarm_without_gpu(lib):
    assert lib.jf_trace_kernels(None, 0) == jb.JF_OK
    assert jb.jf_trace_count() == 0
    assert jb.jf_trace_name(0) is None
    assert jb.jf_kernel_launch_count() == 0   # nothing was launched on this machine


def test_binding_refuses_strided_tensors(lib):
    """Every array is read as dense row-major memory: the binding refuses a
    tensor with other strides instead of passing its address."""
    import torch
    t = torch.zeros(4, 8, dtype=torch.bfloat16).t()
    assert not t.is_contiguous()
    with pytest.raises(ValueError):
        jb.jf_tree_verify(t, A16, A16, A16, A16, A16, None, good_shape(), 4, A16 * 2, workspace_bytes=1 << 30,
                          stream=0, check=False)


def score(shape, top_k=4, budget=8, temperature=1.0, ws_bytes=None, **over):
    args = dict(draft=A16, tokens=A16, parents=A16, n_nodes=A16, node=A16, path=A16, ttok=A16, tlp=A16,
                cpar=A16, ctok=A16, cscore=A16, workspace=A16 * 2)
    args.update(over)
    if ws_bytes is None:
        ws_bytes = jb.jf_workspace_bytes(shape)
    return jb.jf_tree_score(args["draft"], args["tokens"], args["parents"], args["n_nodes"], temperature, top_k,
                            budget, args["node"], args["path"], args["ttok"], args["tlp"], args["cpar"],
                            args["ctok"], args["cscore"], shape, args["workspace"], ws_bytes, stream=0, check=False)


@pytest.mark.parametrize("name", ["draft", "tokens", "parents", "n_nodes", "node", "path", "ttok", "tlp", "cpar",
                                  "ctok", "cscore", "workspace"])
def test_score_null_pointer(lib, name):
    assert score(good_shape(), **{name: None}) == jb.JF_ERR_NULL


def test_score_optional_outputs_may_be_null_when_unused(lib):
    # nothing to report -> the optional outputs are not needed; the call then
    # fails only at the device step on this machine (no GPU), not on NULLs
    rc = score(good_shape(), top_k=0, budget=0, ttok=None, tlp=None, cpar=None, ctok=None, cscore=None)
    assert rc not in (jb.JF_ERR_NULL, jb.JF_ERR_SHAPE, jb.JF_ERR_ALIGN, jb.JF_ERR_WORKSPACE)


@pytest.mark.parametrize("kw", [dict(top_k=-1), dict(top_k=17), dict(budget=-1), dict(top_k=0, budget=1),
                                dict(top_k=2, budget=64 * 2 + 1), dict(temperature=0.0),
                                dict(temperature=float("nan")), dict(temperature=float("inf"))])
def test_score_bad_arguments(lib, kw):
    assert score(good_shape(), **kw) == jb.JF_ERR_SHAPE


def test_score_bad_shape_alignment_workspace(lib):
    assert score(good_shape(vocab=1001)) == jb.JF_ERR_SHAPE
    assert score(good_shape(), draft=A16 + 2) == jb.JF_ERR_ALIGN
    assert score(good_shape(), workspace=A16 + 16) == jb.JF_ERR_ALIGN
    s = good_shape()
    assert score(s, ws_bytes=jb.jf_workspace_bytes(s) - 1) == jb.JF_ERR_WORKSPACE


def paged(shape, page_size=16, num_pages=64, **over):
    args = dict(q=A16, kp=A16, vp=A16, table=A16, prefix_lens=A16, tree_k=A16, tree_v=A16, parents=A16,
                n_nodes=A16, out=A16, workspace=A16 * 2)
    args.update(over)
    return jb.jf_tree_attention_paged(args["q"], args["kp"], args["vp"], args["table"], page_size, num_pages,
                                      args["prefix_lens"], args["tree_k"], args["tree_v"], args["parents"],
                                      args["n_nodes"], args["out"], shape, args["workspace"], workspace_bytes=1 << 40,
                                      stream=0, check=False)


@pytest.mark.parametrize("name", ["q", "kp", "vp", "table", "prefix_lens", "tree_k", "tree_v", "parents", "n_nodes",
                                  "out", "workspace"])
def test_paged_null_pointer(lib, name):
    assert paged(good_shape(prefix_cap=1024), **{name: None}) == jb.JF_ERR_NULL


@pytest.mark.parametrize("ps,npages,cap", [(0, 64, 1024), (12, 64, 1024), (4, 64, 1024), (256, 64, 1024),
                                           (64, 64, 1000), (16, 0, 1024)])
def test_paged_bad_geometry(lib, ps, npages, cap):
    assert paged(good_shape(prefix_cap=cap), page_size=ps, num_pages=npages) == jb.JF_ERR_SHAPE


def test_paged_misaligned(lib):
    assert paged(good_shape(prefix_cap=1024), kp=A16 + 8) == jb.JF_ERR_ALIGN


def test_paged_commit_arguments(lib):
    def call(shape, ps=16, npages=64, md=16, **over):
        args = dict(tk=A16, tv=A16, n=A16, a=A16, p=A16, kp=A16, vp=A16, t=A16, pl=A16)
        args.update(over)
        return jb.jf_tree_commit_kv_paged(args["tk"], args["tv"], args["n"], args["a"], args["p"], args["kp"],
                                          args["vp"], args["t"], ps, npages, args["pl"], shape, md, stream=0,
                                          check=False)
    s = good_shape(prefix_cap=1024)
    for name in ("tk", "tv", "n", "a", "p", "kp", "vp", "t", "pl"):
        assert call(s, **{name: None}) == jb.JF_ERR_NULL
    for ps, npages in ((12, 64), (4, 64), (256, 64), (16, 0)):
        assert call(s, ps=ps, npages=npages) == jb.JF_ERR_SHAPE
    assert call(good_shape(prefix_cap=1000), ps=64) == jb.JF_ERR_SHAPE
    assert call(s, md=-1) == jb.JF_ERR_SHAPE
    assert call(s, kp=A16 + 8) == jb.JF_ERR_ALIGN
