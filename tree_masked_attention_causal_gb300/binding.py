"""Thin ctypes binding of libjf_tree.so (include/jf_tree.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels. The functions keep the C names and argument order.
Tensors are passed as ``data_ptr()``; the stream defaults to torch's current
CUDA stream. If the library has not been built, loading raises. There is
no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libjf_tree.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "jf_tree.h")

JF_OK, JF_ERR_NULL, JF_ERR_SHAPE, JF_ERR_ALIGN, JF_ERR_WORKSPACE, JF_ERR_CUDA = range(6)
JF_STATUS_BAD_TREE, JF_STATUS_TIMEOUT, JF_STATUS_CACHE_FULL = 1, 2, 4


class JfShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_nodes", ctypes.c_int32), ("prefix_cap", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("scale", ctypes.c_float)]


class JfError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code}: {jf_status_string(code)}")
        self.code = code


_lib = None


def open_library(path: str) -> ctypes.CDLL:
    """Open a build of the library at `path` with the argument types of
    include/jf_tree.h set (load() uses this for the package's own build)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with tree_masked_attention_causal_gb300._build.build()")
    return _configure(ctypes.CDLL(path))


def load() -> ctypes.CDLL:
    """Load libjf_tree.so from the package directory (built by _build.build())."""
    global _lib
    if _lib is None:
        _lib = open_library(LIB_PATH)
    return _lib


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    if True:
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        sp = ctypes.POINTER(JfShape)
        lib.jf_workspace_bytes.argtypes = [sp]
        lib.jf_workspace_bytes.restype = sz
        lib.jf_tree_attention.argtypes = [P, P, P, P, P, P, P, P, P, sp, P, sz, P, P]
        lib.jf_tree_attention.restype = i32
        lib.jf_tree_attention_paged.argtypes = [P, P, P, P, i32, i32, P, P, P, P, P, P, sp, P, sz, P, P]
        lib.jf_tree_attention_paged.restype = i32
        lib.jf_tree_verify.argtypes = [P, P, P, P, P, P, P, sp, i32, P, sz, P, P]
        lib.jf_tree_verify.restype = i32
        lib.jf_status_string.argtypes = [i32]
        lib.jf_status_string.restype = ctypes.c_char_p
        lib.jf_kernel_launch_count.argtypes = []
        lib.jf_kernel_launch_count.restype = ctypes.c_uint64
        lib.jf_trace_kernels.argtypes = [P, i32]
        lib.jf_trace_kernels.restype = i32
        lib.jf_trace_count.argtypes = []
        lib.jf_trace_count.restype = i32
        lib.jf_trace_name.argtypes = [i32]
        lib.jf_trace_name.restype = ctypes.c_char_p
        lib.jf_tree_verify_noalloc.argtypes = [P, P, P, P, P, P, P, sp, i32, P, P]
        lib.jf_tree_verify_noalloc.restype = i32
        lib.jf_tree_commit_kv.argtypes = [P, P, P, P, P, P, P, P, sp, i32, P, P]
        lib.jf_tree_commit_kv.restype = i32
        lib.jf_tree_commit_kv_paged.argtypes = [P, P, P, P, P, P, P, P, i32, i32, P, sp, i32, P, P]
        lib.jf_tree_commit_kv_paged.restype = i32
        u64 = ctypes.c_uint64
        lib.jf_tree_verify_sample.argtypes = [P, P, P, P, P, ctypes.c_float, u64, u64, P, P, P, sp, i32, P, sz,
                                              P, P]
        lib.jf_tree_verify_sample.restype = i32
        f32 = ctypes.c_float
        lib.jf_tree_score.argtypes = [P, P, P, P, f32, i32, i32, P, P, P, P, P, P, P, sp, P, sz, P, P]
        lib.jf_tree_score.restype = i32
    return lib


def header_symbols() -> List[str]:
    """Names of every function include/jf_tree.h declares with JF_API."""
    text = open(HEADER).read()
    return re.findall(r"JF_API\s+[\w\s\*]+?\b(jf_\w+)\s*\(", text)


def make_shape(batch, n_q_heads, n_kv_heads, head_dim, max_nodes, prefix_cap, vocab, scale=0.0) -> JfShape:
    return JfShape(batch, n_q_heads, n_kv_heads, head_dim, max_nodes, prefix_cap, vocab, scale)


def _ptr(t) -> Optional[int]:
    """The address of a tensor's first element. The library reads every
    array as dense row-major memory, so a tensor with other strides is
    refused rather than read wrongly."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("jf_tree: tensor arguments must be contiguous (row-major)")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def jf_workspace_bytes(shape: JfShape) -> int:
    return int(load().jf_workspace_bytes(ctypes.byref(shape)))


def jf_status_string(code: int) -> str:
    return load().jf_status_string(int(code)).decode()


def jf_tree_attention(q, k_cache, v_cache, prefix_lens, tree_k, tree_v, parents, n_nodes, out,
                      shape: JfShape, workspace, workspace_bytes: Optional[int] = None, status=None,
                      stream=None, check: bool = True, lib: Optional[ctypes.CDLL] = None) -> int:
    """Tree-causal attention over every node of every tree (see jf_tree.h).
    `lib` selects another build of the library (default: the package's)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = (lib or load()).jf_tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_lens), _ptr(tree_k),
                                  _ptr(tree_v), _ptr(parents), _ptr(n_nodes), _ptr(out), ctypes.byref(shape),
                                  _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_attention", rc)
    return rc


def jf_tree_attention_paged(q, k_pages, v_pages, block_table, page_size: int, num_pages: int, prefix_lens, tree_k,
                            tree_v, parents, n_nodes, out, shape: JfShape, workspace,
                            workspace_bytes: Optional[int] = None, status=None, stream=None,
                            check: bool = True) -> int:
    """Tree attention over a paged prefix cache (see jf_tree.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().jf_tree_attention_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), int(page_size),
                                        int(num_pages), _ptr(prefix_lens), _ptr(tree_k), _ptr(tree_v), _ptr(parents),
                                        _ptr(n_nodes), _ptr(out), ctypes.byref(shape), _ptr(workspace),
                                        int(workspace_bytes), _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_attention_paged", rc)
    return rc


def jf_tree_verify(logits, tree_tokens, parents, n_nodes, accept_len_out, accept_path_out, argmax_out,
                   shape: JfShape, max_depth: int, workspace, workspace_bytes: Optional[int] = None,
                   status=None, stream=None, check: bool = True) -> int:
    """Per-node argmax, then the longest accepted root path (see jf_tree.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().jf_tree_verify(_ptr(logits), _ptr(tree_tokens), _ptr(parents), _ptr(n_nodes),
                               _ptr(accept_len_out), _ptr(accept_path_out), _ptr(argmax_out),
                               ctypes.byref(shape), int(max_depth), _ptr(workspace), int(workspace_bytes),
                               _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_verify", rc)
    return rc


def jf_tree_verify_sample(target_logits, draft_logits, tree_tokens, parents, n_nodes, temperature: float,
                          seed: int, offset: int, accept_len_out, accept_path_out, next_token_out, shape: JfShape,
                          max_depth: int, workspace, workspace_bytes: Optional[int] = None, status=None,
                          stream=None, check: bool = True) -> int:
    """Stochastic tree verification by speculative sampling (see jf_tree.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().jf_tree_verify_sample(_ptr(target_logits), _ptr(draft_logits), _ptr(tree_tokens), _ptr(parents),
                                      _ptr(n_nodes), float(temperature), int(seed) & (2 ** 64 - 1),
                                      int(offset) & (2 ** 64 - 1), _ptr(accept_len_out), _ptr(accept_path_out),
                                      _ptr(next_token_out), ctypes.byref(shape), int(max_depth), _ptr(workspace),
                                      int(workspace_bytes), _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_verify_sample", rc)
    return rc


def jf_tree_score(draft_logits, tree_tokens, parents, n_nodes, temperature: float, top_k: int, budget: int,
                  node_logprob_out, path_logprob_out, topk_token_out, topk_logprob_out, cand_parent_out,
                  cand_token_out, cand_score_out, shape: JfShape, workspace, workspace_bytes: Optional[int] = None,
                  status=None, stream=None, check: bool = True) -> int:
    """Draft-side path scoring: node and path log-probabilities, each
    node's top-k tokens and the budgeted expansion (see jf_tree.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().jf_tree_score(_ptr(draft_logits), _ptr(tree_tokens), _ptr(parents), _ptr(n_nodes),
                              float(temperature), int(top_k), int(budget), _ptr(node_logprob_out),
                              _ptr(path_logprob_out), _ptr(topk_token_out), _ptr(topk_logprob_out),
                              _ptr(cand_parent_out), _ptr(cand_token_out), _ptr(cand_score_out), ctypes.byref(shape),
                              _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_score", rc)
    return rc


def jf_tree_commit_kv(tree_k, tree_v, n_nodes, accept_len, accept_path, k_cache, v_cache, prefix_lens,
                      shape: JfShape, max_depth: int, status=None, stream=None, check: bool = True) -> int:
    """Append each sequence's accepted path to its KV cache (see jf_tree.h)."""
    rc = load().jf_tree_commit_kv(_ptr(tree_k), _ptr(tree_v), _ptr(n_nodes), _ptr(accept_len), _ptr(accept_path),
                                  _ptr(k_cache), _ptr(v_cache), _ptr(prefix_lens), ctypes.byref(shape),
                                  int(max_depth), _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_commit_kv", rc)
    return rc


def jf_tree_commit_kv_paged(tree_k, tree_v, n_nodes, accept_len, accept_path, k_pages, v_pages, block_table,
                            page_size: int, num_pages: int, prefix_lens, shape: JfShape, max_depth: int, status=None,
                            stream=None, check: bool = True) -> int:
    """Append each sequence's accepted path to its paged KV cache (see jf_tree.h)."""
    rc = load().jf_tree_commit_kv_paged(_ptr(tree_k), _ptr(tree_v), _ptr(n_nodes), _ptr(accept_len),
                                        _ptr(accept_path), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                        int(page_size), int(num_pages), _ptr(prefix_lens), ctypes.byref(shape),
                                        int(max_depth), _ptr(status), _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_commit_kv_paged", rc)
    return rc


def jf_kernel_launch_count() -> int:
    return int(load().jf_kernel_launch_count())


def jf_trace_kernels(events, capacity: int) -> int:
    """Arm per-kernel timing with a list of 2*capacity torch.cuda.Event
    objects (enable_timing=True); pass None / 0 to disarm. The handle array
    is kept alive by this module while armed."""
    global _trace_keep
    if not events or capacity <= 0:
        _trace_keep = None
        return load().jf_trace_kernels(None, 0)
    evs = events[: 2 * capacity]
    if any(not e.cuda_event for e in evs):
        import torch
        for e in evs:              # torch creates the CUDA event lazily, on first record
            if not e.cuda_event:
                e.record()
        torch.cuda.synchronize()
    arr = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in evs])
    _trace_keep = arr
    return load().jf_trace_kernels(ctypes.cast(arr, ctypes.c_void_p), capacity)


_trace_keep = None


def jf_trace_count() -> int:
    return int(load().jf_trace_count())


def jf_trace_name(k: int) -> Optional[str]:
    r = load().jf_trace_name(int(k))
    return None if r is None else r.decode()


def jf_tree_verify_noalloc(logits, tree_tokens, parents, n_nodes, accept_len_out, accept_path_out, argmax_out,
                           shape: JfShape, max_depth: int, status=None, stream=None, check: bool = True) -> int:
    """jf_tree_verify without a workspace, for callers that cannot allocate
    device memory: the scratch is a fixed array inside the library (see
    jf_tree.h for its size limit and for when calls race)."""
    fn = load().jf_tree_verify_noalloc
    rc = fn(_ptr(logits), _ptr(tree_tokens), _ptr(parents), _ptr(n_nodes), _ptr(accept_len_out),
            _ptr(accept_path_out), _ptr(argmax_out), ctypes.byref(shape), int(max_depth), _ptr(status),
            _stream(stream))
    if check and rc != JF_OK:
        raise JfError("jf_tree_verify_noalloc", rc)
    return rc
