"""fp64 CPU oracle for tree-causal attention and greedy tree verification.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The product path
(``tree_masked_attention_causal_gb300``) never does, and this package
imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, OpenMP over rows). This module
compiles it with gcc on first use and wraps it with ctypes and numpy.

Parity pins: see the header of ``oracle.c``. Every function here is pinned
by a test under ``tests/test_oracle_pins.py`` that checks it against
something other than itself.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_tree_attention_f64.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                      i32, i32, f64, P, i64, P]
            lib.oracle_tree_attention_f64.restype = None
            lib.oracle_argmax_rows.argtypes = [P, i64, i64, P]
            lib.oracle_argmax_rows.restype = None
            lib.oracle_tree_verify.argtypes = [P, P, P, P, i32, i32, i64, i32, P, P, P]
            lib.oracle_tree_verify.restype = None
            lib.oracle_tree_is_valid.argtypes = [P, i32, i32]
            lib.oracle_tree_is_valid.restype = ctypes.c_int
            lib.oracle_commit_kv.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
            lib.oracle_commit_kv.restype = None
            u64 = ctypes.c_uint64
            lib.oracle_philox4x64_10.argtypes = [P, P, P]
            lib.oracle_philox4x64_10.restype = None
            lib.oracle_uniform.argtypes = [u64, u64, ctypes.c_uint32, i32, i64]
            lib.oracle_uniform.restype = f64
            lib.oracle_tree_verify_sample.argtypes = [P, P, P, P, P, i32, i32, i64, i32, f64, u64, u64,
                                                      P, P, P, P]
            lib.oracle_tree_verify_sample.restype = None
            lib.oracle_tree_score.argtypes = [P, P, P, P, i32, i32, i64, f64, i32, i32, P, P, P, P, P, P, P, P]
            lib.oracle_tree_score.restype = None
            lib.oracle_commit_kv_paged.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, P, i32, i32, i32, i32, i32, P]
            lib.oracle_commit_kv_paged.restype = None
            _lib = lib
    return _lib


def _u16(t) -> np.ndarray:
    """Raw bf16 bits of a CPU torch bf16 tensor (or a uint16 ndarray)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(t) -> np.ndarray:
    a = t if isinstance(t, np.ndarray) else t.numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    return int(env) if env else (os.cpu_count() or 1)


def tree_attention(q, k_cache, v_cache, prefix_lens, tree_k, tree_v, parents, n_nodes,
                   scale: float = 0.0, sel=None, out: np.ndarray | None = None) -> np.ndarray:
    """fp64 tree attention. Returns out [B, Nmax, Hq, d] (float64); rows
    not computed (padded nodes, or rows outside ``sel``) stay NaN unless an
    ``out`` buffer is passed. ``sel`` is an (n, 2) array of (b, i) pairs."""
    lib = _load()
    B, N, Hq, d = q.shape
    Hkv, Pcap = k_cache.shape[1], k_cache.shape[2]
    qa, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    tk, tv = _u16(tree_k), _u16(tree_v)
    pl, par, nn = _i32(prefix_lens), _i32(parents), _i32(n_nodes)
    if out is None:
        out = np.full((B, N, Hq, d), np.nan, dtype=np.float64)
    sel_a = None if sel is None else np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
    lib.oracle_tree_attention_f64(_ptr(qa), _ptr(kc), _ptr(vc), _ptr(pl), _ptr(tk), _ptr(tv),
                                  _ptr(par), _ptr(nn), B, N, Hq, Hkv, d, Pcap, float(scale),
                                  None if sel_a is None else _ptr(sel_a),
                                  0 if sel_a is None else sel_a.shape[0], _ptr(out))
    return out


def argmax_rows(logits) -> np.ndarray:
    """First-max argmax of each row of a [..., V] bf16 tensor (int32)."""
    lib = _load()
    a = _u16(logits)
    V = a.shape[-1]
    rows = a.size // V
    out = np.empty(rows, dtype=np.int32)
    lib.oracle_argmax_rows(_ptr(a), rows, V, _ptr(out))
    return out.reshape(a.shape[:-1])


def tree_verify(logits, tokens, parents, n_nodes, max_depth: int):
    """Greedy verification. Returns (accept_len [B], accept_path [B, max_depth+1],
    argmax [B, Nmax]) as int32 arrays."""
    lib = _load()
    lg = _u16(logits)
    B, N, V = lg.shape
    tok, par, nn = _i32(tokens), _i32(parents), _i32(n_nodes)
    alen = np.empty(B, dtype=np.int32)
    path = np.empty((B, max_depth + 1), dtype=np.int32)
    am = np.empty((B, N), dtype=np.int32)
    lib.oracle_tree_verify(_ptr(lg), _ptr(tok), _ptr(par), _ptr(nn), B, N, V, max_depth,
                           _ptr(alen), _ptr(path), _ptr(am))
    return alen, path, am


def tree_is_valid(parents_row, n: int, max_nodes: int) -> bool:
    lib = _load()
    p = _i32(np.asarray(parents_row))
    return bool(lib.oracle_tree_is_valid(_ptr(p), int(n), int(max_nodes)))


def commit_kv(tree_k, tree_v, n_nodes, accept_len, accept_path, k_cache, v_cache, prefix_lens, max_depth: int):
    """Accepted-path KV commit. Returns (k_cache, v_cache, prefix_lens, flags)
    as new arrays (bf16 bits as uint16, int32); the inputs are not modified.
    flags[b]: 0 done (or nothing to do), 1 malformed request, 2 no room."""
    lib = _load()
    tk, tv = _u16(tree_k), _u16(tree_v)
    kc, vc = _u16(k_cache).copy(), _u16(v_cache).copy()
    B, Nmax, Hkv, d = tk.shape
    Pcap = kc.shape[2]
    nn, al, ap = _i32(n_nodes), _i32(accept_len), _i32(accept_path)
    pl = _i32(prefix_lens).copy()
    flags = np.zeros(B, dtype=np.int32)
    lib.oracle_commit_kv(_ptr(tk), _ptr(tv), _ptr(nn), _ptr(al), _ptr(ap), _ptr(kc), _ptr(vc), _ptr(pl),
                         B, Nmax, Hkv, d, Pcap, int(max_depth), _ptr(flags))
    return kc, vc, pl, flags


def philox4x64_10(counter, key) -> np.ndarray:
    """One Philox4x64-10 block: 4 uint64 words for a 4-word counter and a
    2-word key."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64).reshape(2))
    out = np.empty(4, dtype=np.uint64)
    _load().oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, offset: int, purpose: int, b: int, index: int) -> float:
    """The uniform in (0, 1) of stream `purpose` (0: acceptance, 1: sampling)
    for sequence b and item `index`."""
    return float(_load().oracle_uniform(seed, offset, purpose, b, index))


def tree_verify_sample(target_logits, draft_logits, tokens, parents, n_nodes, max_depth: int,
                       temperature: float, seed: int, offset: int):
    """Stochastic tree verification. Returns (accept_len [B], accept_path
    [B, max_depth+1], next_token [B], margins [B, 3]) where margins holds
    the smallest acceptance-test margin, the smallest residual mass and the
    Gumbel top-2 gap of each sequence."""
    lib = _load()
    tg, dr = _u16(target_logits), _u16(draft_logits)
    B, N, V = tg.shape
    assert dr.shape == tg.shape
    tok, par, nn = _i32(tokens), _i32(parents), _i32(n_nodes)
    alen = np.empty(B, dtype=np.int32)
    path = np.empty((B, max_depth + 1), dtype=np.int32)
    nxt = np.empty(B, dtype=np.int32)
    margins = np.empty((B, 3), dtype=np.float64)
    lib.oracle_tree_verify_sample(_ptr(tg), _ptr(dr), _ptr(tok), _ptr(par), _ptr(nn), B, N, V, max_depth,
                                  float(temperature), int(seed), int(offset), _ptr(alen), _ptr(path),
                                  _ptr(nxt), _ptr(margins))
    return alen, path, nxt, margins


def tree_score(draft_logits, tokens, parents, n_nodes, temperature: float, top_k: int = 0, budget: int = 0):
    """Draft-side path scoring. Returns a dict with node_lp, path_lp [B, N]
    (float64), topk_tok [B, N, top_k] (int32), topk_lp [B, N, top_k],
    cand_parent, cand_token [B, budget] (int32), cand_score [B, budget] and
    gaps [B] (the smallest score gap in and around each selection)."""
    lib = _load()
    dr = _u16(draft_logits)
    B, N, V = dr.shape
    tok, par, nn = _i32(tokens), _i32(parents), _i32(n_nodes)
    k = max(0, int(top_k))
    bud = max(0, int(budget))
    out = dict(node_lp=np.empty((B, N)), path_lp=np.empty((B, N)),
               topk_tok=np.empty((B, N, max(k, 1)), dtype=np.int32), topk_lp=np.empty((B, N, max(k, 1))),
               cand_parent=np.empty((B, max(bud, 1)), dtype=np.int32),
               cand_token=np.empty((B, max(bud, 1)), dtype=np.int32), cand_score=np.empty((B, max(bud, 1))),
               gaps=np.empty(B))
    lib.oracle_tree_score(_ptr(dr), _ptr(tok), _ptr(par), _ptr(nn), B, N, V, float(temperature), k, bud,
                          _ptr(out["node_lp"]), _ptr(out["path_lp"]), _ptr(out["topk_tok"]), _ptr(out["topk_lp"]),
                          _ptr(out["cand_parent"]), _ptr(out["cand_token"]), _ptr(out["cand_score"]),
                          _ptr(out["gaps"]))
    out["topk_tok"], out["topk_lp"] = out["topk_tok"][:, :, :k], out["topk_lp"][:, :, :k]
    for key in ("cand_parent", "cand_token", "cand_score"):
        out[key] = out[key][:, :bud]
    return out


def gather_pages(pages, block_table, prefix_lens, page_size: int, prefix_cap: int) -> np.ndarray:
    """A paged cache [num_pages, page_size, Hkv, d] (bf16 bits) as the
    contiguous [B, Hkv, prefix_cap, d] cache it stands for: row p of
    sequence b, head h is pages[block_table[b, p // page_size], p % page_size,
    h]. Rows at or past prefix_lens[b] are left 0 (never attended)."""
    pg = _u16(pages)
    tab = _i32(block_table)
    pl = _i32(prefix_lens)
    B = tab.shape[0]
    Hkv, d = pg.shape[2], pg.shape[3]
    out = np.zeros((B, Hkv, prefix_cap, d), dtype=np.uint16)
    for b in range(B):
        for p in range(int(pl[b])):
            out[b, :, p, :] = pg[tab[b, p // page_size], p % page_size, :, :]
    return out


def tree_attention_paged(q, k_pages, v_pages, block_table, page_size: int, prefix_cap: int, prefix_lens, tree_k,
                         tree_v, parents, n_nodes, scale: float = 0.0, sel=None) -> np.ndarray:
    """Tree attention over a paged prefix cache: the pages gathered into the
    contiguous cache they stand for, then tree_attention."""
    kc = gather_pages(k_pages, block_table, prefix_lens, page_size, prefix_cap)
    vc = gather_pages(v_pages, block_table, prefix_lens, page_size, prefix_cap)
    return tree_attention(q, kc, vc, prefix_lens, tree_k, tree_v, parents, n_nodes, scale=scale, sel=sel)


def commit_kv_paged(tree_k, tree_v, n_nodes, accept_len, accept_path, k_pages, v_pages, block_table,
                    page_size: int, prefix_lens, max_depth: int):
    """The KV commit into a paged cache. Returns (k_pages, v_pages) as
    updated uint16 copies, prefix_lens and flags (int32)."""
    lib = _load()
    tk, tv = _u16(tree_k), _u16(tree_v)
    B, N, Hkv, d = tk.shape
    kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
    tab = _i32(block_table)
    pl = _i32(prefix_lens).copy()
    flags = np.empty(B, dtype=np.int32)
    lib.oracle_commit_kv_paged(_ptr(tk), _ptr(tv), _ptr(_i32(n_nodes)), _ptr(_i32(accept_len)),
                               _ptr(_i32(accept_path)), _ptr(kp), _ptr(vp), _ptr(tab), int(page_size), kp.shape[0],
                               tab.shape[1], _ptr(pl), B, N, Hkv, d, int(max_depth), _ptr(flags))
    return kp, vp, pl, flags
