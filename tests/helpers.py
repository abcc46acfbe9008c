"""Helpers shared by the GPU tests: run the C-ABI entry points on seeded
inputs and compare them with the fp64 oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from tree_masked_attention_causal_gb300 import _build, binding as jb, synth

# Tolerance on unit-variance bf16 inputs, against the fp64 oracle.
ATOL_MAX = 1e-2
ATOL_MEAN = 1e-3
SENTINEL = 0x3C1D      # bf16 bits written into `out` before a call (~0.0095)
CANARY = 4096          # bf16 elements of guard zone on each side of `out`


def lib():
    _build.build()
    return jb.load()


def shape_of(inp, scale=0.0):
    w = inp["workload"]
    q = inp["q"]
    B, N, Hq, d = q.shape
    return jb.make_shape(B, Hq, inp["k_cache"].shape[1], d, N, inp["k_cache"].shape[2],
                         inp["logits"].shape[-1] if "logits" in inp else w.vocab, scale)


def to_dev(inp, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def new_workspace(shape, device="cuda"):
    n = jb.jf_workspace_bytes(shape)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device=device)


def run_attention(dev, shape, ws=None, status=None):
    """Call jf_tree_attention; returns (out [B,N,Hq,d] bf16 on device with
    guard zones checked, status value)."""
    B, N, Hq, d = dev["q"].shape
    n_out = B * N * Hq * d
    buf = torch.full((n_out + 2 * CANARY,), 0, dtype=torch.int16, device=dev["q"].device)
    buf.fill_(SENTINEL)
    out = buf[CANARY:CANARY + n_out].view(torch.bfloat16).view(B, N, Hq, d)
    if ws is None:
        ws = new_workspace(shape)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev["q"].device)
    jb.jf_tree_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["prefix_lens"], dev["tree_k"], dev["tree_v"],
                         dev["parents"], dev["n_nodes"], out, shape, ws, status=status)
    torch.cuda.synchronize()
    guard = torch.cat([buf[:CANARY], buf[CANARY + n_out:]])
    assert bool((guard == SENTINEL).all()), "write outside `out`"
    return out, int(status.item())


def run_verify(dev, shape, max_depth=16, ws=None):
    B, N = dev["tokens"].shape
    d = dev["tokens"].device
    alen = torch.full((B,), -7, dtype=torch.int32, device=d)
    path = torch.full((B, max_depth + 1), -7, dtype=torch.int32, device=d)
    am = torch.full((B, N), -7, dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    if ws is None:
        ws = new_workspace(shape)
    jb.jf_tree_verify(dev["logits"], dev["tokens"], dev["parents"], dev["n_nodes"], alen, path, am, shape,
                      max_depth, ws, status=status)
    torch.cuda.synchronize()
    return alen.cpu().numpy(), path.cpu().numpy(), am.cpu().numpy(), int(status.item())


def oracle_attention(inp, scale=0.0, sel=None):
    return oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["prefix_lens"], inp["tree_k"],
                                 inp["tree_v"], inp["parents"], inp["n_nodes"], scale=scale, sel=sel)


def valid_rows(inp):
    rows = []
    for b in range(inp["q"].shape[0]):
        for i in range(int(inp["n_nodes"][b])):
            rows.append((b, i))
    return rows


def half_ulp_bf16(x):
    """Half a bf16 ulp at |x|: the representation error of the bf16 output
    format (7 stored mantissa bits), 2^(floor(log2|x|) - 8)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


# (what, max-abs error, mean-abs error, elements that needed the half-ulp
# allowance) of every comparison in this process; printed at the end of a
# run with JF_PARITY_REPORT=1 (tests/conftest.py).
REPORT = []


def assert_attention_close(got, ref, rows, what="", strict=False):
    """Element-wise comparison on the given (b, i) rows (all heads, all d).

    The bound is max-abs 1e-2 and mean-abs 1e-3 against fp64. The output is
    bf16 by contract: where |ref| >= 1, bf16's half-ulp alone (0.0039 and
    up) takes a large part of that budget, on top of the bf16 rounding of
    the attention weights that feed the PV product (few keys: it does not
    average out). So unless `strict`, those elements (and only those) may
    also differ by half a bf16 ulp of their reference value. Rows that see
    few keys reach such magnitudes; the five workloads stay far below and
    run strict.
    """
    g = np.stack([got[b, i] for b, i in rows]).astype(np.float64)
    r = np.stack([ref[b, i] for b, i in rows])
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = ATOL_MAX if strict else ATOL_MAX + np.where(np.abs(r) >= 1.0, half_ulp_bf16(r), 0.0)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{what}: |err| {err[worst]:.3e} > bound {np.broadcast_to(bound, err.shape)[worst]:.3e}"
                                  f" at row {rows[worst[0]]}, head {worst[1]}, d {worst[2]} (ref {r[worst]:.4f})")
    assert err.mean() <= ATOL_MEAN, f"{what}: mean-abs {err.mean():.3e} > {ATOL_MEAN}"
    REPORT.append((what, float(err.max()), float(err.mean()), int((err > ATOL_MAX).sum())))
    return float(err.max()), float(err.mean())


def padding_untouched(out_cpu_bits, inp):
    """Rows of padding nodes must still hold the sentinel."""
    for b in range(out_cpu_bits.shape[0]):
        n = int(inp["n_nodes"][b])
        if n < out_cpu_bits.shape[1]:
            if not bool((out_cpu_bits[b, n:] == SENTINEL).all()):
                return False
    return True


def out_bits(out):
    return out.view(torch.int16).cpu()


def out_f64(out):
    return out.float().cpu().double().numpy()


def small_inputs(seed, B=2, N=20, Hq=8, Hkv=2, d=64, Pcap=200, prefixes=None, parents=None, n_nodes=None,
                 vocab=256, kv_fill=0.0):
    """Hand-shaped inputs for edge cases (no planted path)."""
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    if parents is None:
        parents = torch.tensor([synth.random_tree(g, N, 8, None) for _ in range(B)], dtype=torch.int32)
    if prefixes is None:
        prefixes = torch.randint(0, Pcap + 1, (B,), generator=g, dtype=torch.int32)
    if n_nodes is None:
        n_nodes = torch.full((B,), N, dtype=torch.int32)
    kc = torch.full((B, Hkv, Pcap, d), kv_fill, dtype=torch.bfloat16)
    vc = torch.full((B, Hkv, Pcap, d), kv_fill, dtype=torch.bfloat16)
    for b in range(B):
        P = int(prefixes[b])
        kc[b, :, :P] = bf(Hkv, P, d)
        vc[b, :, :P] = bf(Hkv, P, d)
    w = synth.Workload("edge", B, Hq, Hkv, d, N, 0, Pcap, Pcap, vocab, 8, None, 1, 1, seed)
    tokens = torch.randint(0, vocab, (B, N), generator=g, dtype=torch.int32)
    logits = torch.randn(B, N, vocab, generator=g).clamp(-8, 8).to(torch.bfloat16)
    return dict(workload=w, q=bf(B, N, Hq, d), k_cache=kc, v_cache=vc, tree_k=bf(B, N, Hkv, d),
                tree_v=bf(B, N, Hkv, d), prefix_lens=prefixes.to(torch.int32), parents=parents.to(torch.int32),
                n_nodes=n_nodes.to(torch.int32), tokens=tokens, logits=logits)
