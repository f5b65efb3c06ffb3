"""Helpers for the GPU tests: oracle evaluation of a VerifyRound's inputs and
the tolerance checks.

Tolerances (bf16 outputs: max-abs 2e-2 and rel-L2 5e-3 per layer and output
tensor; committed fp32 state: rel-L2 1e-4 per layer) are the stated targets.
For fp32 outputs (the tiny configuration) the bound is derived from fp32
arithmetic: a few hundred fp32 fused multiply-adds and the 2-ulp exp2 give
errors near 1e-6 relative, so max-abs 1e-4 and rel-L2 1e-5 leave a 10x margin.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.tree_verify as O

BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 5e-3
F32_MAX_ABS, F32_REL_L2 = 1e-4, 1e-5
STATE_REL_L2 = 1e-4


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def check_close(got: torch.Tensor, ref: np.ndarray, what: str):
    g = f64(got)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = float(np.abs(g - ref).max()) if g.size else 0.0
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    if got.dtype == torch.bfloat16:
        ok = err <= BF16_MAX_ABS and rel <= BF16_REL_L2
    else:
        ok = err <= F32_MAX_ABS and rel <= F32_REL_L2
    assert ok, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel


def check_state(got: torch.Tensor, ref: np.ndarray, what: str):
    g = f64(got)
    rel = float(np.linalg.norm(g - ref) / np.linalg.norm(ref))
    assert rel <= STATE_REL_L2, f"{what}: state rel-L2 {rel:.3e}"
    return rel


def seq_slice(r, seq):
    off = sum(r.n_nodes[:seq])
    return off, off + r.n_nodes[seq]


def oracle_attn(r, li, seq, K=None, V=None, L=None):
    """Oracle output of attention layer li for sequence seq (fp64)."""
    a = r.attn[li]
    L = int(r.cfg.ctx_lens[seq]) if L is None else L
    K = a["layer"].K[seq] if K is None else K
    V = a["layer"].V[seq] if V is None else V
    lo, hi = seq_slice(r, seq)
    return O.attn_tree_verify(f64(K[:, :L]), f64(V[:, :L]), L, f64(a["q"][lo:hi]), f64(a["k_t"][lo:hi]),
                              f64(a["v_t"][lo:hi]), r.parents[seq], r.attn_scale)


def oracle_gdn(r, li, seq, S0=None):
    g = r.gdn[li]
    lo, hi = seq_slice(r, seq)
    S0 = g["layer"].S[seq] if S0 is None else S0
    return O.gdn_tree_verify(f64(S0), f64(g["q"][lo:hi]), f64(g["k"][lo:hi]), f64(g["v"][lo:hi]),
                             f64(g["alpha"][lo:hi]), f64(g["beta"][lo:hi]), r.parents[seq], r.gdn_scale)


def oracle_commit_state(r, li, seq, S0, path):
    g = r.gdn[li]
    lo, hi = seq_slice(r, seq)
    return O.commit_gdn(f64(S0), f64(g["k"][lo:hi]), f64(g["v"][lo:hi]), f64(g["alpha"][lo:hi]),
                        f64(g["beta"][lo:hi]), path)
