"""Plain CPU oracle for the attention layer's front end around tree verify:
partial rotary position embedding of queries and keys at each node's logical
position, the layer's own K/V rows, and the gated output.

TEST INFRASTRUCTURE ONLY (as oracle/tree_verify.py): fp64 numpy, one
sequence per call, shares no code with the CUDA path; only tests/,
__graft_entry__.smoke() and bench.py's CPU baseline may use it.

Source (page title, section): "Adding a model", "What is still specific to
Qwen3.8": the model's attention has "a gated output and partial rotary".  The
pages give no formula for either, so this module writes out the plainest
reading:
  * rotary: the first `rot_dims` dimensions of every query and key head turn
    as rot_dims/2 planes; plane j pairs dimension j with j + rot_dims/2 and
    turns by the angle pos * theta^(-2j/rot_dims); the other dimensions pass
    through; rot_dims and theta are parameters;
  * a tree node at depth d has position L + d, the logical position decode
    would give it; the keys in the cache were rotated at their own positions
    when they were written;
  * gate: the output row is multiplied elementwise by sigmoid(gate), gate
    having the output's shape [Hq, D];
  * the layer's K/V rows (k_t, v_t) are the rotated keys and the values.

Parity status: pinned by tests/test_oracle_front_pins.py (identity and
composition properties of rotations, hand-derived angles, an independent
complex-number formulation, shift invariance of scores, the sigmoid's
closed values, and a library causal-attention cross-check on a chain).
"""
from __future__ import annotations

import numpy as np

from .tree_verify import attn_decode, attn_tree_verify, depths


def rope(x, pos, rot_dims: int, theta: float):
    """Rotate x [..., D] (any leading head axes) at integer position `pos`."""
    x = np.asarray(x, dtype=np.float64)
    if rot_dims == 0:
        return x.copy()
    half = rot_dims // 2
    j = np.arange(half, dtype=np.float64)
    angle = float(pos) * theta ** (-2.0 * j / rot_dims)
    c, s = np.cos(angle), np.sin(angle)
    out = x.copy()
    a, b = x[..., :half], x[..., half:rot_dims]
    out[..., :half] = a * c - b * s
    out[..., half:rot_dims] = b * c + a * s
    return out


def sigmoid(g):
    return 1.0 / (1.0 + np.exp(-np.asarray(g, dtype=np.float64)))


def attn_front_tree_verify(K, V, L, q_raw, k_raw, v_raw, gate, parent, scale, rot_dims, theta):
    """Tree verify of one attention layer from the projections' raw outputs.

    q_raw [N, Hq, D], k_raw, v_raw [N, Hkv, D], gate [N, Hq, D] or None;
    K, V [Hkv, cap, D] hold rotated keys for rows 0..L-1.
    Returns (out [N, Hq, D], k_t, v_t): the gated outputs and the layer's
    tree K/V rows (rotated keys, values), which a commit copies to the cache.
    """
    d = depths(parent)
    N = len(parent)
    q = np.stack([rope(q_raw[i], L + d[i], rot_dims, theta) for i in range(N)])
    k_t = np.stack([rope(k_raw[i], L + d[i], rot_dims, theta) for i in range(N)])
    v_t = np.asarray(v_raw, dtype=np.float64).copy()
    o = attn_tree_verify(K, V, L, q, k_t, v_t, parent, scale)
    if gate is not None:
        o = o * sigmoid(gate)
    return o, k_t, v_t


def attn_front_decode(K, V, L, q_raw, k_raw, v_raw, gate, scale, rot_dims, theta):
    """One decode token at position L: its rotated key and value go to cache
    row L (in place) and its gated output is returned [Hq, D]."""
    q = rope(q_raw, L, rot_dims, theta)
    k = rope(k_raw, L, rot_dims, theta)
    o = attn_decode(K, V, L, q, k, np.asarray(v_raw, dtype=np.float64), scale)
    if gate is not None:
        o = o * sigmoid(gate)
    return o
