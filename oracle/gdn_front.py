"""Plain CPU oracle for the Gated DeltaNet layer's front end and output norm
around tree verify: the causal short convolution along each node's ancestor
path (continuing into the committed convolution tail), the q/k L2 norm, the
gates from their raw projections, and the gated RMS norm on the output; plus
the tail update a commit makes.

TEST INFRASTRUCTURE ONLY (as oracle/tree_verify.py): fp64 numpy, one
sequence per call, shares no code with the CUDA path; only tests/,
__graft_entry__.smoke() and bench.py's CPU baseline may use it.

Source (page title, section): "Adding a model", "What is still specific to
Qwen3.8": "the Gated DeltaNet layer with its gated norm"; "The model layer":
per-sequence state is the recurrent state plus the `gdn.conv` tails.  The
pages give no formula for any of these steps, so this module writes out the
plainest reading:
  * channels: the layer's raw query, key and value projections side by side,
    C = 2 * Hk * dk + Hv * dv channels per token;
  * short convolution: depthwise, causal, width W: the output of a token at
    channel c is sum_j w[c][j] * x[token - (W-1) + j][c], j = 0..W-1, over the
    token's own root path, and past the root over the committed tail (the
    last W-1 inputs of the context, oldest first); then SiLU, x * sigmoid(x);
  * q and k: divided per head by sqrt(sum of squares + eps);
  * gates: beta = sigmoid(b_raw), alpha = exp(-softplus(a_raw)) per (node,
    value head), the same distributions the pages' synthetic inputs use;
  * output: per (node, value head) o / sqrt(mean(o^2) + eps) * w_norm *
    SiLU(z), z the output gate projection, w_norm [dv];
  * commit: the tail becomes the last W-1 inputs of (old tail, accepted
    path's raw inputs).

Parity status: pinned by tests/test_oracle_gdn_front_pins.py (a chain tree
against torch.nn.functional.conv1d, identity and closed-form gate values,
unit norms, brute force against sequential decode with real tail commits,
planted mistakes).
"""
from __future__ import annotations

import numpy as np

from .tree_verify import gdn_tree_verify, root_path

EPS_NORM = 1e-6


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def softplus(x):
    x = np.asarray(x, dtype=np.float64)
    return np.logaddexp(0.0, x)


def conv_inputs(x, tail, parent, i):
    """The W inputs [W][C] the convolution of node i reads: its root path's
    raw inputs (root first), preceded by the committed tail, last W."""
    W = tail.shape[0] + 1
    path = root_path(parent, i)
    seq = np.concatenate([tail, x[path]], axis=0)
    return seq[-W:]


def short_conv_tree(x, tail, wconv, parent):
    """x [N][C] raw inputs, tail [W-1][C], wconv [C][W] -> SiLU(conv) [N][C]."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    for i in range(len(parent)):
        win = conv_inputs(x, tail, parent, i)  # [W][C]
        out[i] = silu(np.einsum("jc,cj->c", win, wconv))
    return out


def l2norm_heads(x, heads, eps=EPS_NORM):
    """x [..., heads * d]: each head's d values divided by sqrt(sum sq + eps)."""
    x = np.asarray(x, dtype=np.float64)
    sh = x.shape
    y = x.reshape(sh[:-1] + (heads, sh[-1] // heads))
    y = y / np.sqrt((y * y).sum(axis=-1, keepdims=True) + eps)
    return y.reshape(sh)


def split_channels(u, Hk, dk, Hv, dv):
    n = u.shape[0]
    q = u[:, :Hk * dk].reshape(n, Hk, dk)
    k = u[:, Hk * dk:2 * Hk * dk].reshape(n, Hk, dk)
    v = u[:, 2 * Hk * dk:].reshape(n, Hv, dv)
    return q, k, v


def gdn_front(x, tail, wconv, a_raw, b_raw, parent, Hk, dk, Hv, dv):
    """Raw projections -> (q, k, v, alpha, beta) for tv_gdn_tree_verify."""
    u = short_conv_tree(x, tail, wconv, parent)
    q, k, v = split_channels(u, Hk, dk, Hv, dv)
    q = l2norm_heads(q.reshape(len(parent), -1), Hk).reshape(q.shape)
    k = l2norm_heads(k.reshape(len(parent), -1), Hk).reshape(k.shape)
    alpha = np.exp(-softplus(a_raw))
    beta = sigmoid(b_raw)
    return q, k, v, alpha, beta


def gated_rmsnorm(o, z, w_norm, eps=EPS_NORM):
    """o, z [N][Hv][dv], w_norm [dv] -> o / rms(o) * w_norm * SiLU(z)."""
    o = np.asarray(o, dtype=np.float64)
    r = np.sqrt((o * o).mean(axis=-1, keepdims=True) + eps)
    return o / r * np.asarray(w_norm, dtype=np.float64) * silu(z)


def gdn_layer_tree_verify(S0, x, tail, wconv, a_raw, b_raw, z, w_norm, parent, Hk, dk, Hv, dv, scale):
    """The whole layer on the tree: front end, recurrence, gated norm."""
    q, k, v, alpha, beta = gdn_front(x, tail, wconv, a_raw, b_raw, parent, Hk, dk, Hv, dv)
    o = gdn_tree_verify(S0, q, k, v, alpha, beta, parent, scale)
    return gated_rmsnorm(o, z, w_norm)


def commit_tail(tail, x, path):
    """The tail after committing the accepted path's raw inputs."""
    W1 = tail.shape[0]
    seq = np.concatenate([np.asarray(tail, dtype=np.float64), np.asarray(x, dtype=np.float64)[path]], axis=0)
    return seq[-W1:].copy()
