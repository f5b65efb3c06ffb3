"""Plain CPU oracle for one speculative tree-verify round of a hybrid
Gated DeltaNet + attention mixer stack.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct fp64
definition that the CUDA path is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import it; the library itself never calls it and has no CPU fallback.

It shares no code with the CUDA path.  Every function takes numpy arrays that
the caller has already converted to float64 (bf16 inputs upcast exactly) and
works on ONE sequence.

Sources (page title, section):
  * "One request, end to end", section 2.6 "The decode loop": one forward pass
    verifies the whole draft tree; the walk keeps the longest agreeing path
    plus one token of the model's own; that path's KV rows and recurrent state
    are committed.
  * "Adding a model", step 4 (hot verbs forward_tree / commit_tree /
    rollback_to): every verified row must equal the decode step's row.
  * "Adding a model", "What is still specific to Qwen3.8": Gated DeltaNet
    layers (heads of 128 by 128) and attention layers.
  * The gated delta rule itself, S_t = a_t S_{t-1} (I - b_t k_t k_t^T)
    + b_t v_t k_t^T, and the ancestor-bitmask tree mask are taken as the
    method's definition (they are not printed on the pages).

Readings where the pages are silent:
  * node 0 is the root = the last committed token, not yet in the cache or in
    the state; a node at depth d sees the L context rows plus its d+1
    ancestors-or-self, placed at logical positions L..L+d;
  * query head h reads KV head h // (Hq // Hkv); value head h reads key head
    h // (Hv // Hk);
  * attention scale and GDN output scale are arguments (default D^-1/2, dk^-1/2);
  * the accepted path is the longest root path on which every node's token
    equals the target's greedy token at its parent (ties: lowest end node);
    the bonus token is the greedy token at the path's last node.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(brute force against sequential decode, an independent chunked closed form,
closed-form special cases, a library causal-attention cross-check and
hand-derived values in tests/golden/).
"""
from __future__ import annotations

import numpy as np

MAX_NODES = 64
MAX_PATH = 16  # nodes on a root path, root included


# ---------------------------------------------------------------------------
# tree structure
# ---------------------------------------------------------------------------
def check_parent(parent) -> None:
    """A tree is a parent-index array in topological order: parent[0] = -1,
    0 <= parent[i] < i for i >= 1, at most 64 nodes, at most 16 nodes on a
    root path."""
    parent = [int(p) for p in parent]
    n = len(parent)
    if n < 1 or n > MAX_NODES:
        raise ValueError(f"tree must have 1..{MAX_NODES} nodes, got {n}")
    if parent[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, n):
        if not (0 <= parent[i] < i):
            raise ValueError(f"parent[{i}] = {parent[i]} is not an earlier node")
    if max(len(root_path(parent, i)) for i in range(n)) > MAX_PATH:
        raise ValueError(f"a root path is longer than {MAX_PATH} nodes")


def root_path(parent, i: int) -> list[int]:
    """Nodes from the root to node i, inclusive (the ancestors-or-self of i
    ordered by depth)."""
    path = []
    while i != -1:
        path.append(int(i))
        i = int(parent[i])
    return path[::-1]


def depths(parent) -> list[int]:
    return [len(root_path(parent, i)) - 1 for i in range(len(parent))]


# ---------------------------------------------------------------------------
# attention (tree-masked grouped-query attention over the KV cache)
# ---------------------------------------------------------------------------
def attn_tree_verify(K, V, L, q, k_t, v_t, parent, scale):
    """Output of every tree node for one attention layer.

    K, V   : [Hkv, cap, D] committed cache; rows 0..L-1 are the context.
    q      : [N, Hq, D] queries of the N tree nodes.
    k_t,v_t: [N, Hkv, D] keys / values of the tree nodes themselves.
    Returns o [N, Hq, D]:
        o[i, h] = sum_p softmax_p(scale * q[i,h] . key_p) value_p
    over the visible positions p = the L context rows and the
    ancestors-or-self of i.
    """
    N, Hq, D = q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    o = np.zeros((N, Hq, D), dtype=np.float64)
    for g in range(Hkv):
        ctx_k = K[g, :L]
        ctx_v = V[g, :L]
        heads = list(range(g * G, (g + 1) * G))
        # scores against the context, every node and head of this group at once
        s_ctx = (q[:, heads] @ ctx_k.T) * scale  # [N, G, L]
        w_ctx = np.empty_like(s_ctx)
        for i in range(N):
            path = root_path(parent, i)
            tree_k = k_t[path, g]  # [d+1, D]
            tree_v = v_t[path, g]
            s = np.concatenate([s_ctx[i], (q[i, heads] @ tree_k.T) * scale], axis=1)  # [G, L+d+1]
            w = np.exp(s - s.max(axis=1, keepdims=True))
            w /= w.sum(axis=1, keepdims=True)
            w_ctx[i] = w[:, :L]
            o[i, heads] = w[:, L:] @ tree_v
        # the context part of every weighted sum, as one matrix product
        o[:, heads] += w_ctx @ ctx_v
    return o


def attn_decode(K, V, L, q, k, v, scale):
    """One decode token (no tree): append k, v at row L of the cache (in
    place) and attend over rows 0..L.  q: [Hq, D], k, v: [Hkv, D].
    Returns o [Hq, D].  The caller advances L."""
    Hq, D = q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    K[:, L] = k
    V[:, L] = v
    o = np.zeros((Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // G
        s = (K[g, : L + 1] @ q[h]) * scale
        w = np.exp(s - s.max())
        w /= w.sum()
        o[h] = w @ V[g, : L + 1]
    return o


# ---------------------------------------------------------------------------
# Gated DeltaNet (gated delta rule along each node's root path)
# ---------------------------------------------------------------------------
def gdn_step(S, q, k, v, alpha, beta):
    """One token of the gated delta rule for every value head, written as the
    definition: S <- alpha * S (I - beta k k^T) + beta v k^T.

    S: [Hv, dv, dk]; k: [Hv, dk] (key of each value head's key head);
    v: [Hv, dv]; alpha, beta: [Hv].  Returns the new state."""
    Hv, dv, dk = S.shape
    eye = np.eye(dk)
    out = np.empty_like(S)
    for h in range(Hv):
        kk = np.outer(k[h], k[h])
        out[h] = alpha[h] * S[h] @ (eye - beta[h] * kk) + beta[h] * np.outer(v[h], k[h])
    return out


def _per_value_head(x, Hv):
    """Broadcast a per-key-head vector [Hk, d] to value heads [Hv, d]:
    value head h reads key head h // (Hv // Hk)."""
    Hk = x.shape[0]
    return np.repeat(x, Hv // Hk, axis=0)


def gdn_tree_verify(S0, q, k, v, alpha, beta, parent, scale):
    """Output of every tree node for one Gated DeltaNet layer, by replaying
    the recurrence along each node's root path from the committed state S0.

    S0: [Hv, dv, dk]; q, k: [N, Hk, dk]; v: [N, Hv, dv]; alpha, beta: [N, Hv].
    Returns o [N, Hv, dv] with o[i, h] = scale * S_i[h] q_i (q of h's key head).
    """
    N = q.shape[0]
    Hv = S0.shape[0]
    o = np.zeros((N, Hv, S0.shape[1]), dtype=np.float64)
    for i in range(N):
        S = S0.copy()
        for j in root_path(parent, i):
            S = gdn_step(S, None, _per_value_head(k[j], Hv), v[j], alpha[j], beta[j])
        qh = _per_value_head(q[i], Hv)
        o[i] = scale * np.einsum("hvk,hk->hv", S, qh)
    return o


def gdn_path_state(S0, k, v, alpha, beta, path):
    """State after the tokens of `path` (node indices, in order) from S0."""
    Hv = S0.shape[0]
    S = S0.copy()
    for j in path:
        S = gdn_step(S, None, _per_value_head(k[j], Hv), v[j], alpha[j], beta[j])
    return S


def gdn_decode(S, q, k, v, alpha, beta, scale):
    """One decode token: S <- step(S) in place; returns o = scale * S q.
    q, k: [Hk, dk]; v: [Hv, dv]; alpha, beta: [Hv]."""
    Hv = S.shape[0]
    S[:] = gdn_step(S, None, _per_value_head(k, Hv), v, alpha, beta)
    return scale * np.einsum("hvk,hk->hv", S, _per_value_head(q, Hv))


def gdn_tree_chunked(S0, q, k, v, alpha, beta, parent, scale):
    """Independent closed form of gdn_tree_verify (the tree-masked UT / WY
    form of the delta rule).  With gamma_i the product of alpha over the
    ancestors-or-self of i, and for every node i

        u_i + sum_{j strict ancestor of i} beta_i (gamma_i / gamma_j) (k_i.k_j) u_j
            = beta_i (v_i - gamma_i S0 k_i)

    the output is o_i = scale (gamma_i S0 q_i
                               + sum_{j in anc*(i)} (gamma_i / gamma_j) (k_j.q_i) u_j).
    Solved as one lower-triangular system per value head."""
    N = q.shape[0]
    Hv, dv, dk = S0.shape
    paths = [root_path(parent, i) for i in range(N)]
    o = np.zeros((N, Hv, dv), dtype=np.float64)
    for h in range(Hv):
        g = h // (Hv // k.shape[1])
        kh = k[:, g]  # [N, dk]
        qh = q[:, g]
        gam = np.array([np.prod(alpha[p, h]) for p in paths])
        A = np.zeros((N, N))
        for i in range(N):
            for j in paths[i][:-1]:
                A[i, j] = beta[i, h] * (gam[i] / gam[j]) * (kh[i] @ kh[j])
        rhs = beta[:, h, None] * (v[:, h] - gam[:, None] * (kh @ S0[h].T))
        U = np.linalg.solve(np.eye(N) + A, rhs)  # [N, dv]
        for i in range(N):
            acc = gam[i] * (S0[h] @ qh[i])
            for j in paths[i]:
                acc = acc + (gam[i] / gam[j]) * (kh[j] @ qh[i]) * U[j]
            o[i, h] = scale * acc
    return o


# ---------------------------------------------------------------------------
# accept walk and commit
# ---------------------------------------------------------------------------
def accept_path(parent, tok, greedy):
    """Longest agreeing path plus one token.

    A node agrees when every node on its root path below the root carries the
    token the target chose (greedily) at that node's parent.  The accepted
    path is the root path of the deepest agreeing node (lowest index among
    equally deep ones); the bonus token is the greedy token at its end.
    Returns (path, a, bonus) with a = len(path) >= 1."""
    N = len(parent)
    agree = [False] * N
    agree[0] = True
    for i in range(1, N):
        p = int(parent[i])
        agree[i] = agree[p] and int(tok[i]) == int(greedy[p])
    dep = depths(parent)
    best = 0
    for i in range(N):
        if agree[i] and dep[i] > dep[best]:
            best = i
    path = root_path(parent, best)
    return path, len(path), int(greedy[best])


def commit_attn(K, V, L, k_t, v_t, path):
    """Write the accepted path's K/V rows at cache rows L..L+a-1 (in place)."""
    for j, node in enumerate(path):
        K[:, L + j] = k_t[node]
        V[:, L + j] = v_t[node]
    return L + len(path)


def commit_gdn(S0, k, v, alpha, beta, path):
    """The committed recurrent state: S0 advanced along the accepted path."""
    return gdn_path_state(S0, k, v, alpha, beta, path)
