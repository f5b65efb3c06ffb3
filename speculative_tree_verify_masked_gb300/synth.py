"""Seeded synthetic inputs for the verify round (trees, tokens, per-layer
tensors).  Shared by the tests, the benchmark and the oracle checks; holds none
of the method's arithmetic.

Value distributions (every configuration):
  * attention q, k, v and cache rows ~ N(0, 1);
  * Gated DeltaNet q, k ~ N(0, 1), then L2-normalised per head (the model does
    this before the mixer, so it is an input property here); v ~ N(0, 1);
    beta = sigmoid(N(0, 1)); alpha = exp(-softplus(N(0, 1)));
    initial state ~ N(0, 0.1^2);
  * tokens uniform in [0, 65536) with distinct siblings; greedy tokens set so
    the accept walk follows a chosen root path and stops at its end.
Seeds: layer tensors use 1_000_000*c + 1_000*seq + layer; trees and tokens use
1_000_000*c + 999_000 + seq, with a fixed draw order.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

VOCAB = 65536


# ---------------------------------------------------------------------------
# workload shapes
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Shapes:
    Hq: int
    Hkv: int
    D: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    kv_dtype: torch.dtype  # dtype of cache, q/k/v and outputs


SHAPES_TINY = Shapes(Hq=2, Hkv=1, D=64, Hk=2, Hv=2, dk=64, dv=64, kv_dtype=torch.float32)
SHAPES_27B = Shapes(Hq=24, Hkv=4, D=256, Hk=16, Hv=48, dk=128, dv=128, kv_dtype=torch.bfloat16)


@dataclass
class Workload:
    """One verify-round workload: per-sequence context lengths and trees,
    and the layer pattern of the mixer stack."""
    name: str
    cfg_id: int
    shapes: Shapes
    ctx_lens: list[int]
    tree_kinds: list[tuple]  # per sequence: ("fixed", parent) | ("chain", n) | ("merged", n, chain)
    n_layers: int
    attn_layers: list[int] = field(default_factory=list)  # indices of attention layers
    accept: list = field(default_factory=list)  # per sequence: ("path", [..]) | ("len", a) | ("random",)

    @property
    def n_seq(self):
        return len(self.ctx_lens)

    def is_attn(self, layer):
        return layer in self.attn_layers


def workload(cfg_id: int) -> Workload:
    if cfg_id == 0:
        # 8-node tree: chain of 5 drafted tokens below the root plus side
        # children of nodes 0 and 2; accepted path 0 -> 1 -> 2 -> 7 (length 4).
        return Workload("tiny: 1 attention (Hq 2, Hkv 1, D 64, L 256, fp32) + 1 GDN (2 heads, 64x64)",
                        0, SHAPES_TINY, [256], [("fixed", [-1, 0, 1, 2, 3, 4, 0, 2])], 2,
                        attn_layers=[0], accept=[("path", [0, 1, 2, 7])])
    if cfg_id == 1:
        return Workload("27B-shaped layer pair, L 4096, chain of 16", 1, SHAPES_27B, [4096],
                        [("chain", 16)], 2, attn_layers=[0], accept=[("len_uniform", 16)])
    if cfg_id == 2:
        return Workload("27B-shaped layer pair, L 32768, 64-node merged tree", 2, SHAPES_27B, [32768],
                        [("merged", 64, 16)], 2, attn_layers=[0], accept=[("random",)])
    if cfg_id == 3:
        return Workload("64-layer mixer stack (48 GDN + 16 attention), L 131072, 32-node tree", 3,
                        SHAPES_27B, [131072], [("merged", 32, 16)], 64,
                        attn_layers=[i for i in range(64) if i % 4 == 3], accept=[("random",)])
    if cfg_id == 4:
        return Workload("4 sequences in lockstep over the 64-layer stack, L 65536/8192/8192/8192, 16-node trees",
                        4, SHAPES_27B, [65536, 8192, 8192, 8192], [("merged", 16, 11)] * 4, 64,
                        attn_layers=[i for i in range(64) if i % 4 == 3], accept=[("random",)] * 4)
    raise ValueError(cfg_id)


# ---------------------------------------------------------------------------
# trees and tokens
# ---------------------------------------------------------------------------
def merged_tree(n: int, chain: int, rng: np.random.Generator, max_children=3, max_path=16) -> list[int]:
    """A block-drafter chain of `chain` nodes (root included) with lookup-drafter
    branches attached at random nodes that have fewer than `max_children`
    children and whose children stay within `max_path` nodes of the root."""
    parent = [-1] + list(range(chain - 1))
    depth = list(range(chain))
    nchild = [1] * (chain - 1) + [0]
    while len(parent) < n:
        cand = [i for i in range(len(parent)) if nchild[i] < max_children and depth[i] + 1 < max_path]
        p = int(rng.choice(cand))
        parent.append(p)
        depth.append(depth[p] + 1)
        nchild.append(0)
        nchild[p] += 1
    return parent


def _root_path(parent, i):
    path = []
    while i != -1:
        path.append(i)
        i = parent[i]
    return path[::-1]


def tree_and_tokens(cfg: Workload, seq: int):
    """(parent, tok, greedy, expected_path) for sequence `seq` of a workload."""
    rng = np.random.default_rng(1_000_000 * cfg.cfg_id + 999_000 + seq)
    kind = cfg.tree_kinds[seq]
    if kind[0] == "fixed":
        parent = list(kind[1])
    elif kind[0] == "chain":
        parent = [-1] + list(range(kind[1] - 1))
    elif kind[0] == "merged":
        parent = merged_tree(kind[1], kind[2], rng)
    else:
        raise ValueError(kind)
    n = len(parent)
    children = [[] for _ in range(n)]
    for i in range(1, n):
        children[parent[i]].append(i)
    # tokens: distinct among siblings
    tok = [int(rng.integers(VOCAB))] + [0] * (n - 1)
    for p in range(n):
        used = set()
        for c in children[p]:
            t = int(rng.integers(VOCAB))
            while t in used:
                t = int(rng.integers(VOCAB))
            used.add(t)
            tok[c] = t
    acc = cfg.accept[seq]
    if acc[0] == "path":
        path = list(acc[1])
    elif acc[0] == "len_uniform":
        a = int(rng.integers(1, acc[1] + 1))
        path = _root_path(parent, a - 1)  # chain: node a-1 is at depth a-1
    elif acc[0] == "random":
        path = _root_path(parent, int(rng.integers(n)))
    else:
        raise ValueError(acc)
    greedy = [int(rng.integers(VOCAB)) for _ in range(n)]
    for j in range(len(path) - 1):
        greedy[path[j]] = tok[path[j + 1]]
    last = path[-1]
    child_toks = {tok[c] for c in children[last]}
    g = int(rng.integers(VOCAB))
    while g in child_toks:
        g = int(rng.integers(VOCAB))
    greedy[last] = g
    return parent, tok, greedy, path


# ---------------------------------------------------------------------------
# per-layer tensors
# ---------------------------------------------------------------------------
def _gen(seed: int, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, std=1.0):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x * std if std != 1.0 else x


def attn_layer_inputs(cfg: Workload, layer: int, seq: int, n_nodes: int, cap: int, device="cpu"):
    """K, V [Hkv, cap, D]; q [N, Hq, D]; k_t, v_t [N, Hkv, D] (workload dtype).
    Cache rows past the context are filled too; only rows < L are read."""
    s = cfg.shapes
    g = _gen(1_000_000 * cfg.cfg_id + 1_000 * seq + layer, device)
    dt = s.kv_dtype
    K = _randn((s.Hkv, cap, s.D), g, device).to(dt)
    V = _randn((s.Hkv, cap, s.D), g, device).to(dt)
    q = _randn((n_nodes, s.Hq, s.D), g, device).to(dt)
    k_t = _randn((n_nodes, s.Hkv, s.D), g, device).to(dt)
    v_t = _randn((n_nodes, s.Hkv, s.D), g, device).to(dt)
    return dict(K=K, V=V, q=q, k_t=k_t, v_t=v_t)


def _l2norm(x):
    return x / x.norm(dim=-1, keepdim=True)


def gdn_layer_inputs(cfg: Workload, layer: int, seq: int, n_nodes: int, device="cpu"):
    """S0 fp32 [Hv, dv, dk]; q, k [N, Hk, dk]; v [N, Hv, dv] (workload dtype);
    alpha, beta fp32 [N, Hv]."""
    s = cfg.shapes
    g = _gen(1_000_000 * cfg.cfg_id + 1_000 * seq + layer, device)
    dt = s.kv_dtype
    S0 = _randn((s.Hv, s.dv, s.dk), g, device, std=0.1)
    q = _l2norm(_randn((n_nodes, s.Hk, s.dk), g, device)).to(dt)
    k = _l2norm(_randn((n_nodes, s.Hk, s.dk), g, device)).to(dt)
    v = _randn((n_nodes, s.Hv, s.dv), g, device).to(dt)
    a_raw = _randn((n_nodes, s.Hv), g, device)
    b_raw = _randn((n_nodes, s.Hv), g, device)
    alpha = torch.exp(-torch.nn.functional.softplus(a_raw))
    beta = torch.sigmoid(b_raw)
    return dict(S0=S0, q=q, k=k, v=v, alpha=alpha, beta=beta)
