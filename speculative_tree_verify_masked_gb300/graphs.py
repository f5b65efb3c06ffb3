"""Verify rounds replayed from CUDA graphs, one graph per tree shape.

A drafter hands each round a different tree, but a captured round depends on
the host only through the tree descriptor's sizes: the number of sequences,
the total node count and the largest tree (which bound the grids, the
workspace and the shared-memory carve-up).  Everything else the round reads
-- node offsets, parent arrays, tokens, lengths, node inputs -- lives on the
device.  So one graph per shape key (n_seq, n_total, n_max) serves every
round whose trees have that shape; the caller refills the tree and token
buffers and replays.  ("How ignis serves a request", section 4: decode
rounds replay a graph captured for each exact batch width, because padding a
narrow round to a wider graph moves state the round does not need; "Parallel
requests", "What a slot costs": a slot keeps its own set of verify graphs.
The same holds for tree width: a graph captured for 64 nodes would verify 64
rows for a 16-node tree.)

All graphs of a ShapeGraphs share the buffers of one VerifyRound built for
the widest trees: a graph for a narrower shape uses the leading rows of the
node-input, output and token buffers, and its own small tree buffers.
"""
from __future__ import annotations

import torch

from . import binding as B
from .round import VerifyRound


def shape_key(parents) -> tuple[int, int, int]:
    """(n_seq, n_total, n_max) of a list of per-sequence parent arrays."""
    sizes = [len(p) for p in parents]
    return len(sizes), sum(sizes), max(sizes)


def prefix_trees(parents, width: int):
    """The first `width` nodes of each tree (a prefix of a parent array whose
    parents precede their children is again such an array)."""
    return [list(p[:width]) for p in parents]


class ShapeGraphs:
    """CUDA graphs of one VerifyRound's round, keyed by tree shape."""

    def __init__(self, r: VerifyRound):
        self.r = r
        self.graphs: dict[tuple[int, int, int], tuple[torch.cuda.CUDAGraph, B.Tree]] = {}
        self._overlap = bool(r.tree.c.flags & B.TV_TREE_OVERLAP)

    def _check(self, key):
        n_seq, n_total, n_max = key
        t = self.r.tree
        if n_seq != t.n_seq or n_total > t.n_total or n_max > t.n_max:
            raise ValueError(f"tree shape {key} does not fit the round's buffers "
                             f"({t.n_seq} sequences, {t.n_total} nodes, {t.n_max} per tree)")

    def capture(self, parents) -> tuple[int, int, int]:
        """Capture the round for trees of this shape (the parent arrays only
        give the shape and the warm-up run's trees) and return its key."""
        key = shape_key(parents)
        self._check(key)
        if key in self.graphs:
            return key
        tree = B.Tree(parents, device=self.r.device, n_max=key[2], overlap=self._overlap)
        keep = self.r.tree
        self.r.tree = tree
        try:
            g = self.r.capture()
        finally:
            self.r.tree = keep
        self.graphs[key] = (g, tree)
        return key

    def load(self, parents, tok=None, greedy=None) -> tuple[int, int, int]:
        """Write a round's trees (and optionally its drafted and greedy
        tokens, node-major like the node inputs) into the buffers of the
        graph for their shape, capturing it first if needed."""
        key = self.capture(parents)
        _, tree = self.graphs[key]
        off = [0]
        for p in parents:
            off.append(off[-1] + len(p))
        tree.node_off.copy_(torch.tensor(off, dtype=torch.int32))
        tree.parent.copy_(torch.tensor([int(x) for p in parents for x in p], dtype=torch.int32))
        tree.status.zero_()
        n = key[1]
        if tok is not None:
            self.r.tok[:n].copy_(torch.as_tensor(tok, dtype=torch.int32))
        if greedy is not None:
            self.r.greedy[:n].copy_(torch.as_tensor(greedy, dtype=torch.int32))
        return key

    def replay(self, key) -> None:
        self.graphs[key][0].replay()

    def status(self, key) -> int:
        return self.graphs[key][1].status_code()
