"""Per-shape CUDA graphs of the verify round, on the GPU.

* A graph captured for one tree shape and replayed with other trees of the
  same shape gives the same bits as the eager round on those trees: nothing
  but the shape key is baked into the graph.
* A node's rows do not depend on the rest of its tree (each row is a function
  of its own query and its ancestors), so the graph for a prefix of a tree
  gives exactly the full tree's rows for those nodes -- across the widths
  where the attention path changes its launch (one 128-row block, a CTA
  pair for two blocks, three blocks).  Some of those replays are also checked
  against the oracle directly.
* The accept walk on the prefix stops where the full tree's path leaves it.
"""
import pytest
import torch

import oracle.tree_verify as O
from gpu_helpers import check_close, f64
from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.graphs import ShapeGraphs, prefix_trees, shape_key
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu


def pair_workload(lens, trees, cfg_id):
    return synth.Workload(f"graphs {cfg_id}", cfg_id, synth.SHAPES_27B, list(lens), list(trees), 2,
                          attn_layers=[0], accept=[("random",)] * len(lens))


def snapshot(r):
    return {li: [S.clone() for S in g["layer"].S] for li, g in r.gdn.items()}


def restore(r, snap):
    for li, Ss in snap.items():
        for S, S0 in zip(r.gdn[li]["layer"].S, Ss):
            S.copy_(S0)
    r.len.copy_(r.len0)


def outputs(r, n):
    return {li: d["out"][:n].clone() for d_ in (r.attn, r.gdn) for li, d in d_.items()}


def eager_round(r, parents, tok, greedy):
    """The round on a fresh tree descriptor, eagerly, on r's buffers."""
    keep = r.tree
    r.tree = B.Tree(parents, overlap=bool(keep.c.flags & B.TV_TREE_OVERLAP))
    n = r.tree.n_total
    r.tok[:n].copy_(torch.tensor(tok, dtype=torch.int32))
    r.greedy[:n].copy_(torch.tensor(greedy, dtype=torch.int32))
    try:
        r.run()
        torch.cuda.synchronize()
        assert r.status() == 0
    finally:
        r.tree = keep


def round_result(r, n):
    res = outputs(r, n)
    res["path"] = r.path.clone()
    res["acc"] = r.acc_len.clone()
    res["bonus"] = r.bonus.clone()
    res["len"] = r.len.clone()
    res["S"] = [S.clone() for g in r.gdn.values() for S in g["layer"].S]
    res["K"] = [K.clone() for a in r.attn.values() for K in a["layer"].K]
    res["V"] = [V.clone() for a in r.attn.values() for V in a["layer"].V]
    return res


def assert_same(a, b, what):
    for k in a:
        if isinstance(a[k], list):
            for x, y in zip(a[k], b[k]):
                assert torch.equal(x, y), f"{what}: {k}"
        else:
            assert torch.equal(a[k], b[k]), f"{what}: {k}"


def test_prefix_graphs_give_the_full_trees_rows():
    cfg = pair_workload([3000], [("merged", 64, 16)], 950)
    r = VerifyRound(cfg, split=512)
    snap = snapshot(r)
    parents, tok, greedy, path = synth.tree_and_tokens(cfg, 0)
    r.verify()
    torch.cuda.synchronize()
    assert r.status() == 0
    full = outputs(r, 64)
    sg = ShapeGraphs(r)
    for w in (1, 5, 16, 21, 22, 42, 43, 64):
        key = sg.load(prefix_trees([parents], w), tok[:w], greedy[:w])
        assert key == (1, w, w)
        restore(r, snap)  # the capture's warm-up round committed
        sg.replay(key)
        torch.cuda.synchronize()
        assert sg.status(key) == 0
        got = outputs(r, w)
        for li in got:
            assert torch.equal(got[li], full[li][:w]), f"width {w}, layer {li}"
        if w in (5, 22, 43):  # one width per attention launch form, against the oracle
            pw = parents[:w]
            for li, a in r.attn.items():
                ref = O.attn_tree_verify(f64(a["layer"].K[0][:, :3000]), f64(a["layer"].V[0][:, :3000]), 3000,
                                         f64(a["q"][:w]), f64(a["k_t"][:w]), f64(a["v_t"][:w]), pw, r.attn_scale)
                check_close(got[li], ref, f"graph width {w} attention layer {li}")
            for li, g in r.gdn.items():
                ref = O.gdn_tree_verify(f64(snap[li][0]), f64(g["q"][:w]), f64(g["k"][:w]), f64(g["v"][:w]),
                                        f64(g["alpha"][:w]), f64(g["beta"][:w]), pw, r.gdn_scale)
                check_close(got[li], ref, f"graph width {w} GDN layer {li}")
        want_path = [x for x in path if x < w]
        a = int(r.acc_len[0])
        assert a == len(want_path), (w, a, want_path)
        assert r.path[0, :a].tolist() == want_path
        assert int(r.bonus[0]) == greedy[want_path[-1]]
        assert int(r.len[0]) == 3000 + a


def test_graph_replay_equals_eager_rounds_of_the_same_shape():
    """Two sequences; trees of sizes (a, b) and (b, a) share one graph."""
    cfg = pair_workload([2500, 700], [("merged", 40, 12), ("merged", 40, 9)], 951)
    r = VerifyRound(cfg, split=256)
    snap = snapshot(r)
    trees = [synth.tree_and_tokens(cfg, q) for q in range(2)]
    sg = ShapeGraphs(r)
    shapes = [(30, 12), (12, 30), (21, 21)]
    key0 = None
    for wa, wb in shapes:
        parents = [trees[0][0][:wa], trees[1][0][:wb]]
        tok = trees[0][1][:wa] + trees[1][1][:wb]
        greedy = trees[0][2][:wa] + trees[1][2][:wb]
        if shape_key(parents) != (2, 42, 30):
            continue  # (21, 21) has another n_max: its own graph
        restore(r, snap)
        eager_round(r, parents, tok, greedy)
        want = round_result(r, 42)
        key = sg.load(parents, tok, greedy)
        key0 = key0 or key
        assert key == key0
        restore(r, snap)
        sg.replay(key)
        torch.cuda.synchronize()
        assert sg.status(key) == 0
        assert_same(round_result(r, 42), want, f"trees of {wa} and {wb} nodes")
    assert len(sg.graphs) == 1
    # a shape that does not fit the round's buffers is refused
    with pytest.raises(ValueError):
        sg.load([trees[0][0][:40] + [0], trees[1][0][:5]])
