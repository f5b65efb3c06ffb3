"""Invariants the method fixes, checked on the GPU bit for bit ("Adding a
model", step 4 and its load-time self-check; "Parallel requests", joint
verify):
  * every verified row equals the single-token decode row along its root path;
  * the state committed for the accepted path equals decoding that path;
  * a joint multi-sequence launch equals each sequence launched alone;
  * relabelling the tree in another topological order permutes the rows.
Edge shapes (no context, lengths around tile and split boundaries, the
deepest and the widest trees, other head dims) are checked against the oracle
here as well."""
import numpy as np
import pytest
import torch

import oracle.tree_verify as O
from gpu_helpers import check_close, check_state, f64, oracle_attn, oracle_commit_state, oracle_gdn, seq_slice
from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu


def bits(t):
    """Integer view of a tensor, for bit-for-bit comparison."""
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


def decode_attn_rows(r, li, seq, path):
    """Decode the tokens of `path` one by one on layer li's cache of `seq`,
    starting from the committed length; returns the output rows [len(path), Hq, D]."""
    a = r.attn[li]
    lo, _ = seq_slice(r, seq)
    layer1 = B.AttnLayer([a["layer"].K[seq]], [a["layer"].V[seq]], r.cfg.shapes.Hq)
    len1 = torch.tensor([r.cfg.ctx_lens[seq]], dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    wsb = B.tv_attn_workspace_bytes(r.plan, layer1, 1, 1, r.cap)
    ws = torch.empty(max(16, wsb) // 4 + 4, dtype=torch.float32, device="cuda") if wsb else None
    rows = []
    for node in path:
        i = lo + node
        out = torch.empty_like(a["q"][i:i + 1])
        B.tv_decode_step(r.plan, layer1, None, 1, len1, r.cap, a["q"][i:i + 1].clone(), a["k_t"][i:i + 1].clone(),
                         a["v_t"][i:i + 1].clone(), None, None, out, r.attn_scale, ws, status)
        B.tv_len_advance(len1, None, 1, 1)
        rows.append(out)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    return torch.cat(rows)


def decode_gdn_rows(r, li, seq, path, S0):
    g = r.gdn[li]
    lo, _ = seq_slice(r, seq)
    S = S0.clone()
    layer1 = B.GdnLayer([S], r.cfg.shapes.Hk, r.cfg.shapes.kv_dtype)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rows = []
    for node in path:
        i = lo + node
        out = torch.empty_like(g["out"][i:i + 1])
        # fresh tensors: a one-node slice of a packed batch need not be 16-byte aligned
        B.tv_decode_step(None, None, layer1, 1, None, 0, g["q"][i:i + 1].clone(), g["k"][i:i + 1].clone(),
                         g["v"][i:i + 1].clone(), g["alpha"][i:i + 1].clone(), g["beta"][i:i + 1].clone(), out,
                         r.gdn_scale, None, status)
        rows.append(out)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    return torch.cat(rows), S


def check_rows_equal_decode(r, seqs=None, paths_per_seq=None, rng=None):
    """Verify (no commit), then decode every node's path and compare bitwise."""
    S0 = {(li, s): g["layer"].S[s].clone() for li, g in r.gdn.items() for s in range(r.cfg.n_seq)}
    r.len.copy_(r.len0)
    r.verify()
    torch.cuda.synchronize()
    assert r.status() == 0
    for s in (range(r.cfg.n_seq) if seqs is None else seqs):
        n = r.n_nodes[s]
        lo, _ = seq_slice(r, s)
        if paths_per_seq is None:
            ends = range(n)
        else:
            leaves = [i for i in range(n) if i not in r.parents[s]]
            ends = [r.expected_paths[s][-1]] + list(rng.choice(leaves, size=min(paths_per_seq, len(leaves)),
                                                              replace=False))
        for end in ends:
            path = O.root_path(r.parents[s], int(end))
            idx = [lo + x for x in path]
            for li in r.attn:
                dec = decode_attn_rows(r, li, s, path)
                ver = r.attn[li]["out"][idx]
                assert torch.equal(bits(dec), bits(ver)), f"attn layer {li} seq {s} path {path}: verify row != decode row"
            for li in r.gdn:
                dec, S_end = decode_gdn_rows(r, li, s, path, S0[(li, s)])
                ver = r.gdn[li]["out"][idx]
                assert torch.equal(bits(dec), bits(ver)), f"gdn layer {li} seq {s} path {path}: verify row != decode row"


@pytest.mark.parametrize("cfg_id", [0, 1, 2])
def test_verify_rows_equal_decode_rows(cfg_id):
    check_rows_equal_decode(VerifyRound(synth.workload(cfg_id)))


def test_verify_rows_equal_decode_rows_full_size():
    """128k context, 32-node tree: the accepted path and three random root
    paths on one attention and one GDN layer of the stack."""
    cfg = synth.workload(3)
    r = VerifyRound(cfg, layers=[2, 3])
    check_rows_equal_decode(r, paths_per_seq=3, rng=np.random.default_rng(0))


def test_verify_rows_equal_decode_rows_four_sequences():
    """Four sequences in one launch (contexts 65,536 / 8,192 x 3, 16-node
    trees): for every sequence, its accepted path and three random root
    paths, decoded on that sequence's own cache and state, give the verified
    rows bit for bit on one attention and one GDN layer of the stack."""
    cfg = synth.workload(4)
    r = VerifyRound(cfg, layers=[2, 3])
    check_rows_equal_decode(r, paths_per_seq=3, rng=np.random.default_rng(1))


def test_commit_equals_decode_replay():
    """The committed state is the decode replay of the accepted path, bit for bit."""
    r = VerifyRound(synth.workload(2))
    S0 = {li: g["layer"].S[0].clone() for li, g in r.gdn.items()}
    r.run(reset_len=False)
    torch.cuda.synchronize()
    path = r.expected_paths[0]
    for li in r.gdn:
        _, S_dec = decode_gdn_rows(r, li, 0, path, S0[li])
        assert torch.equal(S_dec, r.gdn[li]["layer"].S[0])


def small_workload(cfg_id, shapes, ctx_lens, tree_kinds, accept=None):
    return synth.Workload(f"edge {cfg_id}", cfg_id, shapes, list(ctx_lens), list(tree_kinds), 2, attn_layers=[0],
                          accept=accept or [("random",)] * len(ctx_lens))


SH128 = synth.Shapes(Hq=8, Hkv=2, D=128, Hk=2, Hv=4, dk=64, dv=64, kv_dtype=torch.bfloat16)
SH64 = synth.Shapes(Hq=4, Hkv=1, D=64, Hk=1, Hv=2, dk=128, dv=100, kv_dtype=torch.bfloat16)
SHF = synth.Shapes(Hq=6, Hkv=2, D=128, Hk=2, Hv=6, dk=128, dv=128, kv_dtype=torch.float32)
SHG64 = synth.Shapes(Hq=64, Hkv=1, D=64, Hk=1, Hv=2, dk=64, dv=64, kv_dtype=torch.bfloat16)  # largest group

EDGES = [
    # (name, shapes, context lengths, trees, split)
    ("no-context", synth.SHAPES_27B, [0], [("merged", 12, 6)], 4096),
    ("len-1", synth.SHAPES_27B, [1], [("chain", 16)], 4096),
    ("len-63", synth.SHAPES_27B, [63], [("chain", 3)], 4096),
    ("len-64", synth.SHAPES_27B, [64], [("merged", 10, 4)], 4096),
    ("tail-crosses-tile", synth.SHAPES_27B, [120], [("chain", 16)], 4096),
    ("tail-crosses-split", synth.SHAPES_27B, [250], [("chain", 16)], 256),
    ("split-64", synth.SHAPES_27B, [700], [("merged", 20, 16)], 64),
    ("continue-split", synth.SHAPES_27B, [4096 + 1000], [("merged", 24, 12)], 1024),
    ("widest-tree", synth.SHAPES_27B, [333], [("merged", 64, 8)], 512),
    ("single-node", synth.SHAPES_27B, [517], [("chain", 1)], 128),
    ("multi-seq", synth.SHAPES_27B, [3000, 65, 0, 1290], [("merged", 16, 11), ("chain", 5), ("merged", 7, 3),
                                                          ("chain", 16)], 1024),
    ("D128", SH128, [1500, 70], [("merged", 30, 10), ("merged", 9, 5)], 512),
    ("D64", SH64, [900], [("merged", 40, 16)], 256),
    ("f32-D128", SHF, [300, 5], [("merged", 20, 8), ("chain", 4)], 4096),
    # the root's row starts its own segment one tile before the deeper rows,
    # which read the last split's snapshot in place of its final state
    ("snapshot-D128", SH128, [191], [("chain", 16)], 512),
    ("snapshot-D64", SH64, [447], [("merged", 20, 8)], 256),
    # more split records than the tail stages in shared memory (the rest read
    # from global memory), and so many that not even their weights are staged
    ("many-splits", synth.SHAPES_27B, [3000], [("merged", 8, 4)], 64),
    ("unstaged-weights", SHG64, [18_000], [("chain", 2)], 64),
]


@pytest.mark.parametrize("name,shapes,lens,trees,split", EDGES, ids=[e[0] for e in EDGES])
def test_edge_parity_and_invariance(name, shapes, lens, trees, split):
    cfg = small_workload(900, shapes, lens, trees)
    r = VerifyRound(cfg, split=split)
    S0 = {(li, s): g["layer"].S[s].clone() for li, g in r.gdn.items() for s in range(cfg.n_seq)}
    r.run(reset_len=False)
    torch.cuda.synchronize()
    assert r.status() == 0
    for s in range(cfg.n_seq):
        lo, hi = seq_slice(r, s)
        for li in r.attn:
            check_close(r.attn[li]["out"][lo:hi], oracle_attn(r, li, s), f"{name} attn seq {s}")
        for li in r.gdn:
            check_close(r.gdn[li]["out"][lo:hi], oracle_gdn(r, li, s, S0[(li, s)]), f"{name} gdn seq {s}")
            check_state(r.gdn[li]["layer"].S[s],
                        oracle_commit_state(r, li, s, S0[(li, s)], r.expected_paths[s]), f"{name} state seq {s}")
    # restore the states and check verify == decode on every node
    for (li, s), S in S0.items():
        r.gdn[li]["layer"].S[s].copy_(S)
    check_rows_equal_decode(r)


def test_joint_equals_lone():
    """Four sequences in one launch give the same bits as each alone."""
    cfg = small_workload(901, synth.SHAPES_27B, [2000, 64, 700, 5], [("merged", 16, 11)] * 4)
    r = VerifyRound(cfg, split=512)
    r.verify()
    torch.cuda.synchronize()
    for s in range(cfg.n_seq):
        lo, hi = seq_slice(r, s)
        t1 = B.Tree([r.parents[s]])
        B.tv_tree_prepare(t1)
        len1 = r.len0[s:s + 1].clone()
        for li, a in r.attn.items():
            l1 = B.AttnLayer([a["layer"].K[s]], [a["layer"].V[s]], cfg.shapes.Hq)
            wsb = B.tv_attn_workspace_bytes(r.plan, l1, 1, t1.n_max, int(len1[0]))
            ws = torch.empty(max(16, wsb) // 4 + 4, dtype=torch.float32, device="cuda")
            out = torch.empty_like(a["q"][lo:hi])
            B.tv_attn_tree_verify(r.plan, l1, t1, len1, int(len1[0]), a["q"][lo:hi].clone(),
                                  a["k_t"][lo:hi].clone(), a["v_t"][lo:hi].clone(), out, r.attn_scale, ws)
            torch.cuda.synchronize()
            assert torch.equal(out, a["out"][lo:hi])
        for li, g in r.gdn.items():
            g1 = B.GdnLayer([g["layer"].S[s]], cfg.shapes.Hk, cfg.shapes.kv_dtype)
            out = torch.empty_like(g["out"][lo:hi])
            B.tv_gdn_tree_verify(g1, t1, g["q"][lo:hi].clone(), g["k"][lo:hi].clone(),
                                 g["v"][lo:hi].clone(), g["alpha"][lo:hi].clone(),
                                 g["beta"][lo:hi].clone(), out, r.gdn_scale)
            torch.cuda.synchronize()
            assert torch.equal(out, g["out"][lo:hi])


def test_relabel_permutes_rows():
    cfg = small_workload(902, synth.SHAPES_27B, [777], [("merged", 24, 10)])
    r = VerifyRound(cfg, split=256)
    r.verify()
    torch.cuda.synchronize()
    parent = r.parents[0]
    n = len(parent)
    rng = np.random.default_rng(5)
    placed, order = {-1}, []
    while len(order) < n:
        ready = [i for i in range(n) if i not in order and parent[i] in placed]
        i = int(rng.choice(ready))
        order.append(i)
        placed.add(i)
    new_of = {old: new for new, old in enumerate(order)}
    parent2 = [-1 if parent[o] == -1 else new_of[parent[o]] for o in order]
    t2 = B.Tree([parent2])
    B.tv_tree_prepare(t2)
    idx = torch.tensor(order, device="cuda")
    for li, a in r.attn.items():
        out = torch.empty_like(a["q"])
        B.tv_attn_tree_verify(r.plan, a["layer"], t2, r.len0, r.max_len, a["q"][idx].clone(),
                              a["k_t"][idx].clone(), a["v_t"][idx].clone(), out, r.attn_scale, r.ws)
        torch.cuda.synchronize()
        assert torch.equal(out, a["out"][idx])
    for li, g in r.gdn.items():
        out = torch.empty_like(g["out"])
        B.tv_gdn_tree_verify(g["layer"], t2, g["q"][idx].clone(), g["k"][idx].clone(),
                             g["v"][idx].clone(), g["alpha"][idx].clone(), g["beta"][idx].clone(),
                             out, r.gdn_scale)
        torch.cuda.synchronize()
        assert torch.equal(out, g["out"][idx])


@pytest.mark.parametrize("cfg_id", [2, 3, 4])
def test_overlapped_launch_gives_same_bits(cfg_id):
    """A round launched with TV_TREE_OVERLAP (programmatic dependent launch)
    gives the same bits as the same round launched plainly: outputs of every
    verified layer, the accepted path, and the committed caches and states.
    On the 64-layer workload the attention layers also run as CTA pairs
    (two 128-row blocks streaming the same tiles)."""
    cfg = synth.workload(cfg_id)
    layers = None if cfg.n_layers <= 2 else [0, 1, 2, 3, 7]
    runs = []
    for overlap in (False, True):
        r = VerifyRound(cfg, layers=layers, overlap=overlap)
        r.run()
        torch.cuda.synchronize()
        assert r.status() == 0
        got = {"path": r.path.clone(), "acc": r.acc_len.clone(), "bonus": r.bonus.clone(), "len": r.len.clone()}
        for li, a in r.attn.items():
            got[f"out{li}"] = bits(a["out"]).clone()
            got[f"K{li}"] = [bits(k).clone() for k in a["layer"].K]
        for li, g in r.gdn.items():
            got[f"out{li}"] = bits(g["out"]).clone()
            got[f"S{li}"] = [bits(st).clone() for st in g["layer"].S]
        runs.append(got)
        del r
        torch.cuda.empty_cache()
    plain, ov = runs
    for k in plain:
        if isinstance(plain[k], list):
            for x, y in zip(plain[k], ov[k]):
                assert torch.equal(x, y), k
        else:
            assert torch.equal(plain[k], ov[k]), k
