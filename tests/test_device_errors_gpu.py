"""Errors only the device can see, made on the host, checked on the GPU.

"Adding a model", step 4 and its load-time self-check: a mismatch turns
speculation off cleanly and names what failed; nothing may crash.  Here a
malformed draft tree, a tree longer than the library's bounds, a commit past
a cache's capacity, a length above the host bound and a decode into a full
cache must each leave the documented status code in the round's status word,
and every later call that shares the word must write nothing: no output row,
no cache row, no state, no length.  None of these faults, traps or hangs a
GPU: the kernels test the status word and return.  The bounded waits of the
pipelined kernels are run out against barriers nothing arrives at.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import check_close, oracle_attn, oracle_gdn, seq_slice
from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu

TV_ERR_TREE, TV_ERR_CAPACITY, TV_ERR_TIMEOUT, TV_ERR_LEN = 5, 6, 9, 10
SH = synth.Shapes(Hq=8, Hkv=2, D=128, Hk=2, Hv=4, dk=64, dv=64, kv_dtype=torch.bfloat16)
SENTINEL = 7.0


def workload(cfg_id, lens, trees, accept=None):
    return synth.Workload(f"errors {cfg_id}", cfg_id, SH, list(lens), list(trees), 2, attn_layers=[0],
                          accept=accept or [("random",)] * len(lens))


def snapshot(r):
    return {"len": r.len.clone(),
            "K": [k.clone() for a in r.attn.values() for k in a["layer"].K],
            "V": [v.clone() for a in r.attn.values() for v in a["layer"].V],
            "S": [S.clone() for g in r.gdn.values() for S in g["layer"].S]}


def assert_untouched(r, snap, what):
    assert torch.equal(r.len, snap["len"]), f"{what}: lengths changed"
    now = snapshot(r)
    for key in ("K", "V", "S"):
        for i, (a, b) in enumerate(zip(now[key], snap[key])):
            assert torch.equal(a, b), f"{what}: {key}[{i}] written"


def fill_outputs(r):
    for d in (r.attn, r.gdn):
        for x in d.values():
            x["out"].fill_(SENTINEL)


def all_sentinel(t):
    return bool((t.float() == SENTINEL).all())


def run_with_tree(r, parents, n_max=None, node_off=None):
    """One round on r's buffers with another tree descriptor (same node count)."""
    keep = r.tree
    r.tree = B.Tree(parents, n_max=n_max, overlap=True)
    assert r.tree.n_total == keep.n_total
    if node_off is not None:
        r.tree.node_off.copy_(torch.tensor(node_off, dtype=torch.int32))
    try:
        r.run(reset_len=False)
        torch.cuda.synchronize()
        return r.tree.status_code()
    finally:
        r.tree = keep


def bad_trees():
    """(name, workload, parents from the workload's trees -> bad parents, n_max, node_off)."""
    small = workload(970, [1500, 300], [("merged", 20, 8), ("merged", 12, 6)])

    def edit(i, v):
        def f(ps):
            p0 = list(ps[0])
            p0[i] = v
            return [p0, ps[1]], None, None
        return f

    def long_path(ps):  # a 17-node root path: one more than a tree may hold
        p0 = [-1] + list(range(16)) + [0] * (len(ps[0]) - 17)
        return [p0, ps[1]], None, None

    def empty_first(ps):  # node offsets that give sequence 0 no nodes
        return ps, None, [0, 0, len(ps[0]) + len(ps[1])]

    big = workload(971, [700, 900], [("merged", 64, 16), ("merged", 64, 16)])

    def too_many(ps):  # 65 and 63 nodes against a bound of 64 per tree
        p0 = [-1] + [(i - 1) // 4 for i in range(1, 65)]
        p1 = [-1] + [(i - 1) // 4 for i in range(1, 63)]
        return [p0, p1], 64, None

    return [("parent-after-child", small, edit(5, 9)), ("second-root", small, edit(4, -1)),
            ("root-with-parent", small, edit(0, 0)), ("17-node-path", small, long_path),
            ("sequence-without-nodes", small, empty_first), ("65-node-tree", big, too_many)]


@pytest.mark.parametrize("name,cfg,make", bad_trees(), ids=[b[0] for b in bad_trees()])
def test_malformed_tree_sets_tree_error_and_writes_nothing(name, cfg, make):
    r = VerifyRound(cfg, split=512)
    parents, n_max, node_off = make(r.parents)
    fill_outputs(r)
    r.path.fill_(5)
    snap = snapshot(r)
    code = run_with_tree(r, parents, n_max=n_max, node_off=node_off)
    assert code == TV_ERR_TREE, (name, code)
    for li in r.layers:
        out = r.attn[li]["out"] if li in r.attn else r.gdn[li]["out"]
        assert all_sentinel(out), f"{name}: layer {li} wrote outputs"
    assert (r.path == -1).all() and (r.acc_len == 0).all() and (r.bonus == -1).all(), name
    assert_untouched(r, snap, name)
    # the same buffers still run a well-formed round afterwards
    r.tree.status.zero_()
    r.run()
    torch.cuda.synchronize()
    assert r.status() == 0


def test_commit_past_capacity_sets_capacity_error_and_commits_nothing():
    # sequence 0 accepts 4 rows on top of L = 1000 with room for one more row
    cfg = workload(972, [1000, 500], [("chain", 8), ("merged", 10, 5)], accept=[("path", [0, 1, 2, 3]), ("random",)])
    r = VerifyRound(cfg, split=256, cap_extra=1)
    assert r.cap == 1001
    S0 = {(li, s): g["layer"].S[s].clone() for li, g in r.gdn.items() for s in range(cfg.n_seq)}
    snap = snapshot(r)
    r.run(reset_len=False)
    torch.cuda.synchronize()
    assert r.status() == TV_ERR_CAPACITY
    # verify and accept ran before the commit found the overflow
    assert int(r.acc_len[0]) == 4 and r.path[0, :4].tolist() == [0, 1, 2, 3]
    for s in range(cfg.n_seq):
        lo, hi = seq_slice(r, s)
        for li in r.attn:
            check_close(r.attn[li]["out"][lo:hi], oracle_attn(r, li, s), f"attn seq {s}")
        for li in r.gdn:
            check_close(r.gdn[li]["out"][lo:hi], oracle_gdn(r, li, s, S0[(li, s)]), f"gdn seq {s}")
    assert_untouched(r, snap, "capacity")


def test_length_above_bound_sets_len_error():
    cfg = workload(973, [900, 400], [("merged", 12, 6), ("merged", 9, 4)])
    r = VerifyRound(cfg, split=256)
    r.len[0] = r.max_len + 1  # within the cache, above the host bound the launch was sized for
    fill_outputs(r)
    snap = snapshot(r)
    r.run(reset_len=False)
    torch.cuda.synchronize()
    assert r.status() == TV_ERR_LEN
    lo, hi = seq_slice(r, 0)
    for li, a in r.attn.items():
        assert all_sentinel(a["out"][lo:hi]), "attention rows of the over-long sequence written"
    for li, g in r.gdn.items():  # after the attention layer: every later call is a no-op
        assert all_sentinel(g["out"]), "GDN layer after the error wrote outputs"
    assert int(r.acc_len[0]) == 0 and int(r.bonus[0]) == -1
    assert_untouched(r, snap, "length")


def test_decode_into_full_cache_sets_capacity_error():
    cfg = workload(974, [500], [("chain", 4)])
    r = VerifyRound(cfg, split=256)
    a = r.attn[0]
    layer1 = B.AttnLayer([a["layer"].K[0]], [a["layer"].V[0]], SH.Hq)
    len1 = torch.tensor([r.cap], dtype=torch.int32, device="cuda")  # no free row left
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    wsb = B.tv_attn_workspace_bytes(r.plan, layer1, 1, 1, r.cap)
    ws = torch.empty(max(16, wsb) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full_like(a["q"][:1], SENTINEL)
    K0, V0 = a["layer"].K[0].clone(), a["layer"].V[0].clone()
    B.tv_decode_step(r.plan, layer1, None, 1, len1, r.cap, a["q"][:1].clone(), a["k_t"][:1].clone(),
                     a["v_t"][:1].clone(), None, None, out, r.attn_scale, ws, status)
    torch.cuda.synchronize()
    assert int(status[0]) == TV_ERR_CAPACITY
    assert all_sentinel(out)
    assert torch.equal(a["layer"].K[0], K0) and torch.equal(a["layer"].V[0], V0)


@pytest.mark.parametrize("limit", [1 << 12, 1 << 20])
def test_bounded_waits_give_up_and_report_timeout(limit):
    """Barriers nothing arrives at: every wait form gives up after its limit,
    the status word says TV_ERR_TIMEOUT, and the context stays usable."""
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    result = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    B.tv_wait_selftest(status, result, limit)
    torch.cuda.synchronize()
    assert result.tolist() == [1, 0, 0, 0]
    assert int(status[0]) == TV_ERR_TIMEOUT
    r = VerifyRound(workload(975, [300], [("chain", 5)]), split=256)
    r.run()
    torch.cuda.synchronize()
    assert r.status() == 0
    assert np.isfinite(r.attn[0]["out"].float().cpu().numpy()).all()
