"""Gated DeltaNet front end and gated output norm on the GPU ("Adding a
model", "What is still specific to Qwen3.8": the Gated DeltaNet layer with its
gated norm; "The model layer": convolution tails): tv_gdn_front ->
tv_gdn_tree_verify -> tv_gdn_out_norm against the fp64 oracle
(oracle/gdn_front.py), verified rows equal to the same tokens decoded one by
one with real tail commits, bit for bit, and the tail commit of the accepted
path equal to the decoded tail; the fused call (front end inside the verify
kernel) equal to the three calls bit for bit."""
import numpy as np
import pytest
import torch

import oracle.gdn_front as G
import oracle.tree_verify as O
from gpu_helpers import check_close, f64
from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth

pytestmark = pytest.mark.gpu

W = 4
TV_ERR_TREE = 5


def check_gated_norm(got, ref, gate, stages, what):
    """Tolerance of the gated-norm output against the oracle run from the raw
    inputs, derived from the arithmetic: the output is n * g with n = o /
    rms(o) of unit RMS and g = w_norm * SiLU(z).  Each bf16 stage between the
    raw inputs and n (q/k/v, o, the output) carries at most the error of a
    bf16 output of unit scale (max-abs 2e-2, the bar of the verify outputs),
    and g multiplies it, so the bound on each element is stages * 2e-2 *
    max(1, |g|); rel-L2 keeps the verify outputs' 5e-3.  fp32: the fp32 bars
    in place of the bf16 ones."""
    g = f64(got)
    err = np.abs(g - ref)
    rel = float(np.linalg.norm(g - ref) / np.linalg.norm(ref))
    if got.dtype == torch.bfloat16:
        bound, rel_bar = stages * 2e-2 * np.maximum(1.0, np.abs(gate)), 5e-3
    else:
        bound, rel_bar = stages * 1e-4 * np.maximum(1.0, np.abs(gate)), 1e-5
    worst = float((err / bound).max())
    assert worst <= 1.0 and rel <= rel_bar, f"{what}: worst err/bound {worst:.3f}, rel-L2 {rel:.3e}"


def check_norm_stage(got, ref, what):
    """The norm kernel alone (the oracle fed the GPU's own bf16 o): fp32
    arithmetic and one final rounding, so each element is within 2^-8 of its
    value (bf16: half an ulp is 2^-9 relative; fp32: 1e-5)."""
    g = f64(got)
    tol = 2.0 ** -8 if got.dtype == torch.bfloat16 else 1e-5
    worst = float((np.abs(g - ref) / np.maximum(np.abs(ref), 1e-3)).max())
    assert worst <= tol, f"{what}: worst relative error {worst:.3e}"


def bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


class Case:
    def __init__(self, cfg_id, seed):
        cfg = synth.workload(cfg_id)
        s = cfg.shapes
        self.dt = s.kv_dtype
        self.Hk, self.Hv, self.dk, self.dv = s.Hk, s.Hv, s.dk, s.dv
        self.C = 2 * s.Hk * s.dk + s.Hv * s.dv
        self.parent = synth.tree_and_tokens(cfg, 0)[0]
        n = self.n = len(self.parent)
        g = torch.Generator(device="cuda").manual_seed(seed)
        rn = lambda *shape, std=1.0, dt=torch.float32: (torch.randn(*shape, generator=g, device="cuda") * std).to(dt)
        self.x = rn(n, self.C, dt=self.dt)
        self.tail0 = rn(W - 1, self.C, dt=self.dt)
        self.wconv = rn(self.C, W, std=0.5)
        self.a_raw, self.b_raw = rn(n, self.Hv), rn(n, self.Hv)
        self.z = rn(n, self.Hv, self.dv, dt=self.dt)
        self.w_norm = 1.0 + rn(self.dv, std=0.1)
        self.S0 = rn(self.Hv, self.dv, self.dk, std=0.1)
        self.scale = self.dk ** -0.5

    def layer(self, tail):
        return B.GdnFrontLayer(self.Hk, self.Hv, self.dk, self.dv, self.wconv, [tail], self.dt)

    def empty(self, rows):
        e = lambda *sh, dt=None: torch.empty(*sh, dtype=dt or self.dt, device="cuda")
        return dict(q=e(rows, self.Hk, self.dk), k=e(rows, self.Hk, self.dk), v=e(rows, self.Hv, self.dv),
                    alpha=e(rows, self.Hv, dt=torch.float32), beta=e(rows, self.Hv, dt=torch.float32),
                    o=e(rows, self.Hv, self.dv), out=e(rows, self.Hv, self.dv))

    def verify(self):
        tree = B.Tree([self.parent])
        B.tv_tree_prepare(tree)
        tail = self.tail0.clone()
        fl = self.layer(tail)
        b = self.empty(self.n)
        B.tv_gdn_front(fl, tree, 1, self.x, self.a_raw, self.b_raw, b["q"], b["k"], b["v"], b["alpha"], b["beta"])
        S = self.S0.clone()
        gl = B.GdnLayer([S], self.Hk, self.dt)
        B.tv_gdn_tree_verify(gl, tree, b["q"], b["k"], b["v"], b["alpha"], b["beta"], b["o"], self.scale)
        B.tv_gdn_out_norm(fl, self.n, b["o"], self.z, self.w_norm, b["out"])
        torch.cuda.synchronize()
        assert tree.status_code() == 0
        return tree, fl, tail, b


@pytest.mark.parametrize("cfg_id", [0, 1, 2])
def test_gdn_front_matches_oracle(cfg_id):
    c = Case(cfg_id, 900 + cfg_id)
    _, _, _, b = c.verify()
    x, tail, wc = f64(c.x), f64(c.tail0), f64(c.wconv)
    q, k, v, alpha, beta = G.gdn_front(x, tail, wc, f64(c.a_raw), f64(c.b_raw), c.parent, c.Hk, c.dk, c.Hv, c.dv)
    check_close(b["q"], q, "front q")
    check_close(b["k"], k, "front k")
    check_close(b["v"], v, "front v")
    check_close(b["alpha"], alpha, "alpha")
    check_close(b["beta"], beta, "beta")
    ref = G.gdn_layer_tree_verify(f64(c.S0), x, tail, wc, f64(c.a_raw), f64(c.b_raw), f64(c.z), f64(c.w_norm),
                                  c.parent, c.Hk, c.dk, c.Hv, c.dv, c.scale)
    gate = f64(c.w_norm) * G.silu(f64(c.z))
    check_norm_stage(b["out"], G.gated_rmsnorm(f64(b["o"]), f64(c.z), f64(c.w_norm)), "gated norm of the GPU's o")
    check_gated_norm(b["out"], ref, gate, 3, "gated-norm output from the raw inputs")


@pytest.mark.parametrize("cfg_id", [0, 2])
def test_gdn_front_verify_rows_equal_decode_rows(cfg_id):
    c = Case(cfg_id, 950 + cfg_id)
    tree, _, _, b = c.verify()
    leaves = [i for i in range(c.n) if i not in c.parent]
    rng = np.random.default_rng(cfg_id)
    ends = [max(range(c.n), key=lambda i: len(O.root_path(c.parent, i)))] + \
        list(rng.choice(leaves, size=min(2, len(leaves)), replace=False))
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for end in ends:
        path = O.root_path(c.parent, int(end))
        tail = c.tail0.clone()
        fl = c.layer(tail)
        S = c.S0.clone()
        gl = B.GdnLayer([S], c.Hk, c.dt)
        rows = []
        for j in path:
            d = c.empty(1)
            xj = c.x[j:j + 1].clone()
            B.tv_gdn_front(fl, None, 1, xj, c.a_raw[j:j + 1].clone(), c.b_raw[j:j + 1].clone(), d["q"], d["k"],
                           d["v"], d["alpha"], d["beta"], status)
            B.tv_decode_step(None, None, gl, 1, None, 0, d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["o"],
                             c.scale, None, status)
            B.tv_gdn_out_norm(fl, 1, d["o"], c.z[j:j + 1].clone(), c.w_norm, d["out"])
            B.tv_gdn_conv_commit(fl, None, 1, xj, status=status)
            rows.append(d["out"])
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        dec = torch.cat(rows)
        assert torch.equal(bits(dec), bits(b["out"][path])), f"path {path}: verified row != decoded row"
        # committing the path on the tree gives the tail decoding it left
        tail2 = c.tail0.clone()
        fl2 = c.layer(tail2)
        pth = torch.full((1, B.TV_MAX_PATH), -1, dtype=torch.int32, device="cuda")
        pth[0, :len(path)] = torch.tensor(path, dtype=torch.int32)
        acc = torch.tensor([len(path)], dtype=torch.int32, device="cuda")
        B.tv_gdn_conv_commit(fl2, tree, 1, c.x, pth, acc)
        torch.cuda.synchronize()
        assert torch.equal(bits(tail2), bits(tail)), f"path {path}: committed tail != decoded tail"
        assert np.array_equal(f64(tail2), G.commit_tail(f64(c.tail0), f64(c.x), path))


@pytest.mark.parametrize("cfg_id,width,dt,overlap", [(0, 1, None, False), (0, 4, None, False), (1, 8, None, False),
                                                     (2, 4, None, False), (3, 4, None, False), (4, 4, None, False),
                                                     (1, 4, torch.float32, False), (4, 2, torch.float32, False),
                                                     (3, 4, None, True), (4, 4, None, True)])
def test_gdn_fused_equals_front_verify_norm(cfg_id, width, dt, overlap):
    """tv_gdn_tree_verify_fused gives the bits of tv_gdn_front ->
    tv_gdn_tree_verify -> tv_gdn_out_norm on every sequence of the workload's
    trees (one 8/16/64/32-node tree, four 16-node trees), for convolution
    widths 1 (no tail), 2, 4 and 8 (windows reaching past the root into each
    sequence's own tail), bf16 and fp32 layers (fp32 on the 27B shapes runs
    the key-head clusters too), plain and overlapped launches (programmatic
    dependent launch, as a round runs them); states and tails stay as they
    were."""
    cfg = synth.workload(cfg_id)
    sh = cfg.shapes
    parents = [synth.tree_and_tokens(cfg, s)[0] for s in range(cfg.n_seq)]
    fused_vs_three(parents, sh.Hk, sh.Hv, sh.dk, dt or sh.kv_dtype, width, 1200 + 10 * cfg_id + width, overlap)


@pytest.mark.parametrize("Hk,Hv,dk,n_seq,width", [(4, 8, 64, 2, 4), (2, 8, 128, 1, 3), (8, 8, 128, 3, 5),
                                                  (2, 2, 64, 2, 8)])
def test_gdn_fused_other_head_shapes(Hk, Hv, dk, n_seq, width):
    """The fused call on head shapes beside the workloads': dk = dv = 64
    (a whole head in one CTA), four value heads to a key head (clusters of
    eight), one value head to a key head (clusters of two), merged trees of
    20-40 nodes, bf16."""
    rng = np.random.default_rng(Hk * 100 + Hv + dk + width)
    parents = [synth.merged_tree(int(rng.integers(20, 41)), 10, rng) for _ in range(n_seq)]
    fused_vs_three(parents, Hk, Hv, dk, torch.bfloat16, width, 1400 + Hk + Hv + dk + width)


def fused_vs_three(parents, Hk, Hv, dk, dt, width, seed, overlap=False):
    """tv_gdn_tree_verify_fused against tv_gdn_front -> tv_gdn_tree_verify ->
    tv_gdn_out_norm on the same inputs: bitwise equal outputs, states and
    tails untouched, status clean."""
    sh = type("Shapes", (), dict(Hk=Hk, Hv=Hv, dk=dk, dv=dk))
    n_seq = len(parents)
    n = sum(len(p) for p in parents)
    C = 2 * sh.Hk * sh.dk + sh.Hv * sh.dv
    g = torch.Generator(device="cuda").manual_seed(seed)
    rn = lambda *shape, std=1.0, d=torch.float32: (torch.randn(*shape, generator=g, device="cuda") * std).to(d)
    x = rn(n, C, d=dt)
    a_raw, b_raw = rn(n, sh.Hv), rn(n, sh.Hv)
    z = rn(n, sh.Hv, sh.dv, d=dt)
    wconv, w_norm = rn(C, width, std=0.5), 1.0 + rn(sh.dv, std=0.1)
    tails = [rn(max(width - 1, 1), C, d=dt) for _ in parents]
    S0 = [rn(sh.Hv, sh.dv, sh.dk, std=0.1) for _ in parents]
    scale = sh.dk ** -0.5
    tree = B.Tree(parents, overlap=overlap)
    B.tv_tree_prepare(tree)
    fl = B.GdnFrontLayer(sh.Hk, sh.Hv, sh.dk, sh.dv, wconv, tails, dt)
    e = lambda *shape, d=dt: torch.empty(*shape, dtype=d, device="cuda")
    q, k, v = e(n, sh.Hk, sh.dk), e(n, sh.Hk, sh.dk), e(n, sh.Hv, sh.dv)
    alpha, beta = e(n, sh.Hv, d=torch.float32), e(n, sh.Hv, d=torch.float32)
    o, ref = e(n, sh.Hv, sh.dv), e(n, sh.Hv, sh.dv)
    S1 = [s.clone() for s in S0]
    B.tv_gdn_front(fl, tree, n_seq, x, a_raw, b_raw, q, k, v, alpha, beta)
    B.tv_gdn_tree_verify(B.GdnLayer(S1, sh.Hk, dt), tree, q, k, v, alpha, beta, o, scale)
    B.tv_gdn_out_norm(fl, n, o, z, w_norm, ref)
    S2 = [s.clone() for s in S0]
    tails0 = [t.clone() for t in tails]
    out = torch.full((n, sh.Hv, sh.dv), float("nan"), dtype=dt, device="cuda")
    B.tv_gdn_tree_verify_fused(B.GdnLayer(S2, sh.Hk, dt), fl, tree, x, a_raw, b_raw, z, w_norm, out, scale)
    torch.cuda.synchronize()
    assert tree.status_code() == 0
    assert torch.equal(bits(out), bits(ref)), "fused output != front -> verify -> norm"
    for s in range(n_seq):
        assert torch.equal(bits(S2[s]), bits(S0[s])), f"sequence {s}: the verify changed a state"
        assert torch.equal(bits(tails[s]), bits(tails0[s])), f"sequence {s}: the verify changed a tail"


def test_gdn_fused_after_a_malformed_tree_does_nothing():
    """A launch whose status word already holds an error (here a malformed
    tree in the second of four sequences) leaves the fused call a no-op:
    every CTA, clusters included, takes the early path through the cluster's
    barriers and returns; the output keeps its fill and the call returns."""
    cfg = synth.workload(4)
    sh = cfg.shapes
    dt = sh.kv_dtype
    parents = [synth.tree_and_tokens(cfg, s)[0] for s in range(cfg.n_seq)]
    parents[1] = list(parents[1])
    parents[1][3] = 7  # a parent after its child
    n = sum(len(p) for p in parents)
    C = 2 * sh.Hk * sh.dk + sh.Hv * sh.dv
    g = torch.Generator(device="cuda").manual_seed(1300)
    rn = lambda *shape, std=1.0, d=torch.float32: (torch.randn(*shape, generator=g, device="cuda") * std).to(d)
    tails = [rn(3, C, d=dt) for _ in parents]
    fl = B.GdnFrontLayer(sh.Hk, sh.Hv, sh.dk, sh.dv, rn(C, 4, std=0.5), tails, dt)
    S = [rn(sh.Hv, sh.dv, sh.dk, std=0.1) for _ in parents]
    tree = B.Tree(parents)
    B.tv_tree_prepare(tree)
    out = torch.full((n, sh.Hv, sh.dv), 7.0, dtype=dt, device="cuda")
    B.tv_gdn_tree_verify_fused(B.GdnLayer(S, sh.Hk, dt), fl, tree, rn(n, C, d=dt), rn(n, sh.Hv), rn(n, sh.Hv),
                               rn(n, sh.Hv, sh.dv, d=dt), 1.0 + rn(sh.dv, std=0.1), out, sh.dk ** -0.5)
    torch.cuda.synchronize()
    assert tree.status_code() == TV_ERR_TREE
    assert bool((out == 7.0).all()), "an output was written after the error"


@pytest.mark.parametrize("cfg_id", [0, 2, 3])
def test_gdn_fused_verify_rows_equal_fused_decode_rows(cfg_id):
    """The fused forms keep the row-invariance rule ("Adding a model", step
    4): each node verified by tv_gdn_tree_verify_fused equals the same token
    decoded by tv_gdn_decode_fused after its ancestors (tails committed token
    by token), bit for bit; and tv_gdn_decode_fused equals tv_gdn_front ->
    tv_decode_step -> tv_gdn_out_norm, outputs and states."""
    c = Case(cfg_id, 1500 + cfg_id)
    tree = B.Tree([c.parent])
    B.tv_tree_prepare(tree)
    tail = c.tail0.clone()
    fl = c.layer(tail)
    S = c.S0.clone()
    ver = torch.empty(c.n, c.Hv, c.dv, dtype=c.dt, device="cuda")
    B.tv_gdn_tree_verify_fused(B.GdnLayer([S], c.Hk, c.dt), fl, tree, c.x, c.a_raw, c.b_raw, c.z, c.w_norm, ver,
                               c.scale)
    torch.cuda.synchronize()
    assert tree.status_code() == 0
    leaves = [i for i in range(c.n) if i not in c.parent]
    rng = np.random.default_rng(cfg_id + 7)
    ends = [max(range(c.n), key=lambda i: len(O.root_path(c.parent, i)))] + \
        list(rng.choice(leaves, size=min(2, len(leaves)), replace=False))
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for end in ends:
        path = O.root_path(c.parent, int(end))
        t1, t2 = c.tail0.clone(), c.tail0.clone()
        f1, f2 = c.layer(t1), c.layer(t2)
        S1, S2 = c.S0.clone(), c.S0.clone()
        g1, g2 = B.GdnLayer([S1], c.Hk, c.dt), B.GdnLayer([S2], c.Hk, c.dt)
        for j in path:
            xj, aj, bj, zj = (c.x[j:j + 1].clone(), c.a_raw[j:j + 1].clone(), c.b_raw[j:j + 1].clone(),
                              c.z[j:j + 1].clone())
            fused = torch.empty(1, c.Hv, c.dv, dtype=c.dt, device="cuda")
            B.tv_gdn_decode_fused(g1, f1, 1, xj, aj, bj, zj, c.w_norm, fused, c.scale, status)
            B.tv_gdn_conv_commit(f1, None, 1, xj, status=status)
            d = c.empty(1)
            B.tv_gdn_front(f2, None, 1, xj, aj, bj, d["q"], d["k"], d["v"], d["alpha"], d["beta"], status)
            B.tv_decode_step(None, None, g2, 1, None, 0, d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["o"],
                             c.scale, None, status)
            B.tv_gdn_out_norm(f2, 1, d["o"], zj, c.w_norm, d["out"])
            B.tv_gdn_conv_commit(f2, None, 1, xj, status=status)
            torch.cuda.synchronize()
            assert int(status[0]) == 0
            assert torch.equal(bits(fused), bits(d["out"])), f"node {j}: fused decode != three calls"
            assert torch.equal(bits(fused[0]), bits(ver[j])), f"node {j}: fused decode != fused verify row"
        assert torch.equal(bits(S1), bits(S2)), f"path {path}: fused decode state != decode state"
        assert torch.equal(bits(t1), bits(t2))
