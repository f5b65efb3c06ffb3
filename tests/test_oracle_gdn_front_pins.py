"""Pins for the Gated DeltaNet front-end oracle (oracle/gdn_front.py) against
things other than itself: torch's depthwise conv1d on a chain, identity and
closed-form values of the gates and the norms, brute force against
sequential decoding with real tail commits, and planted mistakes that a pin
must catch."""
import numpy as np
import pytest
import torch

import oracle.gdn_front as G
import oracle.tree_verify as O

TREE = [-1, 0, 1, 2, 3, 4, 0, 2, 7, 1]  # chain of 6 with side branches (node 7 has a child)


def rand_case(seed, C=12, W=4, n=None, parent=TREE):
    rng = np.random.default_rng(seed)
    n = len(parent) if n is None else n
    x = rng.standard_normal((n, C))
    tail = rng.standard_normal((W - 1, C))
    w = rng.standard_normal((C, W))
    return x, tail, w


def torch_causal_conv(seq, w):
    """Depthwise conv1d of seq [T][C] with weights [C][W], no padding: output
    t corresponds to the window seq[t .. t+W-1]."""
    C, W = w.shape
    inp = torch.tensor(seq.T[None], dtype=torch.float64)
    wt = torch.tensor(w[:, None, :], dtype=torch.float64)
    return torch.nn.functional.conv1d(inp, wt, groups=C)[0].numpy().T


def test_chain_matches_torch_conv1d():
    chain = list(range(-1, 7))
    x, tail, w = rand_case(1, parent=chain)
    got = G.short_conv_tree(x, tail, w, chain)
    ref = G.silu(torch_causal_conv(np.concatenate([tail, x]), w))
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_zero_tail_is_zero_padding():
    chain = list(range(-1, 5))
    x, _, w = rand_case(2, parent=chain)
    tail = np.zeros((3, x.shape[1]))
    C, W = w.shape
    ref = torch.nn.functional.conv1d(torch.tensor(x.T[None]), torch.tensor(w[:, None, :]), groups=C,
                                     padding=W - 1)[0].numpy().T[:len(chain)]
    assert np.allclose(G.short_conv_tree(x, tail, w, chain), G.silu(ref), rtol=0, atol=1e-12)


def test_tree_node_equals_conv_along_its_root_path():
    x, tail, w = rand_case(3)
    got = G.short_conv_tree(x, tail, w, TREE)
    for i in range(len(TREE)):
        path = O.root_path(TREE, i)
        ref = G.silu(torch_causal_conv(np.concatenate([tail, x[path]]), w))[-1]
        assert np.allclose(got[i], ref, rtol=0, atol=1e-12), i


def test_width_one_identity_conv():
    x = np.random.default_rng(4).standard_normal((len(TREE), 5))
    got = G.short_conv_tree(x, np.zeros((0, 5)), np.ones((5, 1)), TREE)
    assert np.allclose(got, x / (1 + np.exp(-x)), rtol=0, atol=1e-15)


def test_gate_closed_values():
    a = np.array([0.0, 50.0, -50.0])
    b = np.array([0.0, 50.0, -50.0])
    _, _, _, alpha, beta = G.gdn_front(np.zeros((1, 2 * 2 + 2)), np.zeros((0, 6)), np.ones((6, 1)), a[None],
                                       b[None], [-1], 1, 2, 1, 2)
    assert alpha[0, 0] == pytest.approx(0.5, abs=1e-15)   # exp(-ln 2)
    assert alpha[0, 1] == pytest.approx(0.0, abs=1e-20)   # strong decay
    assert alpha[0, 2] == pytest.approx(1.0, abs=1e-20)   # no decay
    assert beta[0, 0] == pytest.approx(0.5, abs=1e-15)
    assert beta[0, 1] == pytest.approx(1.0, abs=1e-15)
    assert beta[0, 2] == pytest.approx(0.0, abs=1e-20)


def test_l2norm_unit_rows_and_scale_invariance():
    x = np.random.default_rng(5).standard_normal((4, 3 * 8))
    y = G.l2norm_heads(x, 3)
    n = (y.reshape(4, 3, 8) ** 2).sum(-1)
    assert np.allclose(n, 1.0, atol=1e-6)
    assert np.allclose(G.l2norm_heads(7.0 * x, 3), y, atol=1e-7)


def test_gated_rmsnorm_closed_form():
    o = np.ones((2, 3, 4))
    z = np.random.default_rng(6).standard_normal((2, 3, 4))
    w = np.array([1.0, 2.0, -1.0, 0.5])
    got = G.gated_rmsnorm(o, z, w)
    assert np.allclose(got, w / np.sqrt(1 + G.EPS_NORM) * z / (1 + np.exp(-z)), rtol=0, atol=1e-15)
    # scale invariance of the norm (up to eps)
    o2 = np.random.default_rng(7).standard_normal((2, 3, 4))
    assert np.allclose(G.gated_rmsnorm(5 * o2, z, w), G.gated_rmsnorm(o2, z, w), atol=1e-6)


def layer_case(seed, parent=TREE):
    Hk, dk, Hv, dv = 1, 4, 2, 4
    C = 2 * Hk * dk + Hv * dv
    rng = np.random.default_rng(seed)
    n = len(parent)
    return dict(S0=rng.normal(0, 0.1, (Hv, dv, dk)), x=rng.standard_normal((n, C)),
                tail=rng.standard_normal((3, C)), wconv=rng.standard_normal((C, 4)) * 0.5,
                a_raw=rng.standard_normal((n, Hv)), b_raw=rng.standard_normal((n, Hv)),
                z=rng.standard_normal((n, Hv, dv)), w_norm=rng.standard_normal(dv), Hk=Hk, dk=dk, Hv=Hv, dv=dv)


def decode_layer_path(c, path, scale):
    """Sequential decoding of the path's tokens with real commits of the
    tail and the state after each token; returns the outputs [len][Hv][dv]."""
    tail, S = c["tail"].copy(), c["S0"].copy()
    outs = []
    for j in path:
        win = np.concatenate([tail, c["x"][j:j + 1]])[-4:]
        u = G.silu(np.einsum("jc,cj->c", win, c["wconv"]))
        q, k, v = G.split_channels(u[None], c["Hk"], c["dk"], c["Hv"], c["dv"])
        q = G.l2norm_heads(q.reshape(1, -1), c["Hk"]).reshape(q.shape)[0]
        k = G.l2norm_heads(k.reshape(1, -1), c["Hk"]).reshape(k.shape)[0]
        alpha = np.exp(-np.log1p(np.exp(c["a_raw"][j])))
        beta = 1 / (1 + np.exp(-c["b_raw"][j]))
        o = O.gdn_decode(S, q, k, v[0], alpha, beta, scale)
        outs.append(G.gated_rmsnorm(o[None], c["z"][j:j + 1], c["w_norm"])[0])
        tail = np.concatenate([tail, c["x"][j:j + 1]])[1:]
    return np.stack(outs), tail


def test_layer_brute_force_against_sequential_decode():
    c = layer_case(8)
    scale = c["dk"] ** -0.5
    got = G.gdn_layer_tree_verify(c["S0"], c["x"], c["tail"], c["wconv"], c["a_raw"], c["b_raw"], c["z"],
                                  c["w_norm"], TREE, c["Hk"], c["dk"], c["Hv"], c["dv"], scale)
    for i in range(len(TREE)):
        path = O.root_path(TREE, i)
        dec, tail_end = decode_layer_path(c, path, scale)
        assert np.allclose(got[i], dec[-1], rtol=0, atol=1e-10), i
        assert np.allclose(G.commit_tail(c["tail"], c["x"], path), tail_end, rtol=0, atol=0)


def test_commit_tail_short_and_long_paths():
    tail = np.arange(6.0).reshape(3, 2)
    x = 100 + np.arange(20.0).reshape(10, 2)
    assert np.array_equal(G.commit_tail(tail, x, [0]), np.stack([tail[1], tail[2], x[0]]))
    assert np.array_equal(G.commit_tail(tail, x, [0, 1, 2, 7]), x[[1, 2, 7]])


# ---------------------------------------------------------------------------
# planted mistakes: each must fail a pin above
# ---------------------------------------------------------------------------
def test_planted_mistakes_are_caught(monkeypatch):
    good_inputs = G.conv_inputs

    def off_by_one(x, tail, parent, i):  # skips the parent: reads the grandparent's window
        p = parent[i]
        win = good_inputs(x, tail, parent, p if p >= 0 else i)
        return np.concatenate([win[1:], x[i:i + 1]])

    monkeypatch.setattr(G, "conv_inputs", off_by_one)
    with pytest.raises(AssertionError):
        test_chain_matches_torch_conv1d()
    monkeypatch.undo()

    def reversed_tail(x, tail, parent, i):
        return good_inputs(x, tail[::-1], parent, i)

    monkeypatch.setattr(G, "conv_inputs", reversed_tail)
    with pytest.raises(AssertionError):
        test_chain_matches_torch_conv1d()
    monkeypatch.undo()

    monkeypatch.setattr(G, "softplus", lambda a: -np.logaddexp(0.0, a))  # decay sign flipped
    with pytest.raises(AssertionError):
        test_gate_closed_values()
    monkeypatch.undo()

    good_norm = G.gated_rmsnorm
    monkeypatch.setattr(G, "gated_rmsnorm",
                        lambda o, z, w, eps=G.EPS_NORM: np.asarray(o) / np.sqrt((np.asarray(o) ** 2).sum(-1, keepdims=True) + eps) * w * G.silu(z))
    with pytest.raises(AssertionError):
        test_gated_rmsnorm_closed_form()
    monkeypatch.setattr(G, "gated_rmsnorm", good_norm)
