"""Pins for the attention front-end oracle (oracle/attn_front.py) against
things other than itself: values of the rotation angle derived by hand,
an independent complex-number formulation of the rotary embedding, the
algebra of rotations (identity, composition, norms, shift invariance of
scores), the sigmoid's closed values, and torch's causal attention on a
chain.  The last block plants mistakes in the oracle and checks that a pin
catches each one."""
import math

import numpy as np
import pytest
import torch

import oracle.attn_front as F
import oracle.tree_verify as O


def rope_complex(x, pos, rot_dims, theta):
    """The rotary embedding as complex multiplication: plane j is the complex
    number x_j + i x_{j + r/2}, multiplied by e^{i pos w_j}, w_j = theta^(-2j/r)."""
    x = np.asarray(x, dtype=np.float64)
    half = rot_dims // 2
    z = x[..., :half] + 1j * x[..., half:rot_dims]
    w = np.array([theta ** (-2.0 * j / rot_dims) for j in range(half)])
    z = z * np.exp(1j * pos * w)
    out = x.copy()
    out[..., :half] = z.real
    out[..., half:rot_dims] = z.imag
    return out


def test_identity_cases():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 16))
    assert np.array_equal(F.rope(x, 17, 0, 10000.0), x)
    assert np.allclose(F.rope(x, 0, 16, 10000.0), x, rtol=0, atol=0)


def test_hand_derived_angles():
    # rot_dims 4, theta 100: plane 0 turns by pos, plane 1 by pos / 10.
    x = np.zeros(6)
    x[1] = 1.0  # plane 1, real part (dimension 1 pairs with dimension 3)
    y = F.rope(x, 5, 4, 100.0)
    assert y[1] == pytest.approx(0.8775825618903728, abs=1e-15)  # cos 0.5
    assert y[3] == pytest.approx(0.479425538604203, abs=1e-15)   # sin 0.5
    assert y[0] == 0 and y[2] == 0 and y[4] == 0 and y[5] == 0
    x = np.zeros(6)
    x[2] = 1.0  # plane 0, imaginary part: (0, 1) turned by 5 rad -> (-sin 5, cos 5)
    y = F.rope(x, 5, 4, 100.0)
    assert y[0] == pytest.approx(0.9589242746631385, abs=1e-15)   # -sin 5
    assert y[2] == pytest.approx(0.28366218546322625, abs=1e-15)  # cos 5
    # dimensions past rot_dims pass through
    x = np.arange(6.0)
    assert np.array_equal(F.rope(x, 9, 4, 100.0)[4:], x[4:])


@pytest.mark.parametrize("rot,theta,pos", [(64, 10000.0, 131071), (256, 1e6, 4097), (2, 10.0, 3), (128, 500.0, 0)])
def test_matches_complex_formulation(rot, theta, pos):
    rng = np.random.default_rng(rot)
    x = rng.standard_normal((4, 256))
    # angles up to ~1.3e5 rad: the two formulations' argument reductions differ by ~1e-11
    assert np.allclose(F.rope(x, pos, rot, theta), rope_complex(x, pos, rot, theta), rtol=0, atol=1e-9)


def test_rotation_algebra():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 64))
    r, th = 32, 10000.0
    # norms are kept, rotations compose, and scores depend only on the offset
    assert np.allclose(np.linalg.norm(F.rope(x, 123, r, th), axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    assert np.allclose(F.rope(F.rope(x, 40, r, th), 2, r, th), F.rope(x, 42, r, th), atol=1e-12)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    s1 = F.rope(q, 1000, r, th) @ F.rope(k, 990, r, th)
    s2 = F.rope(q, 7, r, th) @ F.rope(k, -3, r, th)
    assert s1 == pytest.approx(s2, abs=1e-11)


def test_sigmoid_closed_values():
    assert F.sigmoid(0.0) == 0.5
    assert F.sigmoid(math.log(3.0)) == pytest.approx(0.75, abs=1e-15)
    assert F.sigmoid(-math.log(3.0)) == pytest.approx(0.25, abs=1e-15)


def front_case(rng, n, Hq=4, Hkv=2, D=16, L=6, cap=48, rot=8, theta=50.0):
    K = rng.standard_normal((Hkv, cap, D))
    V = rng.standard_normal((Hkv, cap, D))
    # the cache holds keys rotated at their own positions
    for p in range(L):
        K[:, p] = F.rope(K[:, p], p, rot, theta)
    q = rng.standard_normal((n, Hq, D))
    k = rng.standard_normal((n, Hkv, D))
    v = rng.standard_normal((n, Hkv, D))
    gate = rng.standard_normal((n, Hq, D))
    return K, V, L, q, k, v, gate


def test_chain_equals_library_causal_attention_with_rotary():
    """A chain tree is causal attention over context + chain, with every key
    and query rotated at its absolute position (torch, float64)."""
    rng = np.random.default_rng(3)
    n, Hq, Hkv, D, L, rot, th = 7, 4, 2, 16, 6, 8, 50.0
    K, V, L, q, k, v, gate = front_case(rng, n, Hq, Hkv, D, L, rot=rot, theta=th)
    parent = [-1] + list(range(n - 1))
    out, k_t, v_t = F.attn_front_tree_verify(K, V, L, q, k, v, gate, parent, 0.25, rot, th)
    # independent: complex rotation at absolute positions, then causal SDPA
    qr = np.stack([rope_complex(q[i], L + i, rot, th) for i in range(n)])
    kr = np.stack([rope_complex(k[i], L + i, rot, th) for i in range(n)])
    keys = np.concatenate([K[:, :L].transpose(1, 0, 2), kr], axis=0)   # [L+n, Hkv, D]
    vals = np.concatenate([V[:, :L].transpose(1, 0, 2), v], axis=0)
    G = Hq // Hkv
    ref = np.zeros((n, Hq, D))
    for h in range(Hq):
        Q = torch.tensor(qr[:, h])[None, None]
        Kt = torch.tensor(keys[:, h // G])[None, None]
        Vt = torch.tensor(vals[:, h // G])[None, None]
        mask = torch.ones(n, L + n, dtype=torch.bool).tril(diagonal=L)
        ref[:, h] = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, attn_mask=mask, scale=0.25)[0, 0].numpy()
    ref = ref / (1.0 + np.exp(-gate))
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    assert np.allclose(k_t, kr, atol=1e-12) and np.array_equal(v_t, v)


def test_tree_rows_equal_decode_after_committing_the_path():
    """Each node's output equals decoding it at position L + depth after its
    ancestors' rotated keys were committed (the row-invariance rule)."""
    rng = np.random.default_rng(4)
    parent = [-1, 0, 0, 1, 1, 3, 2, 6]
    n = len(parent)
    K, V, L, q, k, v, gate = front_case(rng, n)
    out, k_t, v_t = F.attn_front_tree_verify(K, V, L, q, k, v, gate, parent, 0.3, 8, 50.0)
    for i in range(n):
        Kc, Vc = K.copy(), V.copy()
        path = O.root_path(parent, i)
        for e, j in enumerate(path[:-1]):
            O.commit_attn(Kc, Vc, L + e, k_t[None, j], v_t[None, j], [0])
        o = F.attn_front_decode(Kc, Vc, L + len(path) - 1, q[i], k[i], v[i], gate[i], 0.3, 8, 50.0)
        assert np.allclose(o, out[i], rtol=0, atol=1e-12), i


# ---------------------------------------------------------------------------
# planted mistakes: each must fail a pin above
# ---------------------------------------------------------------------------
def rope_interleaved(x, pos, rot_dims, theta):
    """Planted: pairs adjacent dimensions (2j, 2j+1) instead of j, j + r/2."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    for j in range(rot_dims // 2):
        a = pos * theta ** (-2.0 * j / rot_dims)
        u, w = x[..., 2 * j], x[..., 2 * j + 1]
        out[..., 2 * j] = u * math.cos(a) - w * math.sin(a)
        out[..., 2 * j + 1] = w * math.cos(a) + u * math.sin(a)
    return out


_rope = F.rope


def rope_sign(x, pos, rot_dims, theta):
    """Planted: turns the other way."""
    return _rope(x, -pos, rot_dims, theta)


def rope_freq(x, pos, rot_dims, theta):
    """Planted: frequencies theta^(-j/r) (the factor 2 dropped)."""
    x = np.asarray(x, dtype=np.float64)
    half = rot_dims // 2
    a = pos * theta ** (-np.arange(half) / rot_dims)
    out = x.copy()
    p, r = x[..., :half], x[..., half:rot_dims]
    out[..., :half] = p * np.cos(a) - r * np.sin(a)
    out[..., half:rot_dims] = r * np.cos(a) + p * np.sin(a)
    return out


@pytest.mark.parametrize("planted", [rope_interleaved, rope_sign, rope_freq])
def test_planted_rotary_mistakes_are_caught(monkeypatch, planted):
    monkeypatch.setattr(F, "rope", planted)
    with pytest.raises(AssertionError):
        test_hand_derived_angles()
    with pytest.raises(AssertionError):
        test_chain_equals_library_causal_attention_with_rotary()


def test_planted_gate_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(F, "sigmoid", lambda g: 1.0 / (1.0 + np.exp(np.asarray(g, dtype=np.float64))))
    with pytest.raises(AssertionError):
        test_sigmoid_closed_values()
    with pytest.raises(AssertionError):
        test_chain_equals_library_causal_attention_with_rotary()


def test_planted_position_mistake_is_caught(monkeypatch):
    """Rotating tree nodes at L + i (node index) instead of L + depth."""
    real = F.depths
    monkeypatch.setattr(F, "depths", lambda parent: list(range(len(parent))))
    with pytest.raises(AssertionError):
        test_tree_rows_equal_decode_after_committing_the_path()
    monkeypatch.setattr(F, "depths", real)
