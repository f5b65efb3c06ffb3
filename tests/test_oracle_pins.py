"""Pins for the CPU oracle, against things other than itself: sequential decode
with real commits (brute force), an independent chunked closed form of the
delta rule, closed-form special cases, a library causal-attention routine,
hand-derived values (tests/golden/hand_worked.json) and an exhaustive accept
check.  The last block plants mistakes into the oracle and checks that a pin
catches each one."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle.tree_verify as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def random_tree(rng, n, max_path=16):
    parent = [-1]
    depth = [0]
    for i in range(1, n):
        cand = [j for j in range(i) if depth[j] + 1 < max_path]
        p = int(rng.choice(cand))
        parent.append(p)
        depth.append(depth[p] + 1)
    return parent


def attn_case(rng, n, Hq=4, Hkv=2, D=8, L=5, cap=40):
    K = rng.standard_normal((Hkv, cap, D))
    V = rng.standard_normal((Hkv, cap, D))
    q = rng.standard_normal((n, Hq, D))
    k_t = rng.standard_normal((n, Hkv, D))
    v_t = rng.standard_normal((n, Hkv, D))
    return K, V, L, q, k_t, v_t


def gdn_case(rng, n, Hk=2, Hv=4, dk=6, dv=5):
    S0 = 0.3 * rng.standard_normal((Hv, dv, dk))
    q = rng.standard_normal((n, Hk, dk))
    k = rng.standard_normal((n, Hk, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, Hv, dv))
    alpha = np.exp(-np.log1p(np.exp(rng.standard_normal((n, Hv)))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((n, Hv))))
    return S0, q, k, v, alpha, beta


# ---------------------------------------------------------------------------
# pin checks (raise AssertionError on a mismatch)
# ---------------------------------------------------------------------------
def check_attn_vs_sequential_decode(seed=0, n=9):
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    K, V, L, q, k_t, v_t = attn_case(rng, n)
    scale = 0.37
    o = O.attn_tree_verify(K, V, L, q, k_t, v_t, parent, scale)
    for i in range(n):
        Kc, Vc = K.copy(), V.copy()
        for d, j in enumerate(O.root_path(parent, i)):
            out = O.attn_decode(Kc, Vc, L + d, q[j], k_t[j], v_t[j], scale)
        np.testing.assert_allclose(o[i], out, rtol=0, atol=1e-12)


def check_gdn_vs_sequential_decode(seed=0, n=9):
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    S0, q, k, v, alpha, beta = gdn_case(rng, n)
    o = O.gdn_tree_verify(S0, q, k, v, alpha, beta, parent, 0.5)
    for i in range(n):
        S = S0.copy()
        for j in O.root_path(parent, i):
            out = O.gdn_decode(S, q[j], k[j], v[j], alpha[j], beta[j], 0.5)
        np.testing.assert_allclose(o[i], out, rtol=0, atol=1e-12)


def check_gdn_vs_chunked(seed=0, n=12):
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    S0, q, k, v, alpha, beta = gdn_case(rng, n)
    a = O.gdn_tree_verify(S0, q, k, v, alpha, beta, parent, 0.7)
    c = O.gdn_tree_chunked(S0, q, k, v, alpha, beta, parent, 0.7)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-10)


def check_gdn_closed_forms(seed=0, n=7):
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    S0, q, k, v, alpha, beta = gdn_case(rng, n)
    Hv = S0.shape[0]
    G = Hv // k.shape[1]
    # alpha = 1, beta = 0: the state never moves, o = scale S0 q
    o = O.gdn_tree_verify(S0, q, k, v, np.ones_like(alpha), np.zeros_like(beta), parent, 0.9)
    for i in range(n):
        for h in range(Hv):
            np.testing.assert_allclose(o[i, h], 0.9 * S0[h] @ q[i, h // G], atol=1e-12)
    # alpha = 1, beta = 1, unit k: the delta rule stores v under k exactly
    path = O.root_path(parent, n - 1)
    S = O.gdn_path_state(S0, k, v, np.ones_like(alpha), np.ones_like(beta), path)
    last = path[-1]
    for h in range(Hv):
        np.testing.assert_allclose(S[h] @ k[last, h // G], v[last, h], atol=1e-12)
    # alpha = 0: everything before the last token is forgotten, S = beta v k^T
    S = O.gdn_path_state(S0, k, v, np.zeros_like(alpha), beta, path)
    for h in range(Hv):
        np.testing.assert_allclose(S[h], beta[last, h] * np.outer(v[last, h], k[last, h // G]), atol=1e-12)


def check_attn_closed_forms(seed=0, n=6):
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    K, V, L, q, k_t, v_t = attn_case(rng, n)
    Hq, Hkv = q.shape[1], K.shape[0]
    G = Hq // Hkv
    # L = 0, root only sees itself: o = v_root
    o = O.attn_tree_verify(K, V, 0, q, k_t, v_t, parent, 1.0)
    for h in range(Hq):
        np.testing.assert_allclose(o[0, h], v_t[0, h // G], atol=1e-12)
    # q = 0: uniform weights, o = mean of the visible value rows
    o = O.attn_tree_verify(K, V, L, np.zeros_like(q), k_t, v_t, parent, 1.0)
    for i in range(n):
        path = O.root_path(parent, i)
        for h in range(Hq):
            g = h // G
            rows = np.concatenate([V[g, :L], v_t[path, g]])
            np.testing.assert_allclose(o[i, h], rows.mean(axis=0), atol=1e-12)


def check_attn_chain_vs_library(seed=0, n=7):
    """A chain tree is causal attention over context + chain: compare with
    torch's scaled_dot_product_attention on CPU in float64."""
    rng = np.random.default_rng(seed)
    parent = [-1] + list(range(n - 1))
    K, V, L, q, k_t, v_t = attn_case(rng, n)
    Hq, Hkv, D = q.shape[1], K.shape[0], q.shape[2]
    G = Hq // Hkv
    scale = 0.41
    o = O.attn_tree_verify(K, V, L, q, k_t, v_t, parent, scale)
    keys = np.concatenate([K[:, :L], k_t.transpose(1, 0, 2)], axis=1)  # [Hkv, L+n, D]
    vals = np.concatenate([V[:, :L], v_t.transpose(1, 0, 2)], axis=1)
    keys = np.repeat(keys, G, axis=0)  # [Hq, L+n, D]
    vals = np.repeat(vals, G, axis=0)
    mask = np.arange(L + n)[None, :] < (L + 1 + np.arange(n))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.transpose(1, 0, 2)), torch.from_numpy(keys), torch.from_numpy(vals),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()
    np.testing.assert_allclose(o, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def check_relabel(seed=0, n=10):
    """Relabelling the nodes in another topological order permutes outputs."""
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    # a random topological order: repeatedly pick a random node whose parent is placed
    placed, order = {-1}, []
    while len(order) < n:
        ready = [i for i in range(n) if i not in order and parent[i] in placed]
        i = int(rng.choice(ready))
        order.append(i)
        placed.add(i)
    new_of = {old: new for new, old in enumerate(order)}
    parent2 = [-1 if parent[old] == -1 else new_of[parent[old]] for old in order]
    K, V, L, q, k_t, v_t = attn_case(rng, n)
    o1 = O.attn_tree_verify(K, V, L, q, k_t, v_t, parent, 0.3)
    o2 = O.attn_tree_verify(K, V, L, q[order], k_t[order], v_t[order], parent2, 0.3)
    np.testing.assert_allclose(o2, o1[order], atol=1e-12)
    S0, qg, kg, vg, al, be = gdn_case(rng, n)
    g1 = O.gdn_tree_verify(S0, qg, kg, vg, al, be, parent, 0.3)
    g2 = O.gdn_tree_verify(S0, qg[order], kg[order], vg[order], al[order], be[order], parent2, 0.3)
    np.testing.assert_allclose(g2, g1[order], atol=1e-12)


def check_hand_worked():
    with open(GOLDEN) as f:
        gold = json.load(f)
    a = gold["attention"]
    K = np.array(a["K_ctx"])[None]
    V = np.array(a["V_ctx"])[None]
    q = np.array(a["q"])[:, None]
    k_t = np.array(a["k_t"])[:, None]
    v_t = np.array(a["v_t"])[:, None]
    o = O.attn_tree_verify(K, V, a["L"], q, k_t, v_t, a["parent"], 1.0)
    np.testing.assert_allclose(o[:, 0], np.array(a["expected_o"]), atol=1e-12)
    g = gold["gdn"]
    S0 = np.array(g["S0"])[None]
    qg = np.array(g["q"])[:, None]
    kg = np.array(g["k"])[:, None]
    vg = np.array(g["v"])[:, None]
    al = np.array(g["alpha"])[:, None]
    be = np.array(g["beta"])[:, None]
    o = O.gdn_tree_verify(S0, qg, kg, vg, al, be, g["parent"], 1.0)
    np.testing.assert_allclose(o[:, 0], np.array(g["expected_o"]), atol=1e-12)
    S = O.commit_gdn(S0, kg, vg, al, be, [0, 1])
    np.testing.assert_allclose(S[0], np.array(g["expected_state_after_path_0_1"]), atol=1e-12)
    c = gold["accept"]
    path, alen, bonus = O.accept_path(c["parent"], c["tok"], c["greedy"])
    assert path == c["expected_path"] and alen == len(path) and bonus == c["expected_bonus"]


def _accept_by_enumeration(parent, tok, greedy):
    """Independent definition: list every root path, keep the agreeing ones,
    take the longest (lowest end node among equals)."""
    n = len(parent)
    children = [[c for c in range(n) if parent[c] == p] for p in range(n)]
    best = [0]

    def walk(path):
        nonlocal best
        if len(path) > len(best) or (len(path) == len(best) and path[-1] < best[-1]):
            best = list(path)
        for c in children[path[-1]]:
            if tok[c] == greedy[path[-1]]:
                walk(path + [c])

    walk([0])
    return best, len(best), greedy[best[-1]]


def _accept_by_walk(parent, tok, greedy):
    """The pages' walk: from the root, step to the child carrying the model's
    own token until there is none (trees with distinct sibling tokens)."""
    n = len(parent)
    path = [0]
    while True:
        nxt = [c for c in range(n) if parent[c] == path[-1] and tok[c] == greedy[path[-1]]]
        if not nxt:
            return path, len(path), greedy[path[-1]]
        path.append(nxt[0])


def check_accept_exhaustive(max_n=5, alphabet=2):
    for n in range(1, max_n + 1):
        for parents in itertools.product(*[range(i) for i in range(1, n)]):
            parent = [-1] + list(parents)
            siblings = {}
            for i in range(1, n):
                siblings.setdefault(parent[i], []).append(i)
            for tok_tail in itertools.product(range(alphabet), repeat=n - 1):
                tok = [0] + list(tok_tail)
                distinct = all(len({tok[c] for c in cs}) == len(cs) for cs in siblings.values())
                for greedy in itertools.product(range(alphabet), repeat=n):
                    got = O.accept_path(parent, tok, list(greedy))
                    assert got == _accept_by_enumeration(parent, tok, list(greedy)), (parent, tok, greedy)
                    if distinct:
                        assert got == _accept_by_walk(parent, tok, list(greedy))


def check_commit(seed=0, n=8):
    rng = np.random.default_rng(seed)
    parent = random_tree(rng, n)
    path = O.root_path(parent, n - 1)
    K, V, L, q, k_t, v_t = attn_case(rng, n)
    K2, V2 = K.copy(), V.copy()
    L2 = O.commit_attn(K2, V2, L, k_t, v_t, path)
    assert L2 == L + len(path)
    for j, node in enumerate(path):
        assert np.array_equal(K2[:, L + j], k_t[node]) and np.array_equal(V2[:, L + j], v_t[node])
    assert np.array_equal(K2[:, :L], K[:, :L]) and np.array_equal(K2[:, L2:], K[:, L2:])
    S0, qg, kg, vg, al, be = gdn_case(rng, n)
    S = O.commit_gdn(S0, kg, vg, al, be, path)
    Sd = S0.copy()
    for j in path:
        O.gdn_decode(Sd, qg[j], kg[j], vg[j], al[j], be[j], 1.0)
    np.testing.assert_allclose(S, Sd, atol=1e-13)


def check_tree_validation():
    for bad in ([0], [-1, 1], [-1, 0, 3], [-1, -1], list(range(-1, 16)) + [], [-1] + [0] * 64):
        with pytest.raises(ValueError):
            O.check_parent(bad)
    O.check_parent([-1] + list(range(15)))  # 16 nodes on one path is allowed
    O.check_parent([-1] + [0] * 63)


PINS = [check_attn_vs_sequential_decode, check_gdn_vs_sequential_decode, check_gdn_vs_chunked,
        check_gdn_closed_forms, check_attn_closed_forms, check_attn_chain_vs_library, check_relabel,
        check_hand_worked, check_accept_exhaustive, check_commit]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_bruteforce_more_seeds(seed):
    check_attn_vs_sequential_decode(seed, n=12)
    check_gdn_vs_sequential_decode(seed, n=12)
    check_gdn_vs_chunked(seed, n=16)
    check_relabel(seed)


def test_tree_validation():
    check_tree_validation()


def test_kv_row_bytes_shape_pin():
    """'Parallel requests', 'The shared KV pool': 64 KiB of attention KV a token
    for 16 full-attention layers, i.e. 4 KiB per layer = Hkv x D x {K,V} x bf16."""
    from speculative_tree_verify_masked_gb300.synth import SHAPES_27B as s, workload
    assert s.Hkv * s.D * 2 * 2 == 4096
    assert len(workload(3).attn_layers) == 16 and workload(3).n_layers == 64


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
def _fails(pins):
    for p in pins:
        try:
            p()
        except (AssertionError, ValueError):
            return True
    return False


def test_planted_decay_on_whole_update(monkeypatch):
    """Decay applied to the write term too: alpha (S(I - b k k^T) + b v k^T)."""
    orig = O.gdn_step

    def bad(S, q, k, v, alpha, beta):
        out = orig(S, q, k, v, np.ones_like(alpha), beta)
        return out * alpha[:, None, None]

    monkeypatch.setattr(O, "gdn_step", bad)
    assert _fails([check_gdn_vs_chunked, check_gdn_closed_forms, check_hand_worked])


def test_planted_sign_error(monkeypatch):
    orig = O.gdn_step

    def bad(S, q, k, v, alpha, beta):
        return orig(S, q, k, v, alpha, -beta)

    monkeypatch.setattr(O, "gdn_step", bad)
    assert _fails([check_gdn_vs_chunked, check_gdn_closed_forms, check_hand_worked])


def test_planted_transposed_state(monkeypatch):
    """Output read as S^T q instead of S q."""
    def bad(S0, q, k, v, alpha, beta, parent, scale):
        N, Hv = q.shape[0], S0.shape[0]
        o = np.zeros((N, Hv, S0.shape[1]))
        for i in range(N):
            S = O.gdn_path_state(S0, k, v, alpha, beta, O.root_path(parent, i))
            o[i] = scale * np.einsum("hkv,hk->hv", S, O._per_value_head(q[i], Hv))
        return o

    monkeypatch.setattr(O, "gdn_tree_verify", bad)
    assert _fails([check_gdn_vs_chunked, check_hand_worked])


def test_planted_head_mapping(monkeypatch):
    """Query head h read from KV head h % Hkv instead of h // (Hq/Hkv)."""
    orig = O.attn_tree_verify

    def bad(K, V, L, q, k_t, v_t, parent, scale):
        N, Hq, D = q.shape
        Hkv = K.shape[0]
        perm = [(h % Hkv) * (Hq // Hkv) + h // Hkv for h in range(Hq)]
        return orig(K, V, L, q[:, perm], k_t, v_t, parent, scale)[:, np.argsort(perm)]

    monkeypatch.setattr(O, "attn_tree_verify", bad)
    assert _fails([check_attn_chain_vs_library])


def test_planted_missing_self(monkeypatch):
    """A node that does not see its own key/value."""
    def bad(K, V, L, q, k_t, v_t, parent, scale):
        N, Hq, D = q.shape
        Hkv = K.shape[0]
        G = Hq // Hkv
        o = np.zeros((N, Hq, D))
        for i in range(N):
            path = O.root_path(parent, i)[:-1]
            for h in range(Hq):
                g = h // G
                keys = np.concatenate([K[g, :L], k_t[path, g]])
                vals = np.concatenate([V[g, :L], v_t[path, g]])
                if len(keys) == 0:
                    continue
                s = keys @ q[i, h] * scale
                w = np.exp(s - s.max())
                o[i, h] = (w / w.sum()) @ vals
        return o

    monkeypatch.setattr(O, "attn_tree_verify", bad)
    assert _fails([check_attn_closed_forms, check_hand_worked])


def test_planted_accept_off_by_one(monkeypatch):
    """Bonus token read at the parent of the path's end."""
    orig = O.accept_path

    def bad(parent, tok, greedy):
        path, a, bonus = orig(parent, tok, greedy)
        return path, a, int(greedy[parent[path[-1]]]) if a > 1 else bonus

    monkeypatch.setattr(O, "accept_path", bad)
    assert _fails([check_hand_worked, lambda: check_accept_exhaustive(max_n=3)])
