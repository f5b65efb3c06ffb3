"""Attention front end on the GPU ("Adding a model", "What is still
specific to Qwen3.8": attention with a gated output and partial rotary):
tv_attn_rope at each row's logical position and the gate fused into the
attention epilogue, against the fp64 oracle (oracle/attn_front.py), and the
bit-for-bit rule that a verified row equals the same token decoded after its
ancestors (rotated at the same position, gated by the same function)."""
import numpy as np
import pytest
import torch

import oracle.attn_front as F
import oracle.tree_verify as O
from gpu_helpers import check_close, f64, seq_slice
from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu

# (rotated dimensions, rotary base) per workload: partial rotary on the 27B-shaped heads
ROPE = {0: (32, 10000.0), 1: (64, 1.0e7), 2: (64, 1.0e7)}


def bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


def gate_like(t, seed):
    g = torch.Generator(device=t.device).manual_seed(seed)
    return torch.randn(t.shape, generator=g, device=t.device, dtype=torch.float32).to(t.dtype)


def front_verify(r, li, rot, theta, gate):
    a = r.attn[li]
    q = torch.empty_like(a["q"])
    k = torch.empty_like(a["k_t"])
    out = torch.empty_like(a["out"])
    B.tv_attn_rope(a["layer"], r.tree, r.cfg.n_seq, r.len, r.max_len, rot, theta, a["q"], a["k_t"], q, k)
    B.tv_attn_tree_verify_gated(r.plan, a["layer"], r.tree, r.len, r.max_len, q, k, a["v_t"], gate, out,
                                r.attn_scale, r.ws)
    torch.cuda.synchronize()
    assert r.status() == 0
    return q, k, out


@pytest.mark.parametrize("cfg_id", [0, 1, 2])
def test_front_end_matches_oracle(cfg_id):
    r = VerifyRound(synth.workload(cfg_id))
    r.prepare()
    li = next(iter(r.attn))
    a = r.attn[li]
    rot, theta = ROPE[cfg_id]
    gate = gate_like(a["q"], 4242 + cfg_id)
    q, k, out = front_verify(r, li, rot, theta, gate)
    for s in range(r.cfg.n_seq):
        lo, hi = seq_slice(r, s)
        L = int(r.cfg.ctx_lens[s])
        ref_o, ref_k, ref_v = F.attn_front_tree_verify(
            f64(a["layer"].K[s][:, :L]), f64(a["layer"].V[s][:, :L]), L, f64(a["q"][lo:hi]), f64(a["k_t"][lo:hi]),
            f64(a["v_t"][lo:hi]), f64(gate[lo:hi]), r.parents[s], r.attn_scale, rot, theta)
        check_close(out[lo:hi], ref_o, f"gated output seq {s}")
        check_close(k[lo:hi], ref_k, f"rotated tree keys seq {s}")
        depth = O.depths(r.parents[s])
        ref_q = np.stack([F.rope(f64(a["q"][lo + i]), L + depth[i], rot, theta) for i in range(hi - lo)])
        check_close(q[lo:hi], ref_q, f"rotated queries seq {s}")
    # in place gives the same bits
    q2, k2 = a["q"].clone(), a["k_t"].clone()
    B.tv_attn_rope(a["layer"], r.tree, r.cfg.n_seq, r.len, r.max_len, rot, theta, q2, k2, q2, k2)
    torch.cuda.synchronize()
    assert torch.equal(bits(q2), bits(q)) and torch.equal(bits(k2), bits(k))


def decode_front_rows(r, li, seq, path, rot, theta, gate):
    """Decode `path` token by token through the front end on a copy of the
    cache of `seq`; returns (output rows, rotated key rows, the cache copy)."""
    a = r.attn[li]
    lo, _ = seq_slice(r, seq)
    K, V = a["layer"].K[seq].clone(), a["layer"].V[seq].clone()
    layer1 = B.AttnLayer([K], [V], r.cfg.shapes.Hq)
    len1 = torch.tensor([r.cfg.ctx_lens[seq]], dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    wsb = B.tv_attn_workspace_bytes(r.plan, layer1, 1, 1, r.cap)
    ws = torch.empty(max(16, wsb) // 4 + 4, dtype=torch.float32, device="cuda") if wsb else None
    rows, krows = [], []
    for node in path:
        i = lo + node
        q1, k1 = torch.empty_like(a["q"][i:i + 1]), torch.empty_like(a["k_t"][i:i + 1])
        B.tv_attn_rope(layer1, None, 1, len1, r.cap, rot, theta, a["q"][i:i + 1].clone(), a["k_t"][i:i + 1].clone(),
                       q1, k1, status)
        out = torch.empty_like(q1)
        B.tv_attn_decode_gated(r.plan, layer1, 1, len1, r.cap, q1, k1, a["v_t"][i:i + 1].clone(),
                               gate[i:i + 1].clone(), out, r.attn_scale, ws, status)
        B.tv_len_advance(len1, None, 1, 1)
        rows.append(out)
        krows.append(k1)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    return torch.cat(rows), torch.cat(krows), K


@pytest.mark.parametrize("cfg_id", [0, 2])
def test_front_end_verify_rows_equal_decode_rows(cfg_id):
    r = VerifyRound(synth.workload(cfg_id))
    r.prepare()
    li = next(iter(r.attn))
    rot, theta = ROPE[cfg_id]
    gate = gate_like(r.attn[li]["q"], 777 + cfg_id)
    _, k, out = front_verify(r, li, rot, theta, gate)
    parents = r.parents[0]
    leaves = [i for i in range(len(parents)) if i not in parents]
    rng = np.random.default_rng(5 + cfg_id)
    ends = [r.expected_paths[0][-1]] + list(rng.choice(leaves, size=min(3, len(leaves)), replace=False))
    L = int(r.cfg.ctx_lens[0])
    for end in ends:
        path = O.root_path(parents, int(end))
        dec, dk, Kc = decode_front_rows(r, li, 0, path, rot, theta, gate)
        assert torch.equal(bits(dec), bits(out[path])), f"path {path}: verified row != decoded row"
        assert torch.equal(bits(dk), bits(k[path])), f"path {path}: rotated key differs"
        # the keys decode appended are the rows a commit of this path would copy
        assert torch.equal(bits(Kc[:, L:L + len(path)]), bits(k[path].transpose(0, 1)))
