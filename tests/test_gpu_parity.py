"""GPU vs oracle on the five workloads, through the C ABI, in the launch
configuration the benchmark uses.  Accept paths, lengths and committed KV
rows must match bit for bit; outputs and committed states within the stated
tolerances.  At the full 64-layer sizes the GPU runs every layer and the
oracle checks a sample of layers (every layer is still checked for finite
outputs and bit-exact commits)."""
import pytest
import torch

import oracle.tree_verify as O
from gpu_helpers import check_close, check_state, f64, oracle_attn, oracle_commit_state, oracle_gdn, seq_slice
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu

# layers checked against the oracle at full size: (attention layers, GDN layers)
SAMPLED = {3: ([3, 63], [0, 1, 62]), 4: ([3, 63], [0, 62])}


def run_and_check(r: VerifyRound, attn_chk, gdn_chk):
    cfg = r.cfg
    S0 = {(li, s): r.gdn[li]["layer"].S[s].clone() for li in gdn_chk for s in range(cfg.n_seq)}
    r.run(reset_len=False)
    torch.cuda.synchronize()
    assert r.status() == 0, f"device status {r.status()}"
    path, acc, bonus = r.path.cpu(), r.acc_len.cpu(), r.bonus.cpu()
    tok, greedy = r.tok.cpu().tolist(), r.greedy.cpu().tolist()
    paths = []
    for s in range(cfg.n_seq):
        lo, hi = seq_slice(r, s)
        op, oa, ob = O.accept_path(r.parents[s], tok[lo:hi], greedy[lo:hi])
        assert op == r.expected_paths[s]
        assert path[s, :oa].tolist() == op and int(acc[s]) == oa and int(bonus[s]) == ob
        assert (path[s, oa:] == -1).all()
        paths.append(op)
    assert r.len.cpu().tolist() == [L + len(p) for L, p in zip(cfg.ctx_lens, paths)]
    for li in r.layers:
        out = r.attn[li]["out"] if li in r.attn else r.gdn[li]["out"]
        assert torch.isfinite(out.float()).all(), f"layer {li}: non-finite output"
    # committed KV rows are bit copies of the path's rows, in every attention layer
    for li, a in r.attn.items():
        for s in range(cfg.n_seq):
            lo, _ = seq_slice(r, s)
            L = cfg.ctx_lens[s]
            idx = torch.tensor([lo + n for n in paths[s]], device=a["k_t"].device)
            assert torch.equal(a["layer"].K[s][:, L:L + len(paths[s])], a["k_t"][idx].transpose(0, 1))
            assert torch.equal(a["layer"].V[s][:, L:L + len(paths[s])], a["v_t"][idx].transpose(0, 1))
    for li in attn_chk:
        for s in range(cfg.n_seq):
            lo, hi = seq_slice(r, s)
            check_close(r.attn[li]["out"][lo:hi], oracle_attn(r, li, s), f"attn layer {li} seq {s}")
    for li in gdn_chk:
        for s in range(cfg.n_seq):
            lo, hi = seq_slice(r, s)
            check_close(r.gdn[li]["out"][lo:hi], oracle_gdn(r, li, s, S0[(li, s)]), f"gdn layer {li} seq {s}")
            check_state(r.gdn[li]["layer"].S[s], oracle_commit_state(r, li, s, S0[(li, s)], paths[s]),
                        f"gdn layer {li} seq {s} committed state")


@pytest.mark.parametrize("cfg_id", [0, 1, 2])
def test_parity_layer_pair(cfg_id):
    r = VerifyRound(synth.workload(cfg_id))
    run_and_check(r, list(r.attn), list(r.gdn))


@pytest.mark.parametrize("cfg_id", [3, 4])
def test_parity_full_stack(cfg_id):
    r = VerifyRound(synth.workload(cfg_id))
    attn_chk, gdn_chk = SAMPLED[cfg_id]
    run_and_check(r, attn_chk, gdn_chk)


def test_graph_replay_matches_eager():
    """The captured round produces the same bits as the eager one."""
    cfg = synth.workload(1)
    r = VerifyRound(cfg)
    g = r.capture()
    outs = {li: (r.attn[li]["out"] if li in r.attn else r.gdn[li]["out"]).clone() for li in r.layers}
    r2 = VerifyRound(cfg)
    r2.run()
    torch.cuda.synchronize()
    for li in r.layers:
        o2 = r2.attn[li]["out"] if li in r2.attn else r2.gdn[li]["out"]
        assert torch.equal(outs[li], o2)
    g.replay()
    torch.cuda.synchronize()
    assert r.status() == 0


def test_packed_host_io_gives_the_same_round():
    """A round whose host inputs live in one packed buffer (and whose results
    come back in another) gives the bits of the ordinary round, also when the
    packed inputs are refilled from a pinned host copy."""
    cfg = synth.workload(2)
    plain = VerifyRound(cfg)
    plain.run()
    torch.cuda.synchronize()
    packed = VerifyRound(cfg)
    io_in, io_out = packed.pack_io()
    host_in = io_in.cpu().pin_memory()
    io_in.zero_()
    io_in.copy_(host_in, non_blocking=True)
    packed.run()
    host_out = io_out.cpu()
    torch.cuda.synchronize()
    assert packed.status() == 0 and plain.status() == 0
    for li in plain.layers:
        a = plain.attn[li]["out"] if li in plain.attn else plain.gdn[li]["out"]
        b = packed.attn[li]["out"] if li in packed.attn else packed.gdn[li]["out"]
        assert torch.equal(a, b), li
    for name in ("path", "acc_len", "bonus", "len"):
        assert torch.equal(getattr(plain, name), getattr(packed, name)), name
    # the read-back buffer holds the accepted path first
    n = cfg.n_seq * 16
    assert torch.equal(host_out[:4 * n].view(torch.int32).view(cfg.n_seq, 16), plain.path.cpu())
