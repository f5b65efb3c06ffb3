"""tv_attn_tree_verify_static (scratch in a fixed device array) against the
ordinary tv_attn_tree_verify (caller-supplied workspace), both called
through the C ABI on the same inputs.

The static call runs the same kernels with the same plan, so its output must
be the workspace call's bit for bit.  Every call shares the one array and
finds the previous call's records in it; before each checked call another
workload (different lengths, trees and values) goes through the array, so a
read of a record not written earlier in the same call would see foreign data
and change the bits.  Collected last so that it also runs after every other
GPU test in the same process."""
from __future__ import annotations

import pytest
import torch

from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu

CHECKED = [1, 2, 4]
# the workload that goes through the array before each checked call
POLLUTER = {1: 4, 2: 1, 4: 2}


def _first_attn_layer(cfg):
    return next(li for li in range(cfg.n_layers) if cfg.is_attn(li))


@pytest.fixture(scope="module")
def rounds():
    out = {}
    for cfg_id in CHECKED:
        cfg = synth.workload(cfg_id)
        li = _first_attn_layer(cfg)
        r = VerifyRound(cfg, layers=[li])
        need = B.tv_attn_workspace_bytes(r.plan, r.attn[li]["layer"], cfg.n_seq, r.tree.n_max, r.max_len)
        assert 0 < need <= B.tv_attn_static_scratch_bytes()
        r.prepare()
        r.verify_layer(li)  # the workspace call
        torch.cuda.synchronize()
        assert r.status() == 0
        out[cfg_id] = (r, li, r.attn[li]["out"].clone())
    return out


def _static(r, li):
    a = r.attn[li]
    out = torch.full_like(a["out"], float("nan"))
    B.tv_attn_tree_verify_static(r.plan, a["layer"], r.tree, r.len, r.max_len, a["q"], a["k_t"], a["v_t"], out,
                                 r.attn_scale)
    return out


@pytest.mark.parametrize("cfg_id", CHECKED)
def test_static_scratch_matches_workspace_call(rounds, cfg_id):
    r, li, ref = rounds[cfg_id]
    pr, pli, pref = rounds[POLLUTER[cfg_id]]
    for call in range(2):  # two calls in a row, each after a foreign workload
        other = _static(pr, pli)
        out = _static(r, li)
        torch.cuda.synchronize()
        assert r.status() == 0 and pr.status() == 0
        assert torch.equal(other, pref), f"workload {POLLUTER[cfg_id]} static call {call}"
        assert torch.equal(out, ref), f"workload {cfg_id} layer {li} static call {call}: not the workspace bits"


def test_static_scratch_rejects_oversized_request():
    cfg = synth.workload(2)
    li = _first_attn_layer(cfg)
    r = VerifyRound(cfg, layers=[li])
    a = r.attn[li]
    small = B.plan(64)  # one partial state per 64 positions: far above the fixed scratch
    need = B.tv_attn_workspace_bytes(small, a["layer"], cfg.n_seq, r.tree.n_max, r.max_len)
    assert need > B.tv_attn_static_scratch_bytes()
    r.prepare()
    torch.cuda.synchronize()
    out = torch.full_like(a["out"], 7.0)
    with pytest.raises(B.TvError) as e:
        B.tv_attn_tree_verify_static(small, a["layer"], r.tree, r.len, r.max_len, a["q"], a["k_t"], a["v_t"], out,
                                     r.attn_scale)
    assert e.value.code == 11  # TV_ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call must enqueue nothing"
    assert r.status() == 0
