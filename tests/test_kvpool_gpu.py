"""KV pool on the GPU ("Parallel requests", "The shared KV pool").

Rounds on caches whose address space is reserved whole and whose pages are
committed as the context grows give the same bits as rounds on static
caches: outputs, accepted paths, committed cache rows, states and lengths,
round after round across a page boundary.  The pool's committed bytes are
the pages the committed rows touch, fresh pages read as zeros, and giving
rows back returns exactly the pages no kept row touches.
"""
import pytest
import torch

from gpu_helpers import check_close, check_state, oracle_attn, oracle_commit_state, oracle_gdn, seq_slice
from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import VerifyRound

pytestmark = pytest.mark.gpu


def touched_pages(page, heads, head_stride, row_bytes, rows):
    """Pages of a [heads][cap][dim] range that rows [0, rows) of some head touch."""
    pages = set()
    if rows <= 0:
        return pages
    for h in range(heads):
        lo = h * head_stride
        hi = lo + rows * row_bytes
        pages |= set(range(lo // page, -(-hi // page)))
    return pages


def expected_committed(r, page, rows_of):
    sh = r.cfg.shapes
    es = torch.empty((), dtype=sh.kv_dtype).element_size()
    n = 0
    for _ in r.attn:
        for q in range(r.cfg.n_seq):
            n += 2 * len(touched_pages(page, sh.Hkv, r.cap * sh.D * es, sh.D * es, rows_of(q)))
    return n * page


def test_pooled_rounds_equal_static_rounds():
    L0 = 4077  # bf16, D = 256: 4096 rows of a head per 2 MiB page
    cfg = synth.Workload("kv pool", 960, synth.SHAPES_27B, [L0, 1500], [("merged", 16, 11), ("merged", 12, 8)], 2,
                         attn_layers=[0], accept=[("random",)] * 2)
    pool = B.KVPool(0)
    try:
        margin = B.TV_MAX_PATH
        # cap = 8192 rows: each head's rows start on a page, so crossing row
        # 4096 needs a page of its own
        rs = VerifyRound(cfg, split=512, max_len=8192 - 64)
        rp = VerifyRound(cfg, split=512, max_len=8192 - 64, kv_pool=pool, kv_margin=margin)
        assert rp.cap == 8192
        page = pool.page_bytes
        assert page >= 2 << 20
        sh = cfg.shapes
        es = 2
        assert pool.reserved_bytes == 2 * cfg.n_seq * (-(-sh.Hkv * rp.cap * sh.D * es // page) * page)
        lens = list(cfg.ctx_lens)
        assert pool.committed_bytes == expected_committed(rp, page, lambda q: min(rp.cap, lens[q] + margin))
        # rows past the context in committed pages read as zeros
        K0 = rp.attn[0]["layer"].K[0]
        assert not K0[:, L0:L0 + margin].view(torch.int16).any()
        start = pool.committed_bytes
        for rnd in range(6):
            rp.commit_kv()
            lens = rp.len.tolist()
            assert pool.committed_bytes == expected_committed(rp, page, lambda q: min(rp.cap, lens[q] + margin))
            S_before = {(li, q): S.clone() for li, g in rp.gdn.items() for q, S in enumerate(g["layer"].S)}
            rs.run(reset_len=False)
            rp.run(reset_len=False)
            torch.cuda.synchronize()
            assert rs.status() == 0 and rp.status() == 0
            if rnd in (0, 5):  # pooled rounds against the oracle, before and after the page boundary
                for q, L in enumerate(lens):
                    lo, hi = seq_slice(rp, q)
                    path = rp.path[q, :int(rp.acc_len[q])].tolist()
                    for li in rp.attn:
                        check_close(rp.attn[li]["out"][lo:hi], oracle_attn(rp, li, q, L=L),
                                    f"pooled round {rnd} attention seq {q}")
                    for li in rp.gdn:
                        S0 = S_before[(li, q)]
                        check_close(rp.gdn[li]["out"][lo:hi], oracle_gdn(rp, li, q, S0=S0),
                                    f"pooled round {rnd} GDN seq {q}")
                        check_state(rp.gdn[li]["layer"].S[q], oracle_commit_state(rp, li, q, S0, path),
                                    f"pooled round {rnd} state seq {q}")
            assert torch.equal(rs.len, rp.len), rnd
            for name in ("path", "acc_len", "bonus"):
                assert torch.equal(getattr(rs, name), getattr(rp, name)), (rnd, name)
            for li in rs.attn:
                assert torch.equal(rs.attn[li]["out"], rp.attn[li]["out"]), (rnd, li)
                for q, L in enumerate(rs.len.tolist()):
                    for name in ("K", "V"):
                        a = getattr(rs.attn[li]["layer"], name)[q][:, :L]
                        b = getattr(rp.attn[li]["layer"], name)[q][:, :L]
                        assert torch.equal(a, b), (rnd, li, q, name)
            for li in rs.gdn:
                assert torch.equal(rs.gdn[li]["out"], rp.gdn[li]["out"]), (rnd, li)
                for a, b in zip(rs.gdn[li]["layer"].S, rp.gdn[li]["layer"].S):
                    assert torch.equal(a, b), (rnd, li)
        rp.commit_kv()
        lens = rp.len.tolist()
        assert lens[0] + margin > 4096
        assert pool.committed_bytes == expected_committed(rp, page, lambda q: min(rp.cap, lens[q] + margin))
        assert pool.committed_bytes - start == 2 * sh.Hkv * page  # every head of sequence 0's K and V
        # give back everything past the first context: the pages no kept row touches
        for a in rp.attn.values():
            for q in range(cfg.n_seq):
                pool.release_rows(a["layer"].K[q], cfg.ctx_lens[q])
                pool.release_rows(a["layer"].V[q], cfg.ctx_lens[q])
        assert pool.committed_bytes == expected_committed(rp, page, lambda q: cfg.ctx_lens[q])
        del rp
    finally:
        torch.cuda.synchronize()
        pool.close()
