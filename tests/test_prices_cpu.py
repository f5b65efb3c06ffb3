"""Host logic of the per-shape graphs and the verify-cost table (no GPU)."""
import json
import os

import pytest

from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.graphs import prefix_trees, shape_key
from speculative_tree_verify_masked_gb300.prices import LENS, N_SEQS, WIDTHS, VerifyCost, stack_workload

PRICE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "speculative_tree_verify_masked_gb300", "prices", "mixer64.gb300.json")


def test_shape_key_and_prefixes():
    cfg = stack_workload(4096, 2, 64)
    parents = [synth.tree_and_tokens(cfg, q)[0] for q in range(2)]
    assert shape_key(parents) == (2, 128, 64)
    for w in (1, 2, 16, 17, 40, 64):
        pre = prefix_trees(parents, w)
        assert shape_key(pre) == (2, 2 * w, w)
        for p in pre:
            assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, len(p)))
    assert shape_key([[-1], [-1, 0, 0]]) == (2, 4, 3)
    # the widest prefix of the drafter chain: the first 16 nodes form a chain
    assert prefix_trees(parents, 16)[0] == [-1] + list(range(15))


def bilinear_table():
    """A table whose cost is bilinear in nodes and L, so interpolation is exact."""
    f = lambda n, L, s: 50.0 * s + 3.0 * n + 0.01 * L * s + 0.0005 * n * L
    entries = [dict(n_seq=s, nodes=n, L=L, split=512, us_median=f(n, L, s), us_min=f(n, L, s))
               for s in (1, 2) for L in (4096, 16384, 65536) for n in (1, 8, 32, 64)]
    return {"entries": entries}, f


def test_interpolation_is_exact_for_bilinear_costs():
    table, f = bilinear_table()
    vc = VerifyCost(table)
    for s in (1, 2):
        for n in (1, 5, 8, 20, 32, 50, 64):
            for L in (4096, 10000, 16384, 40000, 65536, 131072):  # 131072: linear beyond the last length
                assert vc.us(n, L, s) == pytest.approx(f(n, L, s), rel=1e-12), (n, L, s)


def test_lookup_errors():
    table, _ = bilinear_table()
    vc = VerifyCost(table)
    with pytest.raises(KeyError):
        vc.us(8, 4096, 3)
    with pytest.raises(ValueError):
        vc.us(65, 4096, 1)
    with pytest.raises(ValueError):
        vc.us(0, 4096, 1)


@pytest.mark.skipif(not os.path.exists(PRICE_FILE), reason="no measured price file")
def test_measured_price_file():
    """The committed table covers its grid, and cost grows with the context
    (the KV stream) and with the tree at long context."""
    with open(PRICE_FILE) as f:
        table = json.load(f)
    got = {(e["n_seq"], e["nodes"], e["L"]) for e in table["entries"]}
    assert got == {(s, n, L) for s in N_SEQS for n in WIDTHS for L in LENS}
    assert all(0 < e["us_min"] <= e["us_median"] for e in table["entries"])
    vc = VerifyCost(table)
    for s in N_SEQS:
        for n in WIDTHS:
            costs = [vc.us(n, L, s) for L in LENS]
            assert all(b > a for a, b in zip(costs, costs[1:])), (s, n, costs)
        assert vc.us(64, LENS[-1], s) > vc.us(1, LENS[-1], s)
    for n in WIDTHS:
        assert vc.us(n, LENS[-1], 4) > vc.us(n, LENS[-1], 1)
