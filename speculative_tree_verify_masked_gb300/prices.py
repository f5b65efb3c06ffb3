"""Verify-cost table: microseconds per verify round against tree size,
context length and sequence count.

The tree cutter sizes each round's tree to maximise expected tokens per
millisecond on the measured cost of verifying it ("One request, end to end"
2.6), from a price file per model and device ("Adding a model", data files).
This module measures that cost on the GPU it runs on -- whole rounds of the
64-layer mixer stack (verify of every layer, accept, commit) replayed from
the per-shape CUDA graphs of `graphs.ShapeGraphs` and timed with CUDA events
-- writes it as JSON, and reads it back for lookups (`VerifyCost`).

Measure:  python -m speculative_tree_verify_masked_gb300.prices --out FILE
"""
from __future__ import annotations

import argparse
import bisect
import json
import statistics

STACK = "64-layer mixer stack (48 GDN + 16 attention; Hq 24, Hkv 4, D 256; Hk 16, Hv 48, dk = dv = 128; bf16)"
WIDTHS = (1, 2, 4, 8, 12, 16, 24, 32, 48, 64)
LENS = (4096, 16384, 65536, 131072)
N_SEQS = (1, 2, 4)


class VerifyCost:
    """Lookups in a measured table.  `us(nodes, L, n_seq)` interpolates
    linearly in the node count between measured widths and linearly in the
    context length between (or beyond) measured lengths; the sequence count
    must be one that was measured (each sequence has a tree of `nodes`)."""

    def __init__(self, table: dict):
        self.table = table
        self.grid: dict[int, dict[int, list[tuple[int, float]]]] = {}
        for e in table["entries"]:
            self.grid.setdefault(int(e["n_seq"]), {}).setdefault(int(e["L"]), []).append(
                (int(e["nodes"]), float(e["us_median"])))
        for by_len in self.grid.values():
            for pts in by_len.values():
                pts.sort()

    @classmethod
    def load(cls, path: str) -> "VerifyCost":
        with open(path) as f:
            return cls(json.load(f))

    @staticmethod
    def _interp(pts, x):
        xs = [p[0] for p in pts]
        if len(pts) == 1:
            return pts[0][1]
        i = bisect.bisect_left(xs, x)
        i = min(max(i, 1), len(pts) - 1)
        (x0, y0), (x1, y1) = pts[i - 1], pts[i]
        return y0 + (y1 - y0) * (x - x0) / (x1 - x0)

    def us(self, nodes: int, L: int, n_seq: int = 1) -> float:
        if n_seq not in self.grid:
            raise KeyError(f"no measurements for {n_seq} sequences (have {sorted(self.grid)})")
        by_len = self.grid[n_seq]
        lo_n = max(min(p[0] for p in pts) for pts in by_len.values())
        hi_n = min(max(p[0] for p in pts) for pts in by_len.values())
        if not lo_n <= nodes <= hi_n:
            raise ValueError(f"{nodes} nodes is outside the measured widths {lo_n}..{hi_n}")
        per_len = sorted((L_, self._interp(pts, nodes)) for L_, pts in by_len.items())
        return self._interp(per_len, L)


def stack_workload(L: int, n_seq: int, width: int):
    """The 64-layer stack with n_seq sequences at context L, each with a
    merged tree of `width` nodes (a 16-node drafter chain plus branches)."""
    from . import synth
    return synth.Workload(f"{STACK}, {n_seq} x L {L}, {width}-node trees", 700 + n_seq, synth.SHAPES_27B,
                          [L] * n_seq, [("merged", width, min(16, width))] * n_seq, 64,
                          attn_layers=[i for i in range(64) if i % 4 == 3], accept=[("random",)] * n_seq)


def _time_widths(r, widths, reps, warmup):
    """Median and minimum us per round for each width (prefix trees), from
    a fresh set of per-shape graphs on r."""
    import torch

    from .graphs import ShapeGraphs, prefix_trees

    sg = ShapeGraphs(r)
    out = {}
    for w in widths:
        parents = prefix_trees(r.parents, w)
        tok = [x for t in r.trees for x in t[1][:w]]
        greedy = [x for t in r.trees for x in t[2][:w]]
        key = sg.load(parents, tok, greedy)
        for _ in range(warmup):
            sg.replay(key)
        ts = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            sg.replay(key)
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1000.0)
        if sg.status(key) != 0:
            raise RuntimeError(f"round status {sg.status(key)} at {w} nodes")
        out[w] = (statistics.median(ts), min(ts))
    return out


def split_candidates(n_seq: int, lens, sms: int) -> list[int]:
    """Splits worth measuring: the makespan-model choice for a few tree
    widths at each length, and round powers of two."""
    from . import synth
    from .round import auto_split
    sh = synth.SHAPES_27B
    c = {auto_split([L] * n_seq, [w] * n_seq, sh.Hq, sh.Hkv, sms) for L in lens for w in (8, 24, 64)}
    return sorted(c | {2048, 4096, 8192})


def choose_split(n_seq: int, lens=(16384, 131072), widths=(8, 24, 64), reps: int = 8, log=print):
    """The plan's split is fixed for a deployment (verify and decode must
    share it), so it is chosen once per sequence count: the candidate with
    the smallest geometric-mean round cost over a few widths and lengths."""
    import math

    import torch

    from .round import VerifyRound

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cands = split_candidates(n_seq, lens, sms)
    score = {c: 0.0 for c in cands}
    sweep = []
    for L in lens:
        r = VerifyRound(stack_workload(L, n_seq, max(widths)), split=cands[0])
        for c in cands:
            r.set_split(c)
            for w, (med, _) in _time_widths(r, widths, reps, 2).items():
                score[c] += math.log(med)
                sweep.append(dict(n_seq=n_seq, split=c, L=L, nodes=w, us_median=round(med, 2)))
                log(json.dumps(sweep[-1]))
        del r
        torch.cuda.empty_cache()
    return min(cands, key=lambda c: (score[c], -c)), sweep


def measure(lens=LENS, widths=WIDTHS, n_seqs=N_SEQS, reps: int = 20, warmup: int = 3, split=None, log=print) -> dict:
    import torch

    from .round import VerifyRound

    widths = sorted(set(widths))
    entries, sweeps, splits = [], [], {}
    for n_seq in n_seqs:
        if split is None:
            splits[n_seq], sw = choose_split(n_seq, log=log)
            sweeps += sw
        else:
            splits[n_seq] = split
        for L in lens:
            r = VerifyRound(stack_workload(L, n_seq, widths[-1]), split=splits[n_seq])
            for w, (med, mn) in _time_widths(r, widths, reps, warmup).items():
                e = dict(n_seq=n_seq, nodes=w, L=L, split=r.split, us_median=round(med, 2), us_min=round(mn, 2))
                entries.append(e)
                log(json.dumps(e))
            del r
            torch.cuda.empty_cache()
    return dict(stack=STACK, device=torch.cuda.get_device_name(),
                sm_count=torch.cuda.get_device_properties(0).multi_processor_count,
                timing=(f"whole rounds (tree prepare, 64 layer verifies, accept, commit; lengths reset in the graph) "
                        f"replayed from one CUDA graph per tree shape; CUDA events around each of {reps} replays "
                        f"after {warmup} warm-up replays; median and minimum"),
                trees="each sequence's tree is the first `nodes` nodes of a 64-node merged tree "
                      "(16-node drafter chain plus branches)",
                split=("one plan split per sequence count (verify and decode must share it): "
                       + ("the candidate with the smallest geometric-mean round cost in `split_sweep`"
                          if split is None else "given")),
                splits={str(k): v for k, v in splits.items()}, entries=entries, split_sweep=sweeps)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--out", required=True)
    ap.add_argument("--lens", type=int, nargs="+", default=list(LENS))
    ap.add_argument("--widths", type=int, nargs="+", default=list(WIDTHS))
    ap.add_argument("--n-seq", type=int, nargs="+", default=list(N_SEQS))
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--split", type=int, default=None, help="plan split for every entry (default: measured choice)")
    a = ap.parse_args(argv)
    table = measure(a.lens, a.widths, a.n_seq, a.reps, split=a.split)
    with open(a.out, "w") as f:
        json.dump(table, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
