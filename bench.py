#!/usr/bin/env python
"""Benchmark of one speculative tree-verify round on GB300.

A step is one round of the whole hot path over the 64-layer mixer stack
(48 Gated DeltaNet + 16 attention layers, 131,072-token bf16 KV context, a
32-node draft tree): tree prepare, every layer's verify, the accept walk and
the commit, captured in one CUDA graph and replayed.  Inputs (8.6 GB of KV
streamed per round) are far larger than L2, so no flush is needed between
rounds.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 0..4] [--impl ours|reference]

Under torchrun every rank runs its own replica of the workload (the round has
no exchange step), timed between barriers, max over ranks; rank 0 prints one
JSON line.  --impl reference times the CPU oracle (the fp64 definition) on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "verify-round µs & tree nodes/s (64-layer mixer stack); HBM GB/s vs GB300 peak"
UNIT = "tree nodes/s"
SPEC_HBM_GBS = 8000.0  # the GB300 HBM3e figure the target is quoted against


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes (every byte the round must move at least once)
# ---------------------------------------------------------------------------
def attn_layer_bytes(cfg, n_nodes_per_seq):
    s = cfg.shapes
    e = 2 if s.kv_dtype == torch.bfloat16 else 4
    total = 0
    for L, n in zip(cfg.ctx_lens, n_nodes_per_seq):
        total += 2 * s.Hkv * L * s.D * e  # K and V context rows
        total += 2 * n * s.Hq * s.D * e  # q in, out
        total += 2 * n * s.Hkv * s.D * e  # the nodes' own k, v
    return total


def round_bytes(cfg, n_nodes_per_seq, acc_lens):
    s = cfg.shapes
    e = 2 if s.kv_dtype == torch.bfloat16 else 4
    n_attn = len(cfg.attn_layers)
    n_gdn = cfg.n_layers - n_attn
    total = n_attn * attn_layer_bytes(cfg, n_nodes_per_seq)
    state = 4 * s.Hv * s.dv * s.dk
    for n, a in zip(n_nodes_per_seq, acc_lens):
        # GDN: state read by verify, read + written by commit; node inputs and outputs
        total += n_gdn * (3 * state + n * (2 * s.Hk * s.dk * e + 2 * s.Hv * s.dv * e + 2 * s.Hv * 4))
        # attention commit: the path's k, v rows read and written
        total += n_attn * 2 * 2 * a * s.Hkv * s.D * e
    return total


# DRAM bytes (read + write) of one attention verify call (split + tail
# kernels) from a single-pass ncu capture at full size on a GB300, keyed by
# workload name; the capture command and the figures are in
# profiles/attn_traffic_64layer_128k.md.  Update together with the kernels.
MEASURED_TRAFFIC = {
    "64-layer mixer stack (48 GDN + 16 attention), L 131072, 32-node tree": 537351424 + 21152768 + 1061888,
}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.4)

    def stop(self, t0: float, t1: float):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 10:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def ts(p):
            try:
                return datetime.datetime.strptime(p, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except Exception:
                return 0.0

        inside = [r for r in rows if t0 - 0.15 <= ts(r[1]) <= t1 + 0.15] or rows
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# oracle sample (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_inputs(cfg, device):
    """Inputs of one 4-layer block (3 GDN + 1 attention) of sequence 0."""
    from speculative_tree_verify_masked_gb300 import synth
    parent, tok, greedy, _ = synth.tree_and_tokens(cfg, 0)
    n = len(parent)
    L = cfg.ctx_lens[0]
    attn_li = cfg.attn_layers[0]
    gdn_lis = [i for i in range(cfg.n_layers) if not cfg.is_attn(i)][:3]
    a = synth.attn_layer_inputs(cfg, attn_li, 0, n, L + 64, device)
    gs = [synth.gdn_layer_inputs(cfg, li, 0, n, device) for li in gdn_lis]
    return parent, tok, greedy, a, gs


def time_oracle(cfg, inputs, attn_kv_heads, attn_nodes, gdn_heads, gdn_nodes):
    """Run the oracle on a sample of one 4-layer block of sequence 0:
    attention for `attn_kv_heads` KV heads over the first `attn_nodes` tree
    nodes (a prefix of a topologically ordered tree is a tree) with the full
    context, and GDN for `gdn_heads` value heads over the first `gdn_nodes`
    nodes of each of the block's GDN layers, plus the accept walk and the
    commit.  The round estimate scales attention by query rows (each costs
    one pass over the context) and GDN by (recurrence steps x value heads).
    Returns (seconds, estimated seconds per round, attention seconds, GDN seconds)."""
    import numpy as np

    import oracle.tree_verify as O
    s = cfg.shapes
    parent, tok, greedy, a, gs = inputs
    n = len(parent)
    L = cfg.ctx_lens[0]
    G = s.Hq // s.Hkv
    d = lambda t: t.detach().double().cpu().numpy()
    ka, na, gh, ng = attn_kv_heads, attn_nodes, gdn_heads, gdn_nodes
    K = d(a["K"][:ka, :L]); V = d(a["V"][:ka, :L])
    q = d(a["q"][:na, :ka * G]); kt = d(a["k_t"][:na, :ka]); vt = d(a["v_t"][:na, :ka])
    kh = max(1, gh // (s.Hv // s.Hk))
    gin = [(d(g["S0"][:gh]), d(g["q"][:ng, :kh]), d(g["k"][:ng, :kh]), d(g["v"][:ng, :gh]),
            d(g["alpha"][:ng, :gh]), d(g["beta"][:ng, :gh])) for g in gs]
    t0 = time.perf_counter()
    O.attn_tree_verify(K, V, L, q, kt, vt, parent[:na], 1.0 / math.sqrt(s.D))
    t1 = time.perf_counter()
    path, alen, bonus = O.accept_path(parent, tok, greedy)
    Kc, Vc = np.zeros((ka, L + 16, s.D)), np.zeros((ka, L + 16, s.D))
    O.commit_attn(Kc, Vc, L, d(a["k_t"][:, :ka]), d(a["v_t"][:, :ka]), path)
    sub_path = [x for x in path if x < ng]
    for (S0, qg, kg, vg, al, be) in gin:
        O.gdn_tree_verify(S0, qg, kg, vg, al, be, parent[:ng], 1.0 / math.sqrt(s.dk))
        O.commit_gdn(S0, kg, vg, al, be, sub_path)
    t2 = time.perf_counter()
    dep = O.depths(parent)
    steps_s = sum(x + 1 for x in dep[:ng]) + len(sub_path)
    steps_f = sum(x + 1 for x in dep) + len(path)
    n_attn = len(cfg.attn_layers)
    n_gdn = cfg.n_layers - n_attn
    est_attn = (t1 - t0) * (n * s.Hq) / (na * ka * G) * n_attn
    est_gdn = (t2 - t1) * (steps_f * s.Hv) / (steps_s * gh) * (n_gdn / len(gs))
    return t2 - t0, est_attn + est_gdn, t1 - t0, t2 - t1


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's value: a replicated job is as slow as its
    slowest replica.  One rank: the value itself."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(nodes_per_round: int, world: int, ms_per_round: float) -> float:
    """Whole-job tree nodes per second: each of the `world` replicas verifies
    its own round of `nodes_per_round` nodes in `ms_per_round` (the slowest
    rank's time), weak scaling."""
    return world * nodes_per_round / (ms_per_round / 1e3)


def run_ours(args, rank, world, local_rank):
    from speculative_tree_verify_masked_gb300 import binding as B
    from speculative_tree_verify_masked_gb300 import build as _build
    from speculative_tree_verify_masked_gb300 import synth
    from speculative_tree_verify_masked_gb300.round import VerifyRound

    _build.build()
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    cfg = synth.workload(args.config)
    pool = B.KVPool(local_rank) if args.kv_pool else None
    extra = {} if args.kv_window is None else {"cap_extra": args.kv_window - max(cfg.ctx_lens)}
    r = VerifyRound(cfg, device=dev, split=args.split, kv_pool=pool, **extra)
    n_nodes = r.n_nodes
    acc_lens = [len(p) for p in r.expected_paths]
    nodes_per_round = sum(n_nodes)
    bytes_round = round_bytes(cfg, n_nodes, acc_lens)

    # --- device-timed: CUDA-graph replay of whole rounds -------------------
    graph = r.capture()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    assert r.status() == 0, f"device status {r.status()}"
    clocks = ClockSampler(local_rank) if not args.no_clocks else None
    if clocks:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record()
    for _ in range(args.steps):
        graph.replay()
    ev1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(t_wall0, t_wall1) if clocks else None
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    assert r.status() == 0, f"device status {r.status()}"
    # the dominant call, one attention layer's verify: CUDA events captured
    # around each attention layer in a second graph of the same round (event
    # nodes would cut the programmatic launch edges of the timed graph),
    # replayed right after the timed region
    attn_ms = None
    if r.attn:
        marked = r.capture(attn_marks=True)
        ms_l = []
        for _ in range(max(3, min(args.steps, 20))):
            marked.replay()
            torch.cuda.synchronize()
            ms_l.append(statistics.mean(r.attn_marks_ms()))
        attn_ms = statistics.median(ms_l)
        assert r.status() == 0, f"device status {r.status()}"
    attn_timing = ("CUDA events around each attention layer, captured in a graph of the same round and "
                   "replayed after the timed region (median over replays of the mean over layers)")

    # --- eager rounds (launch overhead included), for context ---------------
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_eager = max(3, min(args.steps, 30))
    r.run()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n_eager):
        r.run()
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n_eager


    # --- end to end through the C ABI with host buffers ---------------------
    e2e = None
    if not args.no_e2e:
        dev_in = [r.tree.parent, r.tree.node_off, r.tok, r.greedy]
        for a in r.attn.values():
            dev_in += [a["q"], a["k_t"], a["v_t"]]
        for g in r.gdn.values():
            dev_in += [g["q"], g["k"], g["v"], g["alpha"], g["beta"]]
        host_in = [t.cpu().pin_memory() for t in dev_in]
        dev_out = [r.path, r.acc_len, r.bonus]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def e2e_step():
            for d_, h_ in zip(dev_in, host_in):
                d_.copy_(h_, non_blocking=True)
            r.run()
            for d_, h_ in zip(dev_out, host_out):
                h_.copy_(d_, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        n_e2e = max(3, min(args.steps, 50))
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / n_e2e, world, dev)
        assert r.status() == 0
        e2e = {"value": round(job_throughput(nodes_per_round, world, e2e_ms), 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "steps": n_e2e, "path": "eager C-ABI calls (ctypes), pinned host inputs in, accepted path out"}

    # --- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) --------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp = oracle_sample_inputs(cfg, dev)
        s = cfg.shapes
        # calibrate on the smallest sample, then size it for about 12 s of CPU work
        grp = max(1, s.Hv // s.Hk)  # value heads per key head: whole groups only
        _, _, ta, tg = time_oracle(cfg, inp, 1, n_nodes[0], grp, n_nodes[0])
        ka = int(min(s.Hkv, max(1, 6.0 // max(ta, 1e-3))))
        gh = int(min(s.Hv, max(grp, (6.0 / max(tg, 1e-3)) * grp))) // grp * grp
        secs, ests = 0.0, []
        while secs < 10.0 and len(ests) < 5:  # at least 10 s of CPU work in all
            t, e, _, _ = time_oracle(cfg, inp, ka, n_nodes[0], gh, n_nodes[0])
            secs += t
            ests.append(e)
        est = statistics.median(ests)
        cpu = {"value": round(nodes_per_round / est, 3) if cfg.n_seq == 1 else None, "unit": UNIT,
               "cores": blas_threads(), "kind": "oracle",
               "sample": (f"fp64 numpy oracle on sequence 0: one attention layer restricted to {ka} of {s.Hkv} KV "
                          f"heads (all {n_nodes[0]} nodes, full context) and {min(3, cfg.n_layers - 1)} GDN layers "
                          f"restricted to {gh} of {s.Hv} value heads, plus accept and commit, run {len(ests)} times; "
                          f"{secs:.1f} s of CPU work in all, scaled by heads and layers to one "
                          f"{cfg.n_layers}-layer round (median {est:.1f} s estimated per round)"),
               "est_round_s": round(est, 2)}

    hbm_peak, peak_kind = peaks()
    round_gbs = bytes_round / (ms / 1e3) / 1e9
    roof = None
    if attn_ms is not None:
        ab = attn_layer_bytes(cfg, n_nodes)
        ach = ab / (attn_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(ach / hbm_peak, 4),
                "traffic": args.traffic if args.traffic is not None else MEASURED_TRAFFIC.get(cfg.name),
                "kernel": "tv_attn_tree_verify (attn_split_kernel + attn_tail_kernel), one layer",
                "timing": attn_timing,
                "algorithmic_bytes_per_launch": ab, "ms_per_launch": round(attn_ms, 4),
                "peak_kind": peak_kind}
    n_attn = len(r.attn)
    n_gdn = len(r.gdn)
    launches_per_round = 1 + 2 * n_attn + n_gdn + 1 + (1 + math.ceil(n_attn / 16) + math.ceil(n_gdn / 32) + 1)
    line = {
        "metric": METRIC, "value": round(job_throughput(nodes_per_round, world, ms), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "layers": cfg.n_layers, "attention_layers": n_attn, "gdn_layers": n_gdn,
                   "ctx_lens": cfg.ctx_lens, "tree_nodes": n_nodes, "accepted": acc_lens,
                   "Hq_Hkv_D": [cfg.shapes.Hq, cfg.shapes.Hkv, cfg.shapes.D],
                   "Hk_Hv_dk_dv": [cfg.shapes.Hk, cfg.shapes.Hv, cfg.shapes.dk, cfg.shapes.dv],
                   "split": r.split, "timing": "CUDA-graph replay of whole rounds, CUDA events",
                   "l2": "no flush: every round streams inputs far larger than L2 (KV context per round)",
                   "parallelism": f"replicas x{world}",
                   "kv": ("pool: address space reserved for the whole cache, 2 MiB pages committed for rows below "
                          f"L + {r.kv_margin}" if pool else "static buffers"), "kv_window": r.cap},
        "us_per_round": round(ms * 1e3, 2),
        **({"kv_pool": {"committed_bytes": pool.committed_bytes, "reserved_bytes": pool.reserved_bytes,
                        "page_bytes": pool.page_bytes}} if pool else {}),
        "hbm": {"algorithmic_bytes_per_round": bytes_round, "achieved_gbs": round(round_gbs, 1),
                "frac_of_measured": round(round_gbs / hbm_peak, 4), "frac_of_8tbs": round(round_gbs / SPEC_HBM_GBS, 4)},
        "eager_ms_per_step": round(eager_ms, 4),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
        "gpu_launches": launches_per_round * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    if rank != 0:
        return
    from speculative_tree_verify_masked_gb300 import synth
    cfg = synth.workload(args.config)
    s = cfg.shapes
    inp = oracle_sample_inputs(cfg, "cpu")
    n_nodes = len(inp[0])
    # calibrate the smallest sample, then size each step so the run stays near two minutes
    time_oracle(cfg, inp, 1, 1, 1, 1)
    secs1 = time_oracle(cfg, inp, 1, 1, 1, 1)[0]
    budget = 120.0 / max(1, args.steps + args.warmup)
    grow = max(1.0, budget / max(secs1, 1e-4))
    na = max(1, min(n_nodes, int(grow)))
    ng = max(1, min(n_nodes, int(grow)))
    gh = max(1, min(s.Hv // s.Hk, int(grow / ng)))
    for _ in range(args.warmup):
        time_oracle(cfg, inp, 1, na, gh, ng)
    ests = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        est = time_oracle(cfg, inp, 1, na, gh, ng)[1]
        ests.append(est)
    wall = time.perf_counter() - t0
    est = statistics.median(ests)
    value = round(n_nodes * cfg.n_seq / est, 4)
    sample = (f"fp64 numpy oracle, per step: one attention layer restricted to 1 of {s.Hkv} KV heads and the first "
              f"{na} of {n_nodes} tree nodes (full context), 3 GDN layers restricted to {gh} of {s.Hv} value heads "
              f"and the first {ng} nodes, plus accept and commit; scaled by query rows and recurrence steps to one "
              f"{cfg.n_layers}-layer round")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(est * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "layers": cfg.n_layers, "ctx_lens": cfg.ctx_lens,
                       "tree_nodes": [n_nodes] * cfg.n_seq, "parallelism": "rank 0 only (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": sample, "wall_s": round(wall, 1)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=3, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--split", type=int, default=None,
                    help="positions per KV split (multiple of 64); default: the plan chosen for the workload")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--traffic", type=float, default=None, help="ncu DRAM bytes per attention launch, if measured")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--kv-pool", action="store_true", help="attention caches from the KV pool (tv_kvpool_*)")
    ap.add_argument("--kv-window", type=int, default=None,
                    help="cache rows per sequence (default: the context plus 64)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
