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
# kernels) on a GB300, keyed by workload name: dram__bytes_read.sum +
# dram__bytes_write.sum from an ncu capture of the current kernels.  A figure
# is dropped whenever the kernels change and stays absent (reported as null)
# until it is captured again.
MEASURED_TRAFFIC: dict[str, int] = {
    # one attention layer of the stack (bench.py --layers 3): split 538,193,664 read + 2,713,344 written,
    # tail 16,039,424 read; the same kernels and launch as every attention layer of the full round
    "64-layer mixer stack (48 GDN + 16 attention), L 131072, 32-node tree": 538193664 + 2713344 + 16039424,
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
# workload description shared by both arms
# ---------------------------------------------------------------------------
def num_sms_or_default() -> int:
    try:
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    except Exception:
        pass
    return 152  # GB300


def workload_config(cfg, n_nodes, acc_lens, split, world, kv_desc, kv_window, layers_run=None):
    c = {"workload": cfg.name, "layers": cfg.n_layers, "attention_layers": len(cfg.attn_layers),
         "gdn_layers": cfg.n_layers - len(cfg.attn_layers), "ctx_lens": cfg.ctx_lens, "tree_nodes": n_nodes,
         "accepted": acc_lens, "Hq_Hkv_D": [cfg.shapes.Hq, cfg.shapes.Hkv, cfg.shapes.D],
         "Hk_Hv_dk_dv": [cfg.shapes.Hk, cfg.shapes.Hv, cfg.shapes.dk, cfg.shapes.dv], "split": split,
         "timing": "CUDA-graph replay of whole rounds, CUDA events",
         "l2": "no flush: every round streams inputs far larger than L2 (KV context per round)",
         "parallelism": f"replicas x{world}", "kv": kv_desc, "kv_window": kv_window}
    if layers_run is not None:
        c["layers_run"] = layers_run
    return c


# ---------------------------------------------------------------------------
# oracle sample (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
# One step of the oracle is a fixed sample of one round, for every sequence of
# the workload: the first attention layer restricted to KV head 0 (its query
# heads, all tree nodes, the full context), the first GDN layer restricted to
# key head 0 (its value heads, all tree nodes), the accept walk, and the commit
# of that KV head's path rows and those value heads' states.  One round holds
# n_attn x Hkv such attention pieces and n_gdn x Hk such GDN pieces; the round
# estimate is the sum of each piece's time times its count.
def sample_counts(cfg):
    s = cfg.shapes
    n_attn = len(cfg.attn_layers)
    n_gdn = cfg.n_layers - n_attn
    return {"attention": n_attn * s.Hkv, "gdn": n_gdn * s.Hk, "accept": 1, "commit_attention": n_attn * s.Hkv,
            "commit_gdn": n_gdn * s.Hk}


def sample_text(cfg):
    s = cfg.shapes
    c = sample_counts(cfg)
    a0 = cfg.attn_layers[0] if cfg.attn_layers else None
    g0 = next((i for i in range(cfg.n_layers) if not cfg.is_attn(i)), None)
    return (f"fp64 numpy oracle; one step = for each of the {cfg.n_seq} sequence(s): attention layer {a0} "
            f"restricted to KV head 0 ({s.Hq // s.Hkv} query heads, every tree node, the full context), GDN layer "
            f"{g0} restricted to key head 0 ({s.Hv // s.Hk} value heads, every tree node), the accept walk, and "
            f"the commit of that head's path rows and those heads' states; one round = {c['attention']} such "
            f"attention pieces + {c['gdn']} GDN pieces (+ the commits alike), so the round estimate scales each "
            f"piece's measured time by its count")


def oracle_sample_inputs(cfg):
    """The sample's inputs (fp64 numpy, generated on the host), per sequence."""
    from speculative_tree_verify_masked_gb300 import synth
    s = cfg.shapes
    G, grp = s.Hq // s.Hkv, s.Hv // s.Hk
    a0 = cfg.attn_layers[0] if cfg.attn_layers else None
    g0 = next((i for i in range(cfg.n_layers) if not cfg.is_attn(i)), None)
    d = lambda t: t.detach().double().cpu().numpy()
    out = []
    for q in range(cfg.n_seq):
        parent, tok, greedy, _ = synth.tree_and_tokens(cfg, q)
        n, L = len(parent), cfg.ctx_lens[q]
        item = {"parent": parent, "tok": tok, "greedy": greedy, "L": L}
        if a0 is not None:
            a = synth.attn_layer_inputs(cfg, a0, q, n, L + 16, "cpu")
            item["attn"] = (d(a["K"][:1]), d(a["V"][:1]), d(a["q"][:, :G]), d(a["k_t"][:, :1]), d(a["v_t"][:, :1]))
        if g0 is not None:
            g = synth.gdn_layer_inputs(cfg, g0, q, n, "cpu")
            item["gdn"] = (d(g["S0"][:grp]), d(g["q"][:, :1]), d(g["k"][:, :1]), d(g["v"][:, :grp]),
                           d(g["alpha"][:, :grp]), d(g["beta"][:, :grp]))
        out.append(item)
    return out


def run_oracle_sample(cfg, inputs):
    """One step of the sample; returns the wall seconds of each piece."""
    import oracle.tree_verify as O
    s = cfg.shapes
    t = {"attention": 0.0, "gdn": 0.0, "accept": 0.0, "commit_attention": 0.0, "commit_gdn": 0.0}
    for item in inputs:
        parent, L = item["parent"], item["L"]
        c0 = time.perf_counter()
        if "attn" in item:
            K, V, q, kt, vt = item["attn"]
            O.attn_tree_verify(K, V, L, q, kt, vt, parent, 1.0 / math.sqrt(s.D))
        c1 = time.perf_counter()
        if "gdn" in item:
            S0, q, k, v, al, be = item["gdn"]
            O.gdn_tree_verify(S0, q, k, v, al, be, parent, 1.0 / math.sqrt(s.dk))
        c2 = time.perf_counter()
        path, _, _ = O.accept_path(parent, item["tok"], item["greedy"])
        c3 = time.perf_counter()
        if "attn" in item:
            K, V, _, kt, vt = item["attn"]
            O.commit_attn(K, V, L, kt, vt, path)
        c4 = time.perf_counter()
        if "gdn" in item:
            S0, _, k, v, al, be = item["gdn"]
            O.commit_gdn(S0, k, v, al, be, path)
        c5 = time.perf_counter()
        t["attention"] += c1 - c0
        t["gdn"] += c2 - c1
        t["accept"] += c3 - c2
        t["commit_attention"] += c4 - c3
        t["commit_gdn"] += c5 - c4
    return t


def round_estimate_s(cfg, pieces):
    counts = sample_counts(cfg)
    return sum(pieces[k] * counts[k] for k in counts)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                  "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def one_thread_sample(cfg_id: int, runs: int):
    """The sample timed in a fresh process whose BLAS and OpenMP pools have
    one thread (the pools are sized when numpy loads); returns the median
    piece times or None."""
    env = dict(os.environ, **ONE_THREAD_ENV)
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample-worker", "--config",
                              str(cfg_id), "--steps", str(runs)], capture_output=True, text=True, env=env,
                             timeout=900)
        return json.loads(out.stdout.strip().splitlines()[-1])["pieces_s"]
    except Exception:
        return None


def median_pieces(runs):
    return {k: statistics.median(r[k] for r in runs) for k in runs[0]}


def oracle_worker(args):
    """--oracle-sample-worker: time the sample `--steps` times in this process, print JSON."""
    from speculative_tree_verify_masked_gb300 import synth
    cfg = synth.workload(args.config)
    inp = oracle_sample_inputs(cfg)
    runs = [run_oracle_sample(cfg, inp) for _ in range(max(1, args.steps))]
    print(json.dumps({"pieces_s": median_pieces(runs)}), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def gdn_front_timing(r, n_rep: int = 10):
    """Per GDN layer of the round: the front end fused into the verify
    (tv_gdn_tree_verify_fused: raw projections in, gated-norm outputs out)
    against the three calls it replaces (tv_gdn_front -> tv_gdn_tree_verify ->
    tv_gdn_out_norm), each over all the round's GDN layers (their own states,
    synthetic raw inputs of the layer's shape, convolution width 4) captured
    in one CUDA graph on the round's tree and replayed; CUDA events, us per
    layer (median over replays).  The outputs of both are checked equal."""
    from speculative_tree_verify_masked_gb300 import binding as B

    cfg = r.cfg
    s = cfg.shapes
    W = 4
    C = 2 * s.Hk * s.dk + s.Hv * s.dv
    n = sum(r.n_nodes)
    dt = s.kv_dtype
    dev = r.device
    g = torch.Generator(device=dev).manual_seed(4242)
    rn = lambda *shape, std=1.0, d=torch.float32: (torch.randn(*shape, generator=g, device=dev) * std).to(d)
    e = lambda *shape, d=dt: torch.empty(*shape, dtype=d, device=dev)
    layers = []
    for li, gl in r.gdn.items():
        tails = [rn(W - 1, C, d=dt) for _ in range(cfg.n_seq)]
        layers.append(dict(gl=gl["layer"], fl=B.GdnFrontLayer(s.Hk, s.Hv, s.dk, s.dv, rn(C, W, std=0.5), tails, dt),
                           tails=tails, x=rn(n, C, d=dt), a=rn(n, s.Hv), b=rn(n, s.Hv), z=rn(n, s.Hv, s.dv, d=dt),
                           wn=1.0 + rn(s.dv, std=0.1), q=e(n, s.Hk, s.dk), k=e(n, s.Hk, s.dk), v=e(n, s.Hv, s.dv),
                           al=e(n, s.Hv, d=torch.float32), be=e(n, s.Hv, d=torch.float32), o=e(n, s.Hv, s.dv),
                           out3=e(n, s.Hv, s.dv), out1=e(n, s.Hv, s.dv)))
    B.tv_tree_prepare(r.tree)

    def three():
        for L in layers:
            B.tv_gdn_front(L["fl"], r.tree, cfg.n_seq, L["x"], L["a"], L["b"], L["q"], L["k"], L["v"], L["al"], L["be"])
            B.tv_gdn_tree_verify(L["gl"], r.tree, L["q"], L["k"], L["v"], L["al"], L["be"], L["o"], r.gdn_scale)
            B.tv_gdn_out_norm(L["fl"], n, L["o"], L["z"], L["wn"], L["out3"])

    def fused():
        for L in layers:
            B.tv_gdn_tree_verify_fused(L["gl"], L["fl"], r.tree, L["x"], L["a"], L["b"], L["z"], L["wn"], L["out1"],
                                       r.gdn_scale)

    res = {}
    for name, fn in (("three_calls", three), ("fused", fused)):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        for _ in range(3):
            graph.replay()
        ts = []
        for _ in range(n_rep):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / len(layers))
        res[name] = round(statistics.median(ts), 2)
        del graph
    assert r.status() == 0
    same = all(torch.equal(L["out1"].view(torch.int16), L["out3"].view(torch.int16)) for L in layers)
    assert same, "fused GDN front end differs from the three calls"
    return {"fused_us_per_layer": res["fused"], "three_calls_us_per_layer": res["three_calls"],
            "layers": len(layers), "conv_width": W, "bit_equal": same,
            "how": "each form over all GDN layers of the round in one CUDA graph (programmatic launch as in the "
                   "round), CUDA events around replays, median of " + str(n_rep)}


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
    r = VerifyRound(cfg, device=dev, split=args.split, kv_pool=pool, layers=args.layers_list, **extra)
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
    attn_ms = gdn_ms = None
    if r.attn or r.gdn:
        marked = r.capture(layer_marks=True)
        ms_a, ms_g = [], []
        for _ in range(max(3, min(args.steps, 20))):
            marked.replay()
            torch.cuda.synchronize()
            if r.attn:
                ms_a.append(statistics.mean(r.attn_marks_ms()))
            if r.gdn:
                ms_g.append(statistics.mean(r.gdn_marks_ms()))
        attn_ms = statistics.median(ms_a) if ms_a else None
        gdn_ms = statistics.median(ms_g) if ms_g else None
        assert r.status() == 0, f"device status {r.status()}"
        del marked
    attn_timing = ("CUDA events around each layer's verify call, captured in a graph of the same round and "
                   "replayed after the timed region (median over replays of the mean over layers)")

    # --- the GDN front end fused into the verify, against the three calls ---
    gdn_front = gdn_front_timing(r) if (r.gdn and cfg.shapes.kv_dtype == torch.bfloat16 and not args.no_front) \
        else None

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
    # Every input a host hands a round sits in one pinned host buffer and goes
    # in with one copy; the accepted paths, lengths and bonus tokens come back
    # with one copy.
    e2e = None
    if not args.no_e2e:
        io_in, io_out = r.pack_io()
        host_in = torch.empty(io_in.shape, dtype=torch.uint8, pin_memory=True)
        host_in.copy_(io_in)
        host_out = torch.empty(io_out.shape, dtype=torch.uint8, pin_memory=True)

        # the trees, tokens and the first tenth of the layers' inputs go in
        # on the round's stream; the rest on a copy stream, which the round
        # waits for just before the first layer that reads it
        cut, li_cut = r.input_split(0.1)
        side = torch.cuda.Stream()
        arrived = torch.cuda.Event()

        def e2e_step():
            io_in[:cut].copy_(host_in[:cut], non_blocking=True)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                io_in[cut:].copy_(host_in[cut:], non_blocking=True)
                arrived.record(side)
            r.run(layer_waits={li_cut: arrived} if li_cut is not None else None)
            if li_cut is None:
                stream.wait_event(arrived)
            host_out.copy_(io_out, non_blocking=True)
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
               "h2d_bytes_per_step": int(io_in.numel()), "d2h_bytes_per_step": int(io_out.numel()),
               "h2d_copies_per_step": 2, "d2h_copies_per_step": 1, "ms_per_step": round(e2e_ms, 4),
               "steps": n_e2e,
               "path": "eager C-ABI calls (ctypes); the round's host inputs (trees, tokens, every layer's node "
                       "inputs) in from one pinned buffer in two copies (the first tenth on the round's "
                       "stream, the rest on a copy stream the round waits for before the first layer that "
                       "reads it), the accepted paths, lengths and bonus tokens out"}

    # --- CPU baseline: the oracle on its stated sample (rank 0, N = 1) -------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp = oracle_sample_inputs(cfg)
        runs = [run_oracle_sample(cfg, inp) for _ in range(3)]
        pieces = median_pieces(runs)
        est = round_estimate_s(cfg, pieces)
        one = one_thread_sample(args.config, 1)
        est1 = round_estimate_s(cfg, one) if one else None
        cpu = {"value": round(nodes_per_round / est, 4), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": sample_text(cfg), "cpu_model": cpu_model(), "nproc": os.cpu_count(),
               "runs": len(runs), "sample_s": round(sum(pieces.values()), 3),
               "pieces_s": {k: round(v, 4) for k, v in pieces.items()}, "round_estimate_s": round(est, 2),
               "one_thread": ({"value": round(nodes_per_round / est1, 4), "cores": 1,
                               "pieces_s": {k: round(v, 4) for k, v in one.items()},
                               "round_estimate_s": round(est1, 2)} if one else None)}

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
    roof_round = {"bound": "hbm", "achieved": round(round_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                  "frac": round(round_gbs / hbm_peak, 4), "traffic": None,
                  "kernel": "one whole verify round (prepare, every layer's verify, accept, commit)",
                  "timing": "the timed region: CUDA-graph replays of whole rounds",
                  "algorithmic_bytes_per_launch": bytes_round, "ms_per_launch": round(ms, 5),
                  "peak_kind": peak_kind}
    n_attn = len(r.attn)
    n_gdn = len(r.gdn)
    launches_per_round = 1 + 2 * n_attn + n_gdn + 1 + (1 + math.ceil(n_attn / 16) + math.ceil(n_gdn / 64) + 1)
    kv_desc = ("pool: address space reserved for the whole cache, 2 MiB pages committed for rows below "
               f"L + {r.kv_margin}" if pool else "static buffers")
    line = {
        "metric": METRIC, "value": round(job_throughput(nodes_per_round, world, ms), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, n_nodes, acc_lens, r.split, world, kv_desc, r.cap,
                                  layers_run=args.layers_list),
        "us_per_round": round(ms * 1e3, 2),
        **({"kv_pool": {"committed_bytes": pool.committed_bytes, "reserved_bytes": pool.reserved_bytes,
                        "page_bytes": pool.page_bytes}} if pool else {}),
        "hbm": {"algorithmic_bytes_per_round": bytes_round, "achieved_gbs": round(round_gbs, 1),
                "frac_of_measured": round(round_gbs / hbm_peak, 4), "frac_of_8tbs": round(round_gbs / SPEC_HBM_GBS, 4)},
        "eager_ms_per_step": round(eager_ms, 4),
        "layer_us": {"attention_verify": round(attn_ms * 1e3, 2) if attn_ms is not None else None,
                     "gdn_verify": round(gdn_ms * 1e3, 2) if gdn_ms is not None else None,
                     "how": "CUDA events around each layer's verify call in a marked copy of the round's graph "
                            "(median over replays of the mean over layers of that kind; the marks cut the "
                            "programmatic launch overlap between neighbouring layers)"},
        "gdn_front_fused": gdn_front,
        "roofline": roof, "roofline_round": roof_round, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
        "gpu_launches": launches_per_round * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: W untimed and K timed
    steps of the sample (rank 0 only).  ms_per_step is the measured time of
    one step of the sample; value is the round throughput that sample
    implies."""
    if rank != 0:
        return
    from speculative_tree_verify_masked_gb300 import synth
    from speculative_tree_verify_masked_gb300.round import auto_split
    cfg = synth.workload(args.config)
    trees = [synth.tree_and_tokens(cfg, q) for q in range(cfg.n_seq)]
    n_nodes = [len(t[0]) for t in trees]
    acc_lens = [len(t[3]) for t in trees]
    split = args.split or auto_split(cfg.ctx_lens, n_nodes, cfg.shapes.Hq, cfg.shapes.Hkv, num_sms_or_default())
    inp = oracle_sample_inputs(cfg)
    for _ in range(args.warmup):
        run_oracle_sample(cfg, inp)
    runs, walls = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = time.perf_counter()
        runs.append(run_oracle_sample(cfg, inp))
        walls.append(time.perf_counter() - a)
    wall = time.perf_counter() - t0
    pieces = median_pieces(runs)
    est = round_estimate_s(cfg, pieces)
    value = round(sum(n_nodes) / est, 4)
    kv_window = max(cfg.ctx_lens) + 64
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.median(walls) * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, n_nodes, acc_lens, split, world, "static buffers", kv_window),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": sample_text(cfg), "cpu_model": cpu_model(), "nproc": os.cpu_count(),
                             "pieces_s": {k: round(v, 4) for k, v in pieces.items()},
                             "round_estimate_s": round(est, 2), "wall_s": round(wall, 1)},
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
    ap.add_argument("--no-front", action="store_true", help="skip the fused GDN front-end timing")
    ap.add_argument("--kv-pool", action="store_true", help="attention caches from the KV pool (tv_kvpool_*)")
    ap.add_argument("--kv-window", type=int, default=None,
                    help="cache rows per sequence (default: the context plus 64)")
    ap.add_argument("--layers", default=None,
                    help="comma-separated layer indices: run only these layers of the stack (for profiling)")
    ap.add_argument("--oracle-sample-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.layers_list = [int(x) for x in args.layers.split(",")] if args.layers else None
    if args.oracle_sample_worker:
        oracle_worker(args)
        return
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
