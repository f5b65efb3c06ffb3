"""One speculative verify round over a mixer stack, driven through the C ABI.

A round is: tv_tree_prepare, one tv_gdn_tree_verify / tv_attn_tree_verify per
layer (in layer order), tv_accept_path, tv_commit_path.  This module owns the
device buffers of a synthetic workload (caches, states, per-layer node
inputs and outputs, tree tables, workspace) and issues those calls on one
stream; it can also capture the round in a CUDA graph.
"""
from __future__ import annotations

import math

import torch

from . import binding as B
from . import synth

DEFAULT_SPLIT = 4096  # positions per KV split (multiple of 64)
TILE = 64


def auto_split(ctx_lens, n_nodes, Hq, Hkv, num_sms, lo=512, hi=16384):
    """The split size (positions, multiple of 64) whose split-kernel makespan
    is smallest for these context lengths and trees: items (split x KV head x
    128-row block) are dealt round-robin to one persistent CTA per SM, an item
    costs its tiles plus four tiles of start-up and write-back, and among equal makespans the
    larger split (fewer partial states to merge) wins.  A deployment fixes
    the result once; verify and decode must use the same value."""
    G = Hq // Hkv
    best = None
    for split in range(lo, hi + 1, TILE):
        st = split // TILE
        costs = []
        for L, n in zip(ctx_lens, n_nodes):
            # the split kernel's tiles: below the own segment of the deepest
            # possible row, one tile back from its last position's tile
            tend = max((L + min(n - 1, B.TV_MAX_PATH - 1)) // TILE - 1, 0)
            nrb = -(-n * G // 128)
            for sp in range(-(-tend // st)):
                c = min(st, tend - sp * st) + 4
                costs += [c] * (Hkv * nrb)
        loads = [0] * num_sms
        for w, c in enumerate(costs):
            loads[w % num_sms] += c
        key = (max(loads) if costs else 0, -split)
        if best is None or key < best[0]:
            best = (key, split)
    return best[1]


class VerifyRound:
    def __init__(self, cfg: synth.Workload, device="cuda", split: int | None = None, layers=None,
                 cap_extra: int = 64, overlap: bool = True, kv_pool: B.KVPool | None = None,
                 kv_margin: int = 256, max_len: int | None = None):
        self.cfg = cfg
        self.device = device
        s = cfg.shapes
        self.layers = list(range(cfg.n_layers)) if layers is None else list(layers)
        self.trees = [synth.tree_and_tokens(cfg, q) for q in range(cfg.n_seq)]
        self.parents = [t[0] for t in self.trees]
        self.n_nodes = [len(p) for p in self.parents]
        # the round's calls run in round order on one stream, so each kernel may
        # start while the one before it finishes (TV_TREE_OVERLAP)
        self.tree = B.Tree(self.parents, device=device, overlap=overlap)
        self.tok = torch.tensor([x for t in self.trees for x in t[1]], dtype=torch.int32, device=device)
        self.greedy = torch.tensor([x for t in self.trees for x in t[2]], dtype=torch.int32, device=device)
        self.expected_paths = [t[3] for t in self.trees]
        self.len0 = torch.tensor(cfg.ctx_lens, dtype=torch.int32, device=device)
        self.len = self.len0.clone()
        # host bound on the context lengths (above the first round's when
        # rounds run without resetting the lengths); caches hold cap_extra more rows
        self.max_len = max(cfg.ctx_lens) if max_len is None else max_len
        self.cap = self.max_len + cap_extra
        if split is None:
            sms = torch.cuda.get_device_properties(device).multi_processor_count
            split = auto_split(cfg.ctx_lens, self.n_nodes, s.Hq, s.Hkv, sms)
        self.split = split
        self.plan = B.plan(split)
        self._marks = None  # (layer, start, end) events around layers while capturing
        self._graph_marks = None
        # With a KV pool the caches are reserved whole and only the rows below
        # the context length plus kv_margin are committed; the committed rows
        # hold the same values as the static caches'.
        self.kv_pool, self.kv_margin = kv_pool, kv_margin
        self.attn_scale = 1.0 / math.sqrt(s.D)
        self.gdn_scale = 1.0 / math.sqrt(s.dk)
        self.attn, self.gdn = {}, {}
        for li in self.layers:
            if cfg.is_attn(li):
                per = [synth.attn_layer_inputs(cfg, li, q, self.n_nodes[q], self.cap, device) for q in range(cfg.n_seq)]
                if kv_pool is not None:
                    for q, x in enumerate(per):
                        for name in ("K", "V"):
                            t = kv_pool.cache(s.Hkv, self.cap, s.D, s.kv_dtype)
                            kv_pool.commit_rows(t, min(self.cap, cfg.ctx_lens[q] + kv_margin))
                            t[:, :cfg.ctx_lens[q]].copy_(x[name][:, :cfg.ctx_lens[q]])
                            x[name] = t
                layer = B.AttnLayer([x["K"] for x in per], [x["V"] for x in per], s.Hq)
                q_ = torch.cat([x["q"] for x in per]).contiguous()
                k_t = torch.cat([x["k_t"] for x in per]).contiguous()
                v_t = torch.cat([x["v_t"] for x in per]).contiguous()
                out = torch.empty_like(q_)
                self.attn[li] = dict(layer=layer, q=q_, k_t=k_t, v_t=v_t, out=out)
            else:
                per = [synth.gdn_layer_inputs(cfg, li, q, self.n_nodes[q], device) for q in range(cfg.n_seq)]
                layer = B.GdnLayer([x["S0"] for x in per], s.Hk, s.kv_dtype)
                d = {k: torch.cat([x[k] for x in per]).contiguous() for k in ("q", "k", "v", "alpha", "beta")}
                d["out"] = torch.empty((d["v"].shape[0], s.Hv, s.dv), dtype=s.kv_dtype, device=device)
                d["layer"] = layer
                self.gdn[li] = d
        self._alloc_ws()
        self.path = torch.full((cfg.n_seq, B.TV_MAX_PATH), -1, dtype=torch.int32, device=device)
        self.acc_len = torch.zeros(cfg.n_seq, dtype=torch.int32, device=device)
        self.bonus = torch.zeros(cfg.n_seq, dtype=torch.int32, device=device)
        self._build_commit_args()

    def _build_commit_args(self):
        al = [li for li in self.layers if li in self.attn]
        gl = [li for li in self.layers if li in self.gdn]
        self.commit_args = B.CommitArgs(
            [self.attn[li]["layer"] for li in al], [self.attn[li]["k_t"] for li in al],
            [self.attn[li]["v_t"] for li in al], [self.gdn[li]["layer"] for li in gl],
            [self.gdn[li]["k"] for li in gl], [self.gdn[li]["v"] for li in gl],
            [self.gdn[li]["alpha"] for li in gl], [self.gdn[li]["beta"] for li in gl])

    def pack_io(self):
        """Place every input a host hands a round (the trees' node offsets
        and parent arrays, the drafted and greedy tokens, every layer's node
        inputs) in one device byte buffer, and the results it reads back
        (accepted paths, lengths, bonus tokens) in another, each tensor at a
        256-byte aligned offset with its values kept; the round's tensors
        become views of the two buffers.  A host then feeds a round with one
        copy in and reads it with one copy out.  Returns (inputs, outputs)."""
        ins = [("tree", "node_off"), ("tree", "parent"), ("r", "tok"), ("r", "greedy")]
        for li in self.layers:
            names = ("q", "k_t", "v_t") if li in self.attn else ("q", "k", "v", "alpha", "beta")
            ins += [(li, n) for n in names]

        def get(key):
            owner, name = key
            if owner == "tree":
                return getattr(self.tree, name)
            if owner == "r":
                return getattr(self, name)
            return (self.attn.get(owner) or self.gdn[owner])[name]

        def put(key, t):
            owner, name = key
            if owner == "tree":
                setattr(self.tree, name, t)
            elif owner == "r":
                setattr(self, name, t)
            else:
                (self.attn.get(owner) or self.gdn[owner])[name] = t

        def pack(keys, record=False):
            offs, total = [], 0
            for key in keys:
                t = get(key)
                offs.append(total)
                total += (t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.empty(max(total, 256), dtype=torch.uint8, device=self.device)
            for key, o in zip(keys, offs):
                t = get(key)
                nb = t.numel() * t.element_size()
                v = buf[o:o + nb].view(t.dtype).view(t.shape)
                v.copy_(t)
                put(key, v)
            if record:
                self.io_in_offsets = dict(zip(keys, offs))
            return buf

        self.io_in = pack(ins, record=True)
        self.io_out = pack([("r", "path"), ("r", "acc_len"), ("r", "bonus")])
        self.tree.c.node_off = self.tree.node_off.data_ptr()
        self.tree.c.parent = self.tree.parent.data_ptr()
        self._build_commit_args()
        return self.io_in, self.io_out

    def input_split(self, frac: float):
        """(byte offset, layer): the packed inputs from the first layer whose
        inputs start at or past frac of the buffer, and that layer; the bytes
        before it hold the trees, tokens and the earlier layers' inputs."""
        total = self.io_in.numel()
        for li in self.layers:
            first = min(o for (owner, _), o in self.io_in_offsets.items() if owner == li)
            if first >= frac * total:
                return first, li
        return total, None

    def _alloc_ws(self):
        ws_bytes = 0
        if self.attn:
            first = next(iter(self.attn.values()))["layer"]
            ws_bytes = B.tv_attn_workspace_bytes(self.plan, first, self.cfg.n_seq, self.tree.n_max, self.max_len)
        self.ws = (torch.empty(max(16, ws_bytes) // 4 + 4, dtype=torch.float32, device=self.device)
                   if ws_bytes else None)

    def set_split(self, split: int):
        """Another plan (positions per KV split) and a workspace sized for it.
        Graphs captured before hold the old plan and workspace."""
        self.split = split
        self.plan = B.plan(split)
        self.ws = None
        self._alloc_ws()

    def commit_kv(self, lens=None):
        """Commit cache rows up to each sequence's length (default: read from
        the device) plus kv_margin, ahead of the rounds that will write them.
        A host call between rounds; no-op without a KV pool."""
        if self.kv_pool is None:
            return
        lens = self.len.tolist() if lens is None else list(lens)
        for a in self.attn.values():
            for q in range(self.cfg.n_seq):
                rows = min(self.cap, int(lens[q]) + self.kv_margin)
                self.kv_pool.commit_rows(a["layer"].K[q], rows)
                self.kv_pool.commit_rows(a["layer"].V[q], rows)

    # -- steps of the round -------------------------------------------------
    def prepare(self, stream=None):
        B.tv_tree_prepare(self.tree, stream)

    def verify_layer(self, li, stream=None):
        if li in self.attn:
            a = self.attn[li]
            B.tv_attn_tree_verify(self.plan, a["layer"], self.tree, self.len, self.max_len, a["q"], a["k_t"],
                                  a["v_t"], a["out"], self.attn_scale, self.ws, stream)
        else:
            g = self.gdn[li]
            B.tv_gdn_tree_verify(g["layer"], self.tree, g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["out"],
                                 self.gdn_scale, stream)

    def verify(self, stream=None, layer_waits=None):
        """Prepare, then every layer's verify.  layer_waits maps a layer to a
        CUDA event the stream waits for before that layer (inputs that arrive
        by a copy on another stream)."""
        self.prepare(stream)
        for li in self.layers:
            if layer_waits and li in layer_waits:
                s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.current_stream()
                s.wait_event(layer_waits[li])
            marks = self._marks is not None
            if marks:
                # external events become timing-capable record nodes of the graph
                a = torch.cuda.Event(enable_timing=True, external=True)
                b = torch.cuda.Event(enable_timing=True, external=True)
                a.record()
            self.verify_layer(li, stream)
            if marks:
                b.record()
                self._marks.append((li, a, b))

    def accept(self, stream=None):
        B.tv_accept_path(self.tree, self.tok, self.greedy, self.path, self.acc_len, self.bonus, stream)

    def commit(self, stream=None):
        B.tv_commit_path(self.tree, self.path, self.acc_len, self.commit_args, self.len, stream)

    def run(self, stream=None, reset_len: bool = True, layer_waits=None):
        """One round.  With reset_len the context length is first restored so
        repeated rounds do the same work (the caches' rows past it and the
        states are overwritten by each commit)."""
        if reset_len:
            self.len.copy_(self.len0)
        self.verify(stream, layer_waits)
        self.accept(stream)
        self.commit(stream)

    def status(self) -> int:
        return self.tree.status_code()

    def capture(self, layer_marks: bool = False):
        """Capture run() in a CUDA graph on a side stream; returns the graph.
        With layer_marks, CUDA events recorded around every layer's verify
        call become part of the graph; after a replay, attn_marks_ms() and
        gdn_marks_ms() give each layer's time in that replay.  (Event nodes
        cut the programmatic launch edges around them, so a marked graph is
        for breaking a round down, not for timing it.)"""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run()  # warm (attribute setup outside capture)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self._marks = [] if layer_marks else None
        with torch.cuda.graph(g):
            self.run()
        self._graph_marks, self._marks = self._marks, None
        return g

    def attn_marks_ms(self):
        """Per attention layer, the ms between the events around it in the
        latest replay of the graph captured with layer_marks."""
        return [a.elapsed_time(b) for li, a, b in (self._graph_marks or []) if li in self.attn]

    def gdn_marks_ms(self):
        """Per GDN layer, as attn_marks_ms."""
        return [a.elapsed_time(b) for li, a, b in (self._graph_marks or []) if li in self.gdn]
