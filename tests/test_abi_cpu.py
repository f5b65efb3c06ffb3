"""The C ABI without a GPU: the library builds and loads, exports every
function include/tv.h declares, its structs have the layout the Python
binding assumes, and host-visible argument errors come back as status codes
before anything touches the device.  Also the host-side launch planning
(auto_split) and the synthetic tree generator's invariants."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from speculative_tree_verify_masked_gb300 import binding as B
from speculative_tree_verify_masked_gb300 import build as BUILD
from speculative_tree_verify_masked_gb300 import synth
from speculative_tree_verify_masked_gb300.round import TILE, auto_split

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tv.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(B.LIB_PATH):
        BUILD.build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(tv_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert len(names) >= 13, names
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(tv_\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    assert sorted(B.EXPORTED) == names, "binding.EXPORTED differs from the header"
    for n in names:
        assert hasattr(L, n)


def test_struct_layout_matches_c():
    """sizeof/offsetof of every ABI struct from gcc against ctypes."""
    structs = {"tv_tree": B.tv_tree, "tv_attn_layer": B.tv_attn_layer, "tv_gdn_layer": B.tv_gdn_layer,
               "tv_plan": B.tv_plan, "tv_gdn_front_layer": B.tv_gdn_front_layer}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "tv.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{name}.{f} %zu\\n", offsetof({name}, {f}));')
    lines += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write("\n".join(lines))
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        got = dict(l.rsplit(" ", 1) for l in subprocess.run([exe], capture_output=True, text=True,
                                                              check=True).stdout.splitlines())
    for name, cls in structs.items():
        assert int(got[f"{name} size"]) == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert int(got[f"{name}.{f}"]) == getattr(cls, f).offset, f"{name}.{f}"


def test_status_strings_and_version(L):
    for code, name in B.STATUS_NAMES.items():
        s = B.tv_status_string(code)
        assert s and s != "unknown status", name
    assert B.tv_status_string(99) == "unknown status"
    assert "sm_103a" in B.tv_version()


def _bf16_layer(Hq=24, Hkv=4, D=256, cap=4096, n_seq=1):
    K = (ctypes.c_void_p * n_seq)(*([0x1000] * n_seq))
    V = (ctypes.c_void_p * n_seq)(*([0x2000] * n_seq))
    layer = B.tv_attn_layer(B.TV_BF16, Hq, Hkv, D, cap, K, V)
    return layer, (K, V)


def test_workspace_size_formula(L):
    """Per KV head and query row one record of D + 4 fp32 values for each
    split and one for the last split's snapshot."""
    layer, keep = _bf16_layer()
    pl = B.tv_plan(512)
    n_seq, n_max, max_len = 2, 16, 4000
    splits = (max_len + 16 + 512 - 1) // 512 + 1
    want = n_seq * 4 * (splits + 1) * n_max * 6 * (256 + 4) * 4
    assert L.tv_attn_workspace_bytes(ctypes.byref(pl), ctypes.byref(layer), n_seq, n_max, max_len) == want
    bad = B.tv_plan(100)  # not a multiple of 64
    assert L.tv_attn_workspace_bytes(ctypes.byref(bad), ctypes.byref(layer), n_seq, n_max, max_len) == 0
    f32 = B.tv_attn_layer(B.TV_F32, 2, 1, 64, 256, keep[0], keep[1])
    assert L.tv_attn_workspace_bytes(ctypes.byref(pl), ctypes.byref(f32), 1, 4, 100) == 0


def test_host_argument_errors_need_no_device(L):
    """NULL or malformed descriptors return TV_ERR_ARG / TV_ERR_ALIGN without a launch."""
    vp = ctypes.c_void_p
    assert L.tv_tree_prepare(None, None) == 1
    bad_tree = B.tv_tree(0, 0, 0, None, None, None, None)
    assert L.tv_tree_prepare(ctypes.byref(bad_tree), None) == 1
    layer, keep = _bf16_layer()
    pl = B.tv_plan(512)
    assert L.tv_attn_tree_verify(ctypes.byref(pl), ctypes.byref(layer), None, vp(16), 10, vp(16), vp(16), vp(16),
                                 vp(16), 0.1, vp(16), 1 << 20, None) == 1
    assert L.tv_accept_path(None, vp(16), vp(16), vp(16), vp(16), vp(16), None) == 1
    assert L.tv_len_advance(None, None, 1, 1, None) == 1
    # a tree descriptor with a misaligned status word is ill formed
    t = B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4004)
    assert L.tv_tree_prepare(ctypes.byref(t), None) == 1
    # a misaligned node input is TV_ERR_ALIGN
    t = B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.tv_attn_tree_verify(ctypes.byref(pl), ctypes.byref(layer), ctypes.byref(t), vp(16), 10, vp(24), vp(16),
                                 vp(16), vp(16), 0.1, vp(16), 1 << 20, None) == 4
    # decode needs exactly one of attention / GDN
    assert L.tv_decode_step(ctypes.byref(pl), None, None, 1, vp(16), 1, vp(16), vp(16), vp(16), None, None, vp(16),
                            0.1, None, 0, vp(16), None) == 1


def test_front_end_host_argument_errors(L):
    """tv_attn_rope / the gated calls reject bad arguments before any launch."""
    vp = ctypes.c_void_p
    layer, keep = _bf16_layer()
    st = vp(16)

    def rope(lay, tree, n=1, ln=vp(16), ml=10, rot=64, th=1e7, q=vp(16), status=st):
        return L.tv_attn_rope(lay, tree, n, ln, ml, rot, th, q, vp(16), vp(16), vp(16), status, None)

    lay = ctypes.byref(layer)
    assert rope(None, None) == 1
    assert rope(lay, None, rot=63) == 1        # odd rotated dimensions
    assert rope(lay, None, rot=512) == 1       # more than the head dimension
    assert rope(lay, None, th=1.0) == 1        # base must exceed 1
    assert rope(lay, None, status=None) == 1   # decode mode reports to a status word
    assert rope(lay, None, n=0) == 1
    assert rope(lay, None, q=vp(24)) == 4      # misaligned row
    pl = B.tv_plan(512)
    t = B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.tv_attn_tree_verify_gated(ctypes.byref(pl), lay, ctypes.byref(t), vp(16), 10, vp(16), vp(16), vp(16),
                                       None, vp(16), 0.1, vp(16), 1 << 20, None) == 1   # gate required
    assert L.tv_attn_decode_gated(ctypes.byref(pl), lay, 1, vp(16), 10, vp(16), vp(16), vp(16), vp(24), vp(16), 0.1,
                                  vp(16), 1 << 20, vp(16), None) == 4


def test_gdn_front_host_argument_errors(L):
    """tv_gdn_front / tv_gdn_out_norm / tv_gdn_conv_commit reject bad
    arguments before any launch."""
    vp = ctypes.c_void_p
    tails = (vp * 1)(vp(0x1000))
    f = B.tv_gdn_front_layer(B.TV_BF16, 16, 48, 128, 128, 4, vp(0x2000), tails)
    st = vp(16)
    args = [vp(16)] * 8
    assert L.tv_gdn_front(None, None, 1, *args, st, None) == 1
    bad_w = B.tv_gdn_front_layer(B.TV_BF16, 16, 48, 128, 128, 9, vp(0x2000), tails)   # width above 8
    assert L.tv_gdn_front(ctypes.byref(bad_w), None, 1, *args, st, None) == 2
    bad_d = B.tv_gdn_front_layer(B.TV_BF16, 16, 48, 96, 96, 4, vp(0x2000), tails)     # head dim
    assert L.tv_gdn_front(ctypes.byref(bad_d), None, 1, *args, st, None) == 2
    bad_t = B.tv_gdn_front_layer(7, 16, 48, 128, 128, 4, vp(0x2000), tails)           # dtype
    assert L.tv_gdn_front(ctypes.byref(bad_t), None, 1, *args, st, None) == 3
    assert L.tv_gdn_front(ctypes.byref(f), None, 1, *args, None, None) == 1          # decode needs a status word
    assert L.tv_gdn_front(ctypes.byref(f), None, 9, *args, st, None) == 1            # too many sequences
    assert L.tv_gdn_out_norm(ctypes.byref(f), -1, vp(16), vp(16), vp(16), vp(16), None) == 1
    assert L.tv_gdn_out_norm(ctypes.byref(f), 0, vp(16), vp(16), vp(16), vp(16), None) == 0  # nothing to do
    assert L.tv_gdn_conv_commit(ctypes.byref(f), None, 1, None, None, None, st, None) == 1
    t = B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.tv_gdn_conv_commit(ctypes.byref(f), ctypes.byref(t), 1, vp(16), None, vp(16), None, None) == 1


def test_gdn_fused_host_argument_errors(L):
    """tv_gdn_tree_verify_fused and tv_gdn_decode_fused reject a missing or
    mismatched front-end layer, a missing input, a misaligned output or
    status word and a sequence count out of range before any launch."""
    vp = ctypes.c_void_p
    tails = (vp * 1)(vp(0x1000))
    states = (vp * 1)(vp(0x3000))
    g = B.tv_gdn_layer(B.TV_BF16, 16, 48, 128, 128, states)
    f = B.tv_gdn_front_layer(B.TV_BF16, 16, 48, 128, 128, 4, vp(0x2000), tails)
    t = B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4000)
    io = [vp(16)] * 4  # a_raw, b_raw, z, w_norm

    def fused(front, out=vp(16), x=vp(16)):
        return L.tv_gdn_tree_verify_fused(ctypes.byref(g), front, ctypes.byref(t), x, *io, out, 0.1, None)

    assert fused(None) == 1                                                        # no front-end layer
    other = B.tv_gdn_front_layer(B.TV_BF16, 16, 32, 128, 128, 4, vp(0x2000), tails)  # Hv differs
    assert fused(ctypes.byref(other)) == 2
    f32 = B.tv_gdn_front_layer(B.TV_F32, 16, 48, 128, 128, 4, vp(0x2000), tails)      # dtype differs
    assert fused(ctypes.byref(f32)) == 2
    wide = B.tv_gdn_front_layer(B.TV_BF16, 16, 48, 128, 128, 9, vp(0x2000), tails)    # width above 8
    assert fused(ctypes.byref(wide)) == 2
    no_tail = B.tv_gdn_front_layer(B.TV_BF16, 16, 48, 128, 128, 4, vp(0x2000), (vp * 1)(None))
    assert fused(ctypes.byref(no_tail)) == 1                                       # W > 1 needs each tail
    assert fused(ctypes.byref(f), x=None) == 1
    assert fused(ctypes.byref(f), out=vp(24)) == 4                                 # misaligned output
    # the decode form: a status word is required and aligned, n_seq in range
    dec = lambda n, st: L.tv_gdn_decode_fused(ctypes.byref(g), ctypes.byref(f), n, vp(16), vp(16), vp(16), vp(16),
                                              vp(16), vp(16), 0.1, st, None)
    assert dec(1, None) == 1
    assert dec(0, vp(16)) == 1
    assert dec(9, vp(16)) == 1
    assert dec(1, vp(20)) == 4
    assert L.tv_gdn_decode_fused(ctypes.byref(g), ctypes.byref(other), 1, vp(16), vp(16), vp(16), vp(16), vp(16),
                                 vp(16), 0.1, vp(16), None) == 2


def test_static_scratch_rejects_oversized_request_on_host(L):
    """The size check comes before any device call, so it runs here."""
    layer, keep = _bf16_layer(cap=40000)
    t = B.tv_tree(1, 64, 64, 0x1000, 0x2000, 0x3000, 0x4000)
    pl = B.tv_plan(64)
    need = L.tv_attn_workspace_bytes(ctypes.byref(pl), ctypes.byref(layer), 1, 64, 32768)
    assert need > L.tv_attn_static_scratch_bytes() == 48 << 20
    vp = ctypes.c_void_p
    rc = L.tv_attn_tree_verify_static(ctypes.byref(pl), ctypes.byref(layer), ctypes.byref(t), vp(16), 32768, vp(16),
                                      vp(16), vp(16), vp(16), 0.0625, None)
    assert rc == 11  # TV_ERR_SCRATCH


def test_static_scratch_rejects_ill_formed_tree_on_host(L):
    """An ill-formed tree descriptor or a negative length bound is an argument
    error (1) for the static call, as for the workspace call, even when the
    counts would wrap the scratch size computation."""
    layer, keep = _bf16_layer(cap=40000)
    pl = B.tv_plan(4096)
    vp = ctypes.c_void_p
    args = (vp(16), vp(16), vp(16), vp(16), 0.0625, None)
    bad_trees = [
        B.tv_tree(-1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4000),   # negative sequence count
        B.tv_tree(1, 4, -3, 0x1000, 0x2000, 0x3000, 0x4000),   # negative tree bound
        B.tv_tree(1, 4, 65, 0x1000, 0x2000, 0x3000, 0x4000),   # tree bound above 64 nodes
        B.tv_tree(9, 9, 1, 0x1000, 0x2000, 0x3000, 0x4000),    # more than 8 sequences
        B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4008),    # status word not 16-byte aligned
        B.tv_tree(1, 4, 4, 0, 0x2000, 0x3000, 0x4000),         # no node offsets
    ]
    for t in bad_trees:
        rc = L.tv_attn_tree_verify_static(ctypes.byref(pl), ctypes.byref(layer), ctypes.byref(t), vp(16), 32768,
                                          *args)
        assert rc == 1, (t.n_seq, t.n_total, t.n_max, rc)
    good = B.tv_tree(1, 4, 4, 0x1000, 0x2000, 0x3000, 0x4000)
    assert L.tv_attn_tree_verify_static(ctypes.byref(pl), ctypes.byref(layer), ctypes.byref(good), vp(16), -1,
                                        *args) == 1
    assert L.tv_attn_tree_verify_static(ctypes.byref(pl), ctypes.byref(layer), None, vp(16), 32768, *args) == 1
    assert L.tv_attn_tree_verify_static(ctypes.byref(pl), None, ctypes.byref(good), vp(16), 32768, *args) == 1


def test_auto_split_is_the_makespan_minimum():
    """Brute force over every split on a small case, with the stated cost model."""
    lens, nodes, Hq, Hkv, sms = [8192, 1024], [16, 5], 8, 2, 7

    def makespan(split):
        st, costs = split // TILE, []
        for L_, n in zip(lens, nodes):
            tsh, nrb = L_ // TILE, -(-n * (Hq // Hkv) // 128)
            for sp in range(-(-tsh // st)):
                costs += [min(st, tsh - sp * st) + 4] * (Hkv * nrb)
        loads = [0] * sms
        for w, c in enumerate(costs):
            loads[w % sms] += c
        return max(loads)

    got = auto_split(lens, nodes, Hq, Hkv, sms, lo=64, hi=8192)
    assert got % TILE == 0 and 64 <= got <= 8192
    best = min(makespan(s) for s in range(64, 8192 + 1, TILE))
    assert makespan(got) == best
    assert got == max(s for s in range(64, 8192 + 1, TILE) if makespan(s) == best)


@pytest.mark.parametrize("cfg_id", range(5))
def test_synthetic_trees_are_well_formed(cfg_id):
    cfg = synth.workload(cfg_id)
    for q in range(cfg.n_seq):
        parent, tok, greedy, path = synth.tree_and_tokens(cfg, q)
        n = len(parent)
        assert 1 <= n <= B.TV_MAX_NODES and parent[0] == -1
        assert all(0 <= parent[i] < i for i in range(1, n))
        depth = [0] * n
        for i in range(1, n):
            depth[i] = depth[parent[i]] + 1
        assert max(depth) < B.TV_MAX_PATH
        assert len(tok) == len(greedy) == n
        assert path[0] == 0 and all(parent[b] == a for a, b in zip(path, path[1:]))


def test_kvpool_host_errors(L):
    """KV pool calls reject bad handles and arguments on the host; without a
    GPU driver a pool cannot be created."""
    import torch
    vp = ctypes.c_void_p
    assert L.tv_kvpool_create(0, 0, None) == 1
    assert L.tv_kvpool_create(-1, 0, ctypes.byref(vp())) == 1
    assert L.tv_kvpool_reserve(None, 16, ctypes.byref(vp())) == 1
    assert L.tv_kvpool_commit_rows(None, vp(16), 1, 16, 16, 1, None) == 1
    assert L.tv_kvpool_release_rows(None, vp(16), 1, 16, 16, 1) == 1
    assert L.tv_kvpool_committed_bytes(None) == 0 and L.tv_kvpool_reserved_bytes(None) == 0
    assert L.tv_kvpool_destroy(None) == 1
    if not torch.cuda.is_available():
        assert L.tv_kvpool_page_bytes(0, 0) == 0
        h = vp()
        assert L.tv_kvpool_create(0, 0, ctypes.byref(h)) == 7 and not h.value
