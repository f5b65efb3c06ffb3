"""Thin ctypes binding of libtreeverify.so (include/tv.h): the same names as
the C ABI, argument marshalling only.  Every step of the verify round runs in
the library's CUDA kernels; there is no Python or CPU fallback, and loading
fails loudly when the library has not been built.

PyTorch provides the device memory and the stream; tensors are passed as raw
device pointers.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_size_t, c_void_p

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtreeverify.so")

TV_MAX_SEQ = 8
TV_MAX_NODES = 64
TV_MAX_PATH = 16
TV_F32, TV_BF16 = 0, 1

STATUS_NAMES = {0: "TV_OK", 1: "TV_ERR_ARG", 2: "TV_ERR_SHAPE", 3: "TV_ERR_DTYPE", 4: "TV_ERR_ALIGN",
                5: "TV_ERR_TREE", 6: "TV_ERR_CAPACITY", 7: "TV_ERR_CUDA", 8: "TV_ERR_WORKSPACE",
                9: "TV_ERR_TIMEOUT", 10: "TV_ERR_LEN", 11: "TV_ERR_SCRATCH"}


class TvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({tv_status_string(code)})")


class tv_tree(ctypes.Structure):
    _fields_ = [("n_seq", c_int32), ("n_total", c_int32), ("n_max", c_int32), ("node_off", c_void_p),
                ("parent", c_void_p), ("meta", c_void_p), ("status", c_void_p), ("flags", c_int32)]


TV_TREE_OVERLAP = 1


class tv_attn_layer(ctypes.Structure):
    _fields_ = [("dtype", c_int32), ("Hq", c_int32), ("Hkv", c_int32), ("D", c_int32), ("cap", c_int32),
                ("K", POINTER(c_void_p)), ("V", POINTER(c_void_p))]


class tv_gdn_layer(ctypes.Structure):
    _fields_ = [("dtype", c_int32), ("Hk", c_int32), ("Hv", c_int32), ("dk", c_int32), ("dv", c_int32),
                ("S", POINTER(c_void_p))]


class tv_gdn_front_layer(ctypes.Structure):
    _fields_ = [("dtype", c_int32), ("Hk", c_int32), ("Hv", c_int32), ("dk", c_int32), ("dv", c_int32),
                ("width", c_int32), ("wconv", c_void_p), ("tail", POINTER(c_void_p))]


class tv_plan(ctypes.Structure):
    _fields_ = [("split", c_int32)]


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with speculative_tree_verify_masked_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        T, A, G, P = POINTER(tv_tree), POINTER(tv_attn_layer), POINTER(tv_gdn_layer), POINTER(tv_plan)
        vp = c_void_p
        L.tv_status_string.restype = ctypes.c_char_p
        L.tv_status_string.argtypes = [c_int32]
        L.tv_version.restype = ctypes.c_char_p
        L.tv_version.argtypes = []
        L.tv_tree_meta_bytes.restype = c_size_t
        L.tv_tree_meta_bytes.argtypes = [c_int32, c_int32]
        L.tv_tree_prepare.restype = c_int32
        L.tv_tree_prepare.argtypes = [T, vp]
        L.tv_attn_workspace_bytes.restype = c_size_t
        L.tv_attn_workspace_bytes.argtypes = [P, A, c_int32, c_int32, c_int32]
        L.tv_attn_tree_verify.restype = c_int32
        L.tv_attn_tree_verify.argtypes = [P, A, T, vp, c_int32, vp, vp, vp, vp, c_float, vp, c_size_t, vp]
        L.tv_gdn_tree_verify.restype = c_int32
        L.tv_gdn_tree_verify.argtypes = [G, T, vp, vp, vp, vp, vp, vp, c_float, vp]
        L.tv_accept_path.restype = c_int32
        L.tv_accept_path.argtypes = [T, vp, vp, vp, vp, vp, vp]
        L.tv_commit_path.restype = c_int32
        L.tv_commit_path.argtypes = [T, vp, vp, c_int32, A, POINTER(vp), POINTER(vp), c_int32, G, POINTER(vp),
                                     POINTER(vp), POINTER(vp), POINTER(vp), vp, vp]
        L.tv_decode_step.restype = c_int32
        L.tv_decode_step.argtypes = [P, A, G, c_int32, vp, c_int32, vp, vp, vp, vp, vp, vp, c_float, vp, c_size_t,
                                     vp, vp]
        L.tv_len_advance.restype = c_int32
        L.tv_len_advance.argtypes = [vp, vp, c_int32, c_int32, vp]
        L.tv_attn_static_scratch_bytes.restype = c_size_t
        L.tv_attn_static_scratch_bytes.argtypes = []
        L.tv_attn_tree_verify_static.restype = c_int32
        L.tv_attn_tree_verify_static.argtypes = [P, A, T, vp, c_int32, vp, vp, vp, vp, c_float, vp]
        L.tv_attn_rope.restype = c_int32
        L.tv_attn_rope.argtypes = [A, T, c_int32, vp, c_int32, c_int32, c_float, vp, vp, vp, vp, vp, vp]
        L.tv_attn_tree_verify_gated.restype = c_int32
        L.tv_attn_tree_verify_gated.argtypes = [P, A, T, vp, c_int32, vp, vp, vp, vp, vp, c_float, vp, c_size_t, vp]
        L.tv_attn_decode_gated.restype = c_int32
        L.tv_attn_decode_gated.argtypes = [P, A, c_int32, vp, c_int32, vp, vp, vp, vp, vp, c_float, vp, c_size_t, vp,
                                           vp]
        F = POINTER(tv_gdn_front_layer)
        L.tv_gdn_front.restype = c_int32
        L.tv_gdn_front.argtypes = [F, T, c_int32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.tv_gdn_out_norm.restype = c_int32
        L.tv_gdn_out_norm.argtypes = [F, c_int32, vp, vp, vp, vp, vp]
        L.tv_gdn_tree_verify_fused.restype = c_int32
        L.tv_gdn_tree_verify_fused.argtypes = [G, F, T, vp, vp, vp, vp, vp, vp, c_float, vp]
        L.tv_gdn_decode_fused.restype = c_int32
        L.tv_gdn_decode_fused.argtypes = [G, F, c_int32, vp, vp, vp, vp, vp, vp, c_float, vp, vp]
        L.tv_gdn_conv_commit.restype = c_int32
        L.tv_gdn_conv_commit.argtypes = [F, T, c_int32, vp, vp, vp, vp, vp]
        L.tv_kvpool_page_bytes.restype = c_size_t
        L.tv_kvpool_page_bytes.argtypes = [c_int32, c_size_t]
        L.tv_kvpool_create.restype = c_int32
        L.tv_kvpool_create.argtypes = [c_int32, c_size_t, POINTER(vp)]
        L.tv_kvpool_reserve.restype = c_int32
        L.tv_kvpool_reserve.argtypes = [vp, c_size_t, POINTER(vp)]
        L.tv_kvpool_commit_rows.restype = c_int32
        L.tv_kvpool_commit_rows.argtypes = [vp, vp, c_int32, c_size_t, c_size_t, ctypes.c_int64, vp]
        L.tv_kvpool_release_rows.restype = c_int32
        L.tv_kvpool_release_rows.argtypes = [vp, vp, c_int32, c_size_t, c_size_t, ctypes.c_int64]
        L.tv_kvpool_committed_bytes.restype = c_size_t
        L.tv_kvpool_committed_bytes.argtypes = [vp]
        L.tv_kvpool_reserved_bytes.restype = c_size_t
        L.tv_kvpool_reserved_bytes.argtypes = [vp]
        L.tv_kvpool_destroy.restype = c_int32
        L.tv_kvpool_destroy.argtypes = [vp]
        L.tv_wait_selftest.restype = c_int32
        L.tv_wait_selftest.argtypes = [vp, vp, ctypes.c_int64, vp]
        _lib = L
    return _lib


EXPORTED = ["tv_status_string", "tv_version", "tv_tree_meta_bytes", "tv_tree_prepare", "tv_attn_workspace_bytes",
            "tv_attn_tree_verify", "tv_gdn_tree_verify", "tv_accept_path", "tv_commit_path", "tv_decode_step",
            "tv_len_advance", "tv_attn_static_scratch_bytes", "tv_attn_tree_verify_static", "tv_kvpool_page_bytes",
            "tv_kvpool_create", "tv_kvpool_reserve", "tv_kvpool_commit_rows", "tv_kvpool_release_rows",
            "tv_kvpool_committed_bytes", "tv_kvpool_reserved_bytes", "tv_kvpool_destroy", "tv_attn_rope",
            "tv_attn_tree_verify_gated", "tv_attn_decode_gated", "tv_gdn_front", "tv_gdn_out_norm",
            "tv_gdn_conv_commit", "tv_gdn_tree_verify_fused", "tv_gdn_decode_fused", "tv_wait_selftest"]


def _check(code: int, where: str):
    if code != 0:
        raise TvError(code, where)


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return c_void_p(stream.cuda_stream)
    return c_void_p(int(stream))


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return TV_BF16
    if dt == torch.float32:
        return TV_F32
    raise TypeError(f"unsupported dtype {dt}")


def _ptr_array(tensors):
    arr = (c_void_p * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


# ---------------------------------------------------------------------------
# descriptors (own the device buffers / pointer arrays they point to)
# ---------------------------------------------------------------------------
class Tree:
    """Device buffers of a tv_tree for a list of per-sequence parent arrays."""

    def __init__(self, parents, device="cuda", n_max=None, overlap: bool = False):
        sizes = [len(p) for p in parents]
        off = [0]
        for n in sizes:
            off.append(off[-1] + n)
        flat = [int(x) for p in parents for x in p]
        self.n_seq = len(parents)
        self.n_total = off[-1]
        self.n_max = n_max if n_max is not None else max(sizes)
        self.node_off = torch.tensor(off, dtype=torch.int32, device=device)
        self.parent = torch.tensor(flat, dtype=torch.int32, device=device)
        self.meta = torch.zeros(max(16, tv_tree_meta_bytes(self.n_seq, self.n_total)), dtype=torch.uint8,
                                device=device)
        self.status = torch.zeros(4, dtype=torch.int32, device=device)
        self.c = tv_tree(self.n_seq, self.n_total, self.n_max, self.node_off.data_ptr(), self.parent.data_ptr(),
                         self.meta.data_ptr(), self.status.data_ptr(), TV_TREE_OVERLAP if overlap else 0)

    def status_code(self) -> int:
        return int(self.status[0].item())


class AttnLayer:
    """tv_attn_layer over per-sequence caches K[s], V[s] of shape [Hkv, cap, D]."""

    def __init__(self, K, V, Hq: int):
        self.K, self.V = list(K), list(V)
        Hkv, cap, D = self.K[0].shape
        self._k, self._v = _ptr_array(self.K), _ptr_array(self.V)
        self.c = tv_attn_layer(_dtype_code(self.K[0].dtype), Hq, Hkv, D, cap, self._k, self._v)


class GdnLayer:
    """tv_gdn_layer over per-sequence fp32 states S[s] of shape [Hv, dv, dk]."""

    def __init__(self, S, Hk: int, dtype: torch.dtype):
        self.S = list(S)
        Hv, dv, dk = self.S[0].shape
        self._s = _ptr_array(self.S)
        self.c = tv_gdn_layer(_dtype_code(dtype), Hk, Hv, dk, dv, self._s)


def plan(split: int) -> tv_plan:
    return tv_plan(split)


# ---------------------------------------------------------------------------
# the C ABI, one wrapper per entry point
# ---------------------------------------------------------------------------
def tv_status_string(code: int) -> str:
    return lib().tv_status_string(code).decode()


def tv_version() -> str:
    return lib().tv_version().decode()


def tv_tree_meta_bytes(n_seq: int, n_total: int) -> int:
    return int(lib().tv_tree_meta_bytes(n_seq, n_total))


def tv_tree_prepare(tree: Tree, stream=None):
    _check(lib().tv_tree_prepare(ctypes.byref(tree.c), _stream(stream)), "tv_tree_prepare")


def tv_attn_workspace_bytes(pl: tv_plan, layer: AttnLayer, n_seq: int, n_max: int, max_len: int) -> int:
    return int(lib().tv_attn_workspace_bytes(ctypes.byref(pl), ctypes.byref(layer.c), n_seq, n_max, max_len))


def tv_attn_tree_verify(pl, layer: AttnLayer, tree: Tree, len_, max_len, q, k_t, v_t, out, scale, ws, stream=None):
    _check(lib().tv_attn_tree_verify(ctypes.byref(pl) if pl is not None else None, ctypes.byref(layer.c),
                                     ctypes.byref(tree.c), _ptr(len_), max_len, _ptr(q), _ptr(k_t), _ptr(v_t),
                                     _ptr(out), scale, _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                     _stream(stream)), "tv_attn_tree_verify")


def tv_attn_rope(layer: AttnLayer, tree: Tree | None, n_seq, len_, max_len, rot_dims, theta, q_raw, k_raw, q, k,
                 status=None, stream=None):
    """Rotary embedding of one layer's query and key rows at each row's
    logical position (tree: L + depth; tree None: one decode token per
    sequence at L)."""
    _check(lib().tv_attn_rope(ctypes.byref(layer.c), ctypes.byref(tree.c) if tree is not None else None, n_seq,
                              _ptr(len_), max_len, rot_dims, theta, _ptr(q_raw), _ptr(k_raw), _ptr(q), _ptr(k),
                              _ptr(status), _stream(stream)), "tv_attn_rope")


def tv_attn_tree_verify_gated(pl, layer: AttnLayer, tree: Tree, len_, max_len, q, k_t, v_t, gate, out, scale, ws,
                              stream=None):
    _check(lib().tv_attn_tree_verify_gated(ctypes.byref(pl) if pl is not None else None, ctypes.byref(layer.c),
                                           ctypes.byref(tree.c), _ptr(len_), max_len, _ptr(q), _ptr(k_t), _ptr(v_t),
                                           _ptr(gate), _ptr(out), scale, _ptr(ws),
                                           0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "tv_attn_tree_verify_gated")


def tv_attn_decode_gated(pl, attn: AttnLayer, n_seq, len_, max_len, q, k, v, gate, out, scale, ws, status,
                         stream=None):
    _check(lib().tv_attn_decode_gated(ctypes.byref(pl) if pl is not None else None, ctypes.byref(attn.c), n_seq,
                                      _ptr(len_), max_len, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), scale,
                                      _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _ptr(status),
                                      _stream(stream)), "tv_attn_decode_gated")


class GdnFrontLayer:
    """A tv_gdn_front_layer over torch tensors: wconv [C][W] fp32, one tail
    [W-1][C] per sequence."""

    def __init__(self, Hk: int, Hv: int, dk: int, dv: int, wconv, tails, dtype: torch.dtype):
        self.wconv, self.tails = wconv, list(tails)
        self._tail = _ptr_array(self.tails)
        self.c = tv_gdn_front_layer(_dtype_code(dtype), Hk, Hv, dk, dv, wconv.shape[1], _ptr(wconv), self._tail)


def tv_gdn_front(layer: GdnFrontLayer, tree: Tree | None, n_seq, x, a_raw, b_raw, q, k, v, alpha, beta, status=None,
                 stream=None):
    _check(lib().tv_gdn_front(ctypes.byref(layer.c), ctypes.byref(tree.c) if tree is not None else None, n_seq,
                              _ptr(x), _ptr(a_raw), _ptr(b_raw), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                              _ptr(status), _stream(stream)), "tv_gdn_front")


def tv_gdn_out_norm(layer: GdnFrontLayer, rows, o, z, w_norm, out, stream=None):
    _check(lib().tv_gdn_out_norm(ctypes.byref(layer.c), rows, _ptr(o), _ptr(z), _ptr(w_norm), _ptr(out),
                                 _stream(stream)), "tv_gdn_out_norm")


def tv_gdn_conv_commit(layer: GdnFrontLayer, tree: Tree | None, n_seq, x, path=None, acc_len=None, status=None,
                       stream=None):
    _check(lib().tv_gdn_conv_commit(ctypes.byref(layer.c), ctypes.byref(tree.c) if tree is not None else None, n_seq,
                                    _ptr(x), _ptr(path), _ptr(acc_len), _ptr(status), _stream(stream)),
           "tv_gdn_conv_commit")


def tv_attn_static_scratch_bytes() -> int:
    return int(lib().tv_attn_static_scratch_bytes())


def tv_attn_tree_verify_static(pl, layer: AttnLayer, tree: Tree, len_, max_len, q, k_t, v_t, out, scale,
                               stream=None):
    _check(lib().tv_attn_tree_verify_static(ctypes.byref(pl) if pl is not None else None, ctypes.byref(layer.c),
                                            ctypes.byref(tree.c), _ptr(len_), max_len, _ptr(q), _ptr(k_t),
                                            _ptr(v_t), _ptr(out), scale, _stream(stream)),
           "tv_attn_tree_verify_static")


def tv_gdn_tree_verify(layer: GdnLayer, tree: Tree, q, k, v, alpha, beta, out, scale, stream=None):
    _check(lib().tv_gdn_tree_verify(ctypes.byref(layer.c), ctypes.byref(tree.c), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(alpha), _ptr(beta), _ptr(out), scale, _stream(stream)),
           "tv_gdn_tree_verify")


def tv_gdn_tree_verify_fused(layer: GdnLayer, front: GdnFrontLayer, tree: Tree, x, a_raw, b_raw, z, w_norm, out,
                             scale, stream=None):
    _check(lib().tv_gdn_tree_verify_fused(ctypes.byref(layer.c), ctypes.byref(front.c), ctypes.byref(tree.c), _ptr(x),
                                          _ptr(a_raw), _ptr(b_raw), _ptr(z), _ptr(w_norm), _ptr(out), scale,
                                          _stream(stream)), "tv_gdn_tree_verify_fused")


def tv_gdn_decode_fused(layer: GdnLayer, front: GdnFrontLayer, n_seq, x, a_raw, b_raw, z, w_norm, out, scale, status,
                        stream=None):
    _check(lib().tv_gdn_decode_fused(ctypes.byref(layer.c), ctypes.byref(front.c), n_seq, _ptr(x), _ptr(a_raw),
                                     _ptr(b_raw), _ptr(z), _ptr(w_norm), _ptr(out), scale, _ptr(status),
                                     _stream(stream)), "tv_gdn_decode_fused")


def tv_accept_path(tree: Tree, tok, greedy, path, acc_len, bonus, stream=None):
    _check(lib().tv_accept_path(ctypes.byref(tree.c), _ptr(tok), _ptr(greedy), _ptr(path), _ptr(acc_len),
                                _ptr(bonus), _stream(stream)), "tv_accept_path")


class CommitArgs:
    """Marshalled argument block of tv_commit_path for fixed layer lists."""

    def __init__(self, attn_layers, k_t, v_t, gdn_layers, k, v, alpha, beta):
        self.n_attn, self.n_gdn = len(attn_layers), len(gdn_layers)
        self.attn = (tv_attn_layer * max(1, self.n_attn))(*[l.c for l in attn_layers])
        self.gdn = (tv_gdn_layer * max(1, self.n_gdn))(*[l.c for l in gdn_layers])
        self.keep = (attn_layers, gdn_layers, k_t, v_t, k, v, alpha, beta)
        self.k_t, self.v_t = _ptr_array(k_t), _ptr_array(v_t)
        self.k, self.v = _ptr_array(k), _ptr_array(v)
        self.alpha, self.beta = _ptr_array(alpha), _ptr_array(beta)


def tv_commit_path(tree: Tree, path, acc_len, args: CommitArgs, len_, stream=None):
    _check(lib().tv_commit_path(ctypes.byref(tree.c), _ptr(path), _ptr(acc_len), args.n_attn, args.attn, args.k_t,
                                args.v_t, args.n_gdn, args.gdn, args.k, args.v, args.alpha, args.beta, _ptr(len_),
                                _stream(stream)), "tv_commit_path")


def tv_decode_step(pl, attn: AttnLayer | None, gdn: GdnLayer | None, n_seq, len_, max_len, q, k, v, alpha, beta,
                   out, scale, ws, status, stream=None):
    _check(lib().tv_decode_step(ctypes.byref(pl) if pl is not None else None,
                                ctypes.byref(attn.c) if attn is not None else None,
                                ctypes.byref(gdn.c) if gdn is not None else None, n_seq, _ptr(len_), max_len,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(out), scale, _ptr(ws),
                                0 if ws is None else ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
           "tv_decode_step")


def tv_len_advance(len_, by, inc: int, n_seq: int, stream=None):
    _check(lib().tv_len_advance(_ptr(len_), _ptr(by), inc, n_seq, _stream(stream)), "tv_len_advance")


# ---------------------------------------------------------------------------
# KV pool
# ---------------------------------------------------------------------------
def tv_wait_selftest(status, result, limit_cycles: int, stream=None):
    _check(lib().tv_wait_selftest(_ptr(status), _ptr(result), int(limit_cycles), _stream(stream)), "tv_wait_selftest")


def tv_kvpool_page_bytes(device: int, page_bytes: int = 0) -> int:
    return int(lib().tv_kvpool_page_bytes(device, page_bytes))


def tv_kvpool_create(device: int, page_bytes: int = 0) -> c_void_p:
    h = c_void_p()
    _check(lib().tv_kvpool_create(device, page_bytes, ctypes.byref(h)), "tv_kvpool_create")
    return h


def tv_kvpool_reserve(pool, nbytes: int) -> int:
    base = c_void_p()
    _check(lib().tv_kvpool_reserve(pool, nbytes, ctypes.byref(base)), "tv_kvpool_reserve")
    return int(base.value)


def tv_kvpool_commit_rows(pool, base: int, n_heads: int, head_stride: int, row_bytes: int, rows: int, stream=None):
    _check(lib().tv_kvpool_commit_rows(pool, c_void_p(base), n_heads, head_stride, row_bytes, rows, _stream(stream)),
           "tv_kvpool_commit_rows")


def tv_kvpool_release_rows(pool, base: int, n_heads: int, head_stride: int, row_bytes: int, keep_rows: int):
    _check(lib().tv_kvpool_release_rows(pool, c_void_p(base), n_heads, head_stride, row_bytes, keep_rows),
           "tv_kvpool_release_rows")


def tv_kvpool_committed_bytes(pool) -> int:
    return int(lib().tv_kvpool_committed_bytes(pool))


def tv_kvpool_reserved_bytes(pool) -> int:
    return int(lib().tv_kvpool_reserved_bytes(pool))


def tv_kvpool_destroy(pool):
    _check(lib().tv_kvpool_destroy(pool), "tv_kvpool_destroy")


class _DeviceRange:
    """A device address range presented to torch through the CUDA array
    interface (torch keeps this object alive with the tensor)."""

    def __init__(self, ptr: int, numel: int, typestr: str, pool):
        self.pool = pool
        self.__cuda_array_interface__ = {"shape": (numel,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None, "stream": None}


class KVPool:
    """Caches [H][cap][D] whose address space is reserved whole and whose
    pages are committed as rows are written (tv_kvpool_*)."""

    _TYPESTR = {torch.float32: "<f4", torch.bfloat16: "<i2", torch.float16: "<f2"}

    def __init__(self, device: int = 0, page_bytes: int = 0):
        self.device = device
        self.h = tv_kvpool_create(device, page_bytes)
        self.page_bytes = tv_kvpool_page_bytes(device, page_bytes)

    def cache(self, heads: int, cap: int, dim: int, dtype: torch.dtype) -> torch.Tensor:
        """A [heads, cap, dim] tensor over a fresh reservation; row 0 of every
        head is committed (zeroed), nothing else."""
        esize = torch.empty((), dtype=dtype).element_size()
        numel = heads * cap * dim
        base = tv_kvpool_reserve(self.h, numel * esize)
        tv_kvpool_commit_rows(self.h, base, heads, cap * dim * esize, dim * esize, 1)
        t = torch.as_tensor(_DeviceRange(base, numel, self._TYPESTR[dtype], self), device=f"cuda:{self.device}")
        return t.view(dtype).view(heads, cap, dim)

    @staticmethod
    def _geom(t: torch.Tensor):
        heads, cap, dim = t.shape
        es = t.element_size()
        return t.data_ptr(), heads, cap * dim * es, dim * es

    def commit_rows(self, t: torch.Tensor, rows: int, stream=None):
        base, heads, hs, rb = self._geom(t)
        tv_kvpool_commit_rows(self.h, base, heads, hs, rb, rows, stream)

    def release_rows(self, t: torch.Tensor, keep_rows: int):
        base, heads, hs, rb = self._geom(t)
        tv_kvpool_release_rows(self.h, base, heads, hs, rb, keep_rows)

    @property
    def committed_bytes(self) -> int:
        return tv_kvpool_committed_bytes(self.h)

    @property
    def reserved_bytes(self) -> int:
        return tv_kvpool_reserved_bytes(self.h)

    def close(self):
        """Frees every page and reservation: tensors from cache() must not be
        used afterwards."""
        if self.h is not None:
            tv_kvpool_destroy(self.h)
            self.h = None
