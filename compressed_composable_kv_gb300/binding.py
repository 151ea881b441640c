"""ctypes binding of libc2kv.so: same names as the C ABI (include/c2kv.h).

Argument marshalling only -- every step of the path runs in the CUDA
library.  Device tensors are torch CUDA tensors (their data pointers are
passed through); host inputs are numpy arrays or CPU tensors.  A missing
library raises ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from .build import LIB

C2KV_OK, C2KV_EINVAL, C2KV_ENOMEM, C2KV_ENOTFOUND = 0, 1, 2, 3
C2KV_ECAPACITY, C2KV_ECUDA, C2KV_ETIMEOUT, C2KV_EDEVICE, C2KV_EIO = 4, 5, 6, 7, 8
C2KV_MASK_CAUSAL, C2KV_MASK_STRUCTURED, C2KV_MASK_ANCHOR = 0, 1, 2

STATUS_NAMES = {0: "C2KV_OK", 1: "C2KV_EINVAL", 2: "C2KV_ENOMEM", 3: "C2KV_ENOTFOUND",
                4: "C2KV_ECAPACITY", 5: "C2KV_ECUDA", 6: "C2KV_ETIMEOUT", 7: "C2KV_EDEVICE", 8: "C2KV_EIO"}


class C2KVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class c2kv_geometry(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_theta", ctypes.c_double)]


_i32, _sz, _vp = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pvp = ctypes.POINTER(ctypes.c_void_p)
_pg = ctypes.POINTER(c2kv_geometry)

_SIGNATURES = {
    "c2kv_store_save": (_i32, [_vp, ctypes.c_char_p]),
    "c2kv_store_load": (_i32, [_vp, ctypes.c_char_p]),
    "c2kv_test_expire_next_waits": (_i32, [_i32]),
    "c2kv_last_error": (ctypes.c_char_p, []),
    "c2kv_version": (ctypes.c_char_p, []),
    "c2kv_store_create": (_i32, [_pg, _sz, ctypes.POINTER(_vp)]),
    "c2kv_store_destroy": (None, [_vp]),
    "c2kv_store_segments": (_i32, [_vp, _i32, _pi32, _pi32, _pi32, _i32, _pvp, _pvp]),
    "c2kv_store_lookup": (_i32, [_vp, _i32, _pi32, _pi32, _pi32]),
    "c2kv_plan": (_i32, [_i32, _pi32, _pi32, _pi32, _pi32, _pi32, _pi32, _pi32]),
    "c2kv_compose": (_i32, [_vp, _i32, _pi32, _pi32, _i32, _vp, _vp, _i32, _vp, _vp, _pi32, _pi32, _vp]),
    "c2kv_compose_layers": (_i32, [_vp, _i32, _pi32, _pi32, _i32, ctypes.c_uint32, _i32, _i32, _vp, _vp, _i32,
                                   _vp, _vp, _pi32, _pi32, _vp]),
    "c2kv_rope_table_bytes": (_sz, [_pg, _i32]),
    "c2kv_rope_table": (_i32, [_pg, _vp, _i32, _vp, _vp]),
    "c2kv_attend_workspace_size": (_sz, [_pg, _i32, _i32, _i32]),
    "c2kv_masked_extra_bytes": (_sz, [_pg, _i32]),
    "c2kv_workspace_init": (_i32, [_vp, _sz, _vp]),
    "c2kv_attend_prefill": (_i32, [_pg, _i32, _i32, _pvp, _pvp, _pvp, _i32, _pi32, _i32,
                                   _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "c2kv_attend_decode": (_i32, [_pg, _i32, _i32, _pvp, _pvp, _pvp, _i32, _vp, _i32,
                                  _vp, _vp, _vp, _vp, _vp, _sz, ctypes.c_uint32, _vp]),
    "c2kv_attend_decode_noalloc": (_i32, [_pg, _i32, _i32, _pvp, _pvp, _pvp, _i32, _vp, _i32,
                                          _vp, _vp, _vp, _vp, _vp]),
    "c2kv_seq_advance": (_i32, [_i32, _vp, _i32, _vp]),
    "c2kv_attend_masked": (_i32, [_pg, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "c2kv_device_error": (_i32, [_pi32]),
    "c2kv_kernel_launches": (_i32, [ctypes.POINTER(ctypes.c_uint64)]),
    "c2kv_linear_workspace_size": (_sz, [_i32, _i32]),
    "c2kv_linear": (_i32, [_vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _sz,
                           ctypes.c_uint32, _vp]),
    "c2kv_rmsnorm": (_i32, [_vp, _i32, _i32, _vp, ctypes.c_float, _vp, ctypes.c_uint32, _vp]),
}

_lib = None


def load_library(path: str = LIB) -> ctypes.CDLL:
    """Load libc2kv.so (built by build.build_library) and declare signatures."""
    global _lib
    if _lib is not None and path == LIB:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libc2kv.so is not built ({path}); run "
                          "compressed_composable_kv_gb300.build.build_library()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB:
        _lib = lib
    return lib


def _check(status: int):
    if status != C2KV_OK:
        raise C2KVError(status, load_library().c2kv_last_error().decode())


def as_geometry(g) -> c2kv_geometry:
    if isinstance(g, c2kv_geometry):
        return g
    return c2kv_geometry(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, float(g.rope_theta))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: Optional[torch.Tensor], dtype=None, name="tensor") -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _nbytes(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _need(t: Optional[torch.Tensor], nbytes: int, name: str, exact: bool = False) -> None:
    """The C side reads or writes nbytes of t's memory (it only sees a pointer),
    so t must hold that many bytes: exactly, for per-token inputs and outputs."""
    have = _nbytes(t)
    if have < nbytes or (exact and have != nbytes):
        raise ValueError(f"{name} holds {have} bytes, expected {'' if exact else 'at least '}{nbytes}")


def _i32arr(vals) -> ctypes.Array:
    vals = [int(v) for v in vals]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def _host_ptr(a, nbytes: Optional[int], name: str) -> int:
    """Address of a host array of 2-byte elements that the caller keeps alive
    (no conversion: a temporary copy would be freed before the C call reads
    it).  nbytes, when known, is the exact size the C side will read."""
    if isinstance(a, torch.Tensor):
        if a.is_cuda or not a.is_contiguous() or a.element_size() != 2:
            raise ValueError(f"{name} must be a contiguous CPU tensor of 2-byte elements")
        size, ptr = a.numel() * 2, a.data_ptr()
    elif isinstance(a, np.ndarray):
        if not a.flags.c_contiguous or a.itemsize != 2:
            raise ValueError(f"{name} must be a C-contiguous array of 2-byte elements (bf16 bits)")
        size, ptr = a.nbytes, a.ctypes.data
    else:
        raise ValueError(f"{name} must be a numpy array or a CPU tensor, got {type(a).__name__}")
    if nbytes is not None and size != nbytes:
        raise ValueError(f"{name} holds {size} bytes, expected {nbytes}")
    return ptr


_STORE_GEOMETRY = {}   # store handle -> geometry, for the binding's size checks


# --------------------------------------------------------------------- API

def c2kv_last_error() -> str:
    return load_library().c2kv_last_error().decode()


def c2kv_version() -> str:
    return load_library().c2kv_version().decode()


def c2kv_store_create(geom, pinned_bytes: int) -> int:
    g = as_geometry(geom)
    h = ctypes.c_void_p()
    _check(load_library().c2kv_store_create(ctypes.byref(g), int(pinned_bytes), ctypes.byref(h)))
    _STORE_GEOMETRY[h.value] = c2kv_geometry(g.n_layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.rope_theta)
    return h.value


def c2kv_store_destroy(store: int) -> None:
    _STORE_GEOMETRY.pop(store, None)
    load_library().c2kv_store_destroy(store)


def c2kv_store_segments(store: int, doc_ids, n_tokens, n_slots, k: int, k_pre, v) -> None:
    """k_pre[i], v[i]: host bf16 bits [n_layers][n_kv_heads][n_slots[i]][head_dim]
    (numpy uint16 or a CPU tensor), checked against the store's geometry."""
    n = len(doc_ids)
    if not (len(n_tokens) == len(n_slots) == len(k_pre) == len(v) == n):
        raise ValueError("doc_ids, n_tokens, n_slots, k_pre and v must have one entry per document")
    g = _STORE_GEOMETRY.get(store)
    row = None if g is None else g.n_layers * g.n_kv_heads * g.head_dim * 2
    sizes = [None if row is None or int(s) < 1 else row * int(s) for s in n_slots]
    keep = list(k_pre) + list(v)   # keep the arrays alive through the call
    kp = (ctypes.c_void_p * max(1, n))(*[_host_ptr(a, b, f"k_pre[{i}]") for i, (a, b) in enumerate(zip(k_pre, sizes))])
    vp = (ctypes.c_void_p * max(1, n))(*[_host_ptr(a, b, f"v[{i}]") for i, (a, b) in enumerate(zip(v, sizes))])
    _check(load_library().c2kv_store_segments(store, n, _i32arr(doc_ids), _i32arr(n_tokens),
                                              _i32arr(n_slots), int(k), kp, vp))
    del keep


def c2kv_store_lookup(store: int, doc_id: int):
    nt, ns, k = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().c2kv_store_lookup(store, int(doc_id), ctypes.byref(nt), ctypes.byref(ns),
                                            ctypes.byref(k)))
    return nt.value, ns.value, k.value


def c2kv_plan(n_tokens: Sequence[int], n_slots: Sequence[int], order: Optional[Sequence[int]] = None):
    """Returns (slot_start[c], pos_offset[c], total_slots, total_tokens)."""
    n = len(n_tokens)
    ss, po = _i32arr([0] * n), _i32arr([0] * n)
    ts, tt = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().c2kv_plan(n, _i32arr(n_tokens), _i32arr(n_slots),
                                    None if order is None else _i32arr(order), ss, po,
                                    ctypes.byref(ts), ctypes.byref(tt)))
    return list(ss)[:n], list(po)[:n], ts.value, tt.value


def _check_compose_buffers(store, k_cache, v_cache, cap, rope_table, pos_dev_out) -> None:
    """Caches [n_layers][n_kv_heads][cap][head_dim] bf16, a RoPE table of cap
    rows and pos_dev_out of cap entries, for stores made through this module
    (whose geometry it knows)."""
    g = _STORE_GEOMETRY.get(store)
    if g is None or int(cap) <= 0:
        return
    cache = 2 * g.n_layers * g.n_kv_heads * int(cap) * g.head_dim
    _need(k_cache, cache, "k_cache")
    _need(v_cache, cache, "v_cache")
    _need(rope_table, c2kv_rope_table_bytes(g, int(cap)), "rope_table")
    if pos_dev_out is not None:
        _need(pos_dev_out, 4 * int(cap), "pos_dev_out")


def c2kv_compose(store: int, doc_ids, order, k: int, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 cap: int, rope_table: torch.Tensor, pos_dev_out: Optional[torch.Tensor] = None, stream=None):
    """Returns (n_slots, next_pos).  rope_table: device buffer of
    c2kv_rope_table_bytes(geom, cap) bytes (any dtype)."""
    _check_compose_buffers(store, k_cache, v_cache, cap, rope_table, pos_dev_out)
    ns, nxt = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().c2kv_compose(
        store, len(doc_ids), _i32arr(doc_ids), None if order is None else _i32arr(order), int(k),
        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"), int(cap),
        _dev(rope_table, None, "rope_table"), _dev(pos_dev_out, torch.int32, "pos_dev_out"),
        ctypes.byref(ns), ctypes.byref(nxt), _stream(stream)))
    return ns.value, nxt.value


C2KV_COMPOSE_NO_REALIGN = 1
C2KV_COMPOSE_CONTINUE = 2


def c2kv_compose_layers(store: int, doc_ids, order, k: int, flags: int, layer_begin: int, layer_end: int,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, cap: int, rope_table: torch.Tensor,
                        pos_dev_out: Optional[torch.Tensor] = None, stream=None):
    """c2kv_compose over layers [layer_begin, layer_end) with C2KV_COMPOSE_* flags.
    Returns (n_slots, next_pos)."""
    _check_compose_buffers(store, k_cache, v_cache, cap, rope_table, pos_dev_out)
    ns, nxt = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().c2kv_compose_layers(
        store, len(doc_ids), _i32arr(doc_ids), None if order is None else _i32arr(order), int(k), int(flags),
        int(layer_begin), int(layer_end), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), int(cap), _dev(rope_table, None, "rope_table"),
        _dev(pos_dev_out, torch.int32, "pos_dev_out"), ctypes.byref(ns), ctypes.byref(nxt), _stream(stream)))
    return ns.value, nxt.value


def c2kv_rope_table_bytes(geom, rows: int) -> int:
    g = as_geometry(geom)
    return int(load_library().c2kv_rope_table_bytes(ctypes.byref(g), int(rows)))


def c2kv_rope_table(geom, pos_dev: torch.Tensor, table_out: torch.Tensor, stream=None) -> None:
    g = as_geometry(geom)
    _need(table_out, c2kv_rope_table_bytes(g, pos_dev.numel()), "table_out")
    _check(load_library().c2kv_rope_table(ctypes.byref(g), _dev(pos_dev, torch.int32, "pos_dev"),
                                          pos_dev.numel(), _dev(table_out, None, "table_out"),
                                          _stream(stream)))


def c2kv_attend_workspace_size(geom, batch: int, t_len: int, max_keys: int) -> int:
    g = as_geometry(geom)
    return int(load_library().c2kv_attend_workspace_size(ctypes.byref(g), batch, t_len, max_keys))


def c2kv_masked_extra_bytes(geom, n_tokens: int) -> int:
    g = as_geometry(geom)
    return int(load_library().c2kv_masked_extra_bytes(ctypes.byref(g), n_tokens))


def c2kv_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _check(load_library().c2kv_workspace_init(_dev(workspace, None, "workspace"),
                                              workspace.numel() * workspace.element_size(),
                                              _stream(stream)))


def _ptrs(ts, name):
    return (ctypes.c_void_p * len(ts))(*[_dev(t, torch.bfloat16, name) for t in ts])


def _tabs(ts):
    return (ctypes.c_void_p * len(ts))(*[_dev(t, None, "rope_table") for t in ts])


def _check_request_state(g, k_caches, v_caches, rope_tables, cap: int) -> None:
    """Per-sequence caches [n_layers][n_kv_heads][cap][head_dim] bf16 and RoPE
    tables of cap rows, one of each per sequence."""
    B = len(k_caches)
    if not (len(v_caches) == len(rope_tables) == B):
        raise ValueError("k_caches, v_caches and rope_tables need one entry per sequence")
    cache = 2 * g.n_layers * g.n_kv_heads * max(0, int(cap)) * g.head_dim
    table = c2kv_rope_table_bytes(g, max(0, int(cap)))
    for b in range(B):
        _need(k_caches[b], cache, f"k_caches[{b}]")
        _need(v_caches[b], cache, f"v_caches[{b}]")
        _need(rope_tables[b], table, f"rope_tables[{b}]")


def _check_decode_args(g, k_caches, v_caches, rope_tables, cap, n_cached_dev, q, k_new, v_new, out) -> None:
    B = len(k_caches)
    _check_request_state(g, k_caches, v_caches, rope_tables, cap)
    _need(n_cached_dev, 4 * B, "n_cached_dev")
    _need(q, 2 * B * g.n_q_heads * g.head_dim, "q", exact=True)
    _need(k_new, 2 * B * g.n_kv_heads * g.head_dim, "k_new", exact=True)
    _need(v_new, 2 * B * g.n_kv_heads * g.head_dim, "v_new", exact=True)
    _need(out, 2 * B * g.n_q_heads * g.head_dim, "out", exact=True)


def c2kv_attend_prefill(geom, layer: int, k_caches, v_caches, rope_tables, cap: int, n_cached,
                        q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, out: torch.Tensor,
                        workspace: Optional[torch.Tensor], stream=None) -> None:
    g = as_geometry(geom)
    B = len(k_caches)
    q_len = q.shape[1]
    _check_request_state(g, k_caches, v_caches, rope_tables, cap)
    if len(n_cached) != B:
        raise ValueError("n_cached needs one entry per sequence")
    _need(q, 2 * B * q_len * g.n_q_heads * g.head_dim, "q", exact=True)
    _need(k_new, 2 * B * q_len * g.n_kv_heads * g.head_dim, "k_new", exact=True)
    _need(v_new, 2 * B * q_len * g.n_kv_heads * g.head_dim, "v_new", exact=True)
    _need(out, 2 * B * q_len * g.n_q_heads * g.head_dim, "out", exact=True)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().c2kv_attend_prefill(
        ctypes.byref(g), int(layer), B, _ptrs(k_caches, "k_cache"), _ptrs(v_caches, "v_cache"),
        _tabs(rope_tables), int(cap), _i32arr(n_cached), int(q_len), _dev(q, torch.bfloat16, "q"),
        _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(out, torch.bfloat16, "out"), _dev(workspace, None, "workspace"), ws, _stream(stream)))


C2KV_DECODE_OVERLAP_PREVIOUS = 1


def c2kv_attend_decode(geom, layer: int, k_caches, v_caches, rope_tables, cap: int, n_cached_dev: torch.Tensor,
                       max_keys: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       out: torch.Tensor, workspace: Optional[torch.Tensor], stream=None, flags: int = 0) -> None:
    g = as_geometry(geom)
    B = len(k_caches)
    _check_decode_args(g, k_caches, v_caches, rope_tables, cap, n_cached_dev, q, k_new, v_new, out)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().c2kv_attend_decode(
        ctypes.byref(g), int(layer), B, _ptrs(k_caches, "k_cache"), _ptrs(v_caches, "v_cache"),
        _tabs(rope_tables), int(cap), _dev(n_cached_dev, torch.int32, "n_cached_dev"), int(max_keys),
        _dev(q, torch.bfloat16, "q"), _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(out, torch.bfloat16, "out"), _dev(workspace, None, "workspace"), ws, int(flags), _stream(stream)))


def c2kv_attend_decode_noalloc(geom, layer: int, k_caches, v_caches, rope_tables, cap: int,
                               n_cached_dev: torch.Tensor, max_keys: int, q: torch.Tensor, k_new: torch.Tensor,
                               v_new: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """c2kv_attend_decode for callers that cannot allocate device memory: the
    split-K scratch is the library's own fixed 4 MiB device array (shared by
    all calls, so calls must not overlap on the GPU)."""
    g = as_geometry(geom)
    B = len(k_caches)
    _check_decode_args(g, k_caches, v_caches, rope_tables, cap, n_cached_dev, q, k_new, v_new, out)
    _check(load_library().c2kv_attend_decode_noalloc(
        ctypes.byref(g), int(layer), B, _ptrs(k_caches, "k_cache"), _ptrs(v_caches, "v_cache"),
        _tabs(rope_tables), int(cap), _dev(n_cached_dev, torch.int32, "n_cached_dev"), int(max_keys),
        _dev(q, torch.bfloat16, "q"), _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
        _dev(out, torch.bfloat16, "out"), _stream(stream)))


def c2kv_seq_advance(n_cached_dev: torch.Tensor, delta: int = 1, stream=None) -> None:
    _check(load_library().c2kv_seq_advance(n_cached_dev.numel(), _dev(n_cached_dev, torch.int32),
                                           int(delta), _stream(stream)))


def c2kv_attend_masked(geom, mask: int, n_doc: int, n_slot: int, k: int, q: torch.Tensor,
                       kk: torch.Tensor, v: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                       stream=None) -> None:
    g = as_geometry(geom)
    N = int(n_doc) + int(n_slot)
    _need(q, 2 * N * g.n_q_heads * g.head_dim, "q", exact=True)
    _need(kk, 2 * N * g.n_kv_heads * g.head_dim, "kk", exact=True)
    _need(v, 2 * N * g.n_kv_heads * g.head_dim, "v", exact=True)
    _need(out, 2 * N * g.n_q_heads * g.head_dim, "out", exact=True)
    _check(load_library().c2kv_attend_masked(
        ctypes.byref(g), int(mask), int(n_doc), int(n_slot), int(k), _dev(q, torch.bfloat16, "q"),
        _dev(kk, torch.bfloat16, "kk"), _dev(v, torch.bfloat16, "v"), _dev(out, torch.bfloat16, "out"),
        _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)))


def masked_workspace_bytes(geom, n_tokens: int) -> int:
    """Scratch bytes c2kv_attend_masked needs for one n_tokens sequence."""
    a = c2kv_attend_workspace_size(geom, 1, n_tokens, n_tokens)
    return ((a + 255) // 256) * 256 + c2kv_masked_extra_bytes(geom, n_tokens)


def c2kv_store_save(store: int, path: str) -> None:
    """Writes every stored document of `store` to `path`."""
    _check(load_library().c2kv_store_save(store, os.fsencode(path)))


def c2kv_store_load(store: int, path: str) -> None:
    """Adds the documents of a file written by c2kv_store_save to `store`."""
    _check(load_library().c2kv_store_load(store, os.fsencode(path)))


def c2kv_test_expire_next_waits(n_launches: int) -> None:
    """Test hook: the next n decode launches take their bounded-wait timeout path."""
    _check(load_library().c2kv_test_expire_next_waits(int(n_launches)))


def c2kv_device_error() -> int:
    code = ctypes.c_int32()
    _check(load_library().c2kv_device_error(ctypes.byref(code)))
    return code.value


def c2kv_kernel_launches() -> int:
    """Kernel launches the library has enqueued in this process (a launch
    captured into a CUDA graph counts once, at capture)."""
    n = ctypes.c_uint64()
    _check(load_library().c2kv_kernel_launches(ctypes.byref(n)))
    return n.value


# ---------------------------------------------------------------- decoder step
C2KV_LINEAR_STORE = 0
C2KV_LINEAR_ADD = 1
C2KV_LINEAR_SPLIT3 = 2
C2KV_LINEAR_SWIGLU = 3
C2KV_LINEAR_OVERLAP_PREVIOUS = 1


def c2kv_linear_workspace_size(tokens: int, n_out: int) -> int:
    return int(load_library().c2kv_linear_workspace_size(int(tokens), int(n_out)))


def c2kv_linear(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, workspace: torch.Tensor,
                epilogue: int = C2KV_LINEAR_STORE, residual: Optional[torch.Tensor] = None,
                y2: Optional[torch.Tensor] = None, y3: Optional[torch.Tensor] = None, split1: int = 0,
                split2: int = 0, stream=None, flags: int = 0) -> None:
    """y = x @ w.T on the tensor cores with an epilogue (see include/c2kv.h):
    x [tokens][k_in], w [n_out][k_in] bf16; y per the epilogue."""
    tokens, k_in = x.shape
    n_out = w.shape[0]
    if w.shape[1] != k_in:
        raise ValueError("w must be [n_out][k_in] with the k_in of x")
    width = {C2KV_LINEAR_SPLIT3: split1, C2KV_LINEAR_SWIGLU: n_out // 2}.get(epilogue, n_out)
    _need(y, 2 * tokens * width, "y", exact=True)
    if epilogue == C2KV_LINEAR_ADD:
        _need(residual, 2 * tokens * n_out, "residual", exact=True)
    if epilogue == C2KV_LINEAR_SPLIT3:
        _need(y2, 2 * tokens * (split2 - split1), "y2", exact=True)
        _need(y3, 2 * tokens * (n_out - split2), "y3", exact=True)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().c2kv_linear(
        _dev(x, torch.bfloat16, "x"), int(tokens), int(k_in), _dev(w, torch.bfloat16, "w"), int(n_out),
        int(epilogue), _dev(residual, torch.bfloat16, "residual"), _dev(y, torch.bfloat16, "y"),
        _dev(y2, torch.bfloat16, "y2"), _dev(y3, torch.bfloat16, "y3"), int(split1), int(split2),
        _dev(workspace, None, "workspace"), ws, int(flags), _stream(stream)))


def c2kv_rmsnorm(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, eps: float = 1e-5, stream=None,
                 flags: int = 0) -> None:
    tokens, dim = x.shape
    _need(w, 2 * dim, "w", exact=True)
    _need(y, 2 * tokens * dim, "y", exact=True)
    _check(load_library().c2kv_rmsnorm(_dev(x, torch.bfloat16, "x"), int(tokens), int(dim),
                                       _dev(w, torch.bfloat16, "w"), float(eps), _dev(y, torch.bfloat16, "y"),
                                       int(flags), _stream(stream)))
