"""Python binding of libmtkv (include/mtkv.h): the same entry points, by name.

Argument marshalling only: tensors become device pointers, Python lists of
moves become mt_move arrays, the current torch stream becomes the CUDA
stream. Every step of the path runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback, and calling any entry point without the built
library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmtkv.so")

MT_KV_F32, MT_KV_F16, MT_KV_Q8_0 = 0, 1, 2
FORMATS = {"f32": MT_KV_F32, "f16": MT_KV_F16, "q8_0": MT_KV_Q8_0}
MT_INVALID_BLOCK_ID = -1

STATUS_NAMES = {0: "MT_OK", 1: "MT_ERR_INVALID_ARG", 2: "MT_ERR_UNSUPPORTED", 3: "MT_ERR_ORDER",
                4: "MT_ERR_TIMEOUT", 5: "MT_ERR_DEVICE_CHECK", 6: "MT_ERR_CUDA"}
MT_OK, MT_ERR_INVALID_ARG, MT_ERR_UNSUPPORTED, MT_ERR_ORDER = 0, 1, 2, 3
MT_ERR_TIMEOUT, MT_ERR_DEVICE_CHECK, MT_ERR_CUDA = 4, 5, 6

EXPORTED = ("mt_kv_row_bytes", "mt_kv_store", "mt_paged_attn_workspace_bytes",
            "mt_paged_attn_decode", "mt_order_moves", "mt_check_moves", "mt_copy_cells",
            "mt_kv_quant_int4", "mt_kv_dequant_int4", "mt_kv_relayout", "mt_kv_grow_capacity",
            "mt_check_device_status", "mt_selftest_bounded_wait", "mt_last_error", "mt_version")


class MtError(RuntimeError):
    def __init__(self, status: int, where: str, reason: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {reason}")
        self.status = status


class mt_move(ctypes.Structure):
    _fields_ = [("src", ctypes.c_int64), ("dst", ctypes.c_int64), ("len", ctypes.c_int64)]


MT_KV_MAP_MAX_SPANS = 8


class mt_paged_prefill_args(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("q_start", ctypes.c_void_p),
                ("spans", ctypes.c_void_p), ("kv_map", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("n_seqs", ctypes.c_int),
                ("n_tokens", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("block_size", ctypes.c_int), ("max_blocks", ctypes.c_int),
                ("n_phys_blocks", ctypes.c_int64), ("scale", ctypes.c_float)]


class mt_prefix_group(ctypes.Structure):
    _fields_ = [("seq_begin", ctypes.c_int32), ("seq_end", ctypes.c_int32),
                ("n_prefix_blocks", ctypes.c_int32)]


class mt_paged_attn_args(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("spans", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("n_seqs", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("max_blocks", ctypes.c_int), ("n_phys_blocks", ctypes.c_int64),
                ("scale", ctypes.c_float), ("n_ctas", ctypes.c_int),
                ("kv_map", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmtkv.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmtkv is not built ({LIB_PATH} missing): run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ, U32P = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    sig = {
        "mt_kv_row_bytes": (SZ, [I, I, I]),
        "mt_kv_store": (I, [I, P, P, I64, I, I, P, P, P, I, U32P, P]),
        "mt_paged_attn_workspace_bytes": (SZ, [ctypes.POINTER(mt_paged_attn_args)]),
        "mt_paged_attn_decode": (I, [ctypes.POINTER(mt_paged_attn_args), P, SZ, P]),
        "mt_paged_attn_decode_append": (I, [ctypes.POINTER(mt_paged_attn_args), P, P, P, SZ, P]),
        "mt_paged_attn_decode_static": (I, [ctypes.POINTER(mt_paged_attn_args), U32P, P]),
        "mt_paged_prefill_workspace_bytes": (SZ, [ctypes.POINTER(mt_paged_prefill_args)]),
        "mt_paged_attn_prefill": (I, [ctypes.POINTER(mt_paged_prefill_args), P, SZ, P]),
        "mt_paged_attn_cascade_workspace_bytes": (SZ, [ctypes.POINTER(mt_paged_attn_args),
                                                       ctypes.POINTER(mt_prefix_group), I]),
        "mt_paged_attn_decode_cascade": (I, [ctypes.POINTER(mt_paged_attn_args),
                                             ctypes.POINTER(mt_prefix_group), I, P, SZ, P]),
        "mt_paged_attn_decode_cascade_append": (I, [ctypes.POINTER(mt_paged_attn_args),
                                                    ctypes.POINTER(mt_prefix_group), I, P, P, P,
                                                    SZ, P]),
        "mt_order_moves": (I, [ctypes.POINTER(mt_move), I, ctypes.POINTER(I)]),
        "mt_check_moves": (I, [ctypes.POINTER(mt_move), I, I64, ctypes.POINTER(I)]),
        "mt_copy_cells": (I, [ctypes.POINTER(P), I, SZ, I64, ctypes.POINTER(mt_move), I, U32P,
                              P]),
        "mt_kv_quant_int4": (I, [I, P, I, I, I, I64, P, I, P, P, U32P, P]),
        "mt_kv_dequant_int4": (I, [I, P, I, I, I, I64, P, I, P, P, U32P, P]),
        "mt_kv_relayout": (I, [P, P, I, I64, I64, SZ, P]),
        "mt_kv_grow_capacity": (I64, [I64, I64, I64]),
        "mt_check_device_status": (I, [U32P, P]),
        "mt_selftest_bounded_wait": (I, [ctypes.c_uint64, U32P, P]),
        "mt_last_error": (ctypes.c_char_p, []),
        "mt_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        if fmt not in FORMATS:
            raise ValueError(f"unknown KV format {fmt!r}")
        return FORMATS[fmt]
    return int(fmt)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str) -> None:
    if st != MT_OK:
        raise MtError(st, where, mt_last_error())


def mt_last_error() -> str:
    return lib().mt_last_error().decode()


def mt_version() -> str:
    return lib().mt_version().decode()


def mt_kv_row_bytes(fmt, n_kv_heads: int, head_dim: int) -> int:
    return int(lib().mt_kv_row_bytes(_fmt(fmt), n_kv_heads, head_dim))


def mt_kv_store(fmt, k_pool, v_pool, n_kv_heads, head_dim, k_new, v_new, cells,
                status=None, stream=None, n_cells=None) -> None:
    rb = mt_kv_row_bytes(fmt, n_kv_heads, head_dim)
    if n_cells is None:
        n_cells = k_pool.numel() * k_pool.element_size() // rb
    n_rows = int(cells.numel())
    _check(lib().mt_kv_store(_fmt(fmt), _ptr(k_pool), _ptr(v_pool), n_cells, n_kv_heads,
                             head_dim, _ptr(k_new), _ptr(v_new), _ptr(cells), n_rows,
                             _ptr(status), _stream(stream)), "mt_kv_store")


def paged_attn_args(fmt, q, k_pool, v_pool, block_table, context_lens, out, *, n_kv_heads,
                    block_size, n_phys_blocks, scale, spans=None, lse=None, n_ctas=0,
                    kv_map=None):
    B, Hq, D = q.shape
    a = mt_paged_attn_args()
    a.fmt = _fmt(fmt)
    a.q, a.k_pool, a.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    a.block_table, a.context_lens = _ptr(block_table), _ptr(context_lens)
    a.spans = _ptr(spans)
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.n_seqs, a.n_heads, a.n_kv_heads, a.head_dim = B, Hq, n_kv_heads, D
    a.block_size = block_size
    a.max_blocks = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    a.n_phys_blocks = int(n_phys_blocks)
    a.scale = float(scale)
    a.n_ctas = int(n_ctas)
    # the struct holds raw addresses: keep the tensors alive as long as it is
    a.kv_map = _ptr(kv_map)
    a._tensors = (q, k_pool, v_pool, block_table, context_lens, out, spans, lse, kv_map)
    return a


def mt_paged_attn_workspace_bytes(args: mt_paged_attn_args) -> int:
    return int(lib().mt_paged_attn_workspace_bytes(ctypes.byref(args)))


def mt_paged_attn_decode(args: mt_paged_attn_args, workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().mt_paged_attn_decode(ctypes.byref(args), _ptr(workspace), nbytes,
                                      _stream(stream)), "mt_paged_attn_decode")


def mt_paged_attn_decode_append(args: mt_paged_attn_args, k_new, v_new, workspace,
                                stream=None) -> None:
    """Decode with each sequence's new K/V row (float32 [n_seqs][Hkv*d])
    stored into the cell of position context_lens[s]-1 in the same launch."""
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().mt_paged_attn_decode_append(ctypes.byref(args), _ptr(k_new), _ptr(v_new),
                                             _ptr(workspace), nbytes, _stream(stream)),
           "mt_paged_attn_decode_append")


def prefill_args(fmt, q, k_pool, v_pool, block_table, context_lens, q_start, out, *,
                 n_kv_heads, block_size, n_phys_blocks, scale, spans=None, kv_map=None,
                 lse=None):
    """Arguments of mt_paged_attn_prefill from device tensors: q [n_tokens][Hq][d],
    q_start int32 [n_seqs + 1], spans [n_tokens][2] or kv_map
    [n_tokens][MT_KV_MAP_MAX_SPANS][2] (optional)."""
    n_tok, Hq, D = q.shape
    a = mt_paged_prefill_args()
    a.fmt = _fmt(fmt)
    a.q, a.k_pool, a.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    a.block_table, a.context_lens, a.q_start = _ptr(block_table), _ptr(context_lens), _ptr(q_start)
    a.spans, a.kv_map = _ptr(spans), _ptr(kv_map)
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.n_seqs = int(context_lens.numel())
    a.n_tokens, a.n_heads, a.n_kv_heads, a.head_dim = n_tok, Hq, n_kv_heads, D
    a.block_size = block_size
    a.max_blocks = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    a.n_phys_blocks = int(n_phys_blocks)
    a.scale = float(scale)
    a._tensors = (q, k_pool, v_pool, block_table, context_lens, q_start, spans, kv_map, out, lse)
    return a


def mt_paged_prefill_workspace_bytes(args: mt_paged_prefill_args) -> int:
    return int(lib().mt_paged_prefill_workspace_bytes(ctypes.byref(args)))


def mt_paged_attn_prefill(args: mt_paged_prefill_args, workspace, stream=None) -> None:
    """Multi-query (prefill) attention through the paged cache."""
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().mt_paged_attn_prefill(ctypes.byref(args), _ptr(workspace), nbytes,
                                       _stream(stream)), "mt_paged_attn_prefill")


def _groups_array(groups):
    """mt_prefix_group array for (seq_begin, seq_end, n_prefix_blocks) triples."""
    n = len(groups)
    arr = (mt_prefix_group * max(n, 1))()
    for i, (b, e, nb) in enumerate(groups):
        arr[i].seq_begin, arr[i].seq_end, arr[i].n_prefix_blocks = int(b), int(e), int(nb)
    return arr, n


def mt_paged_attn_cascade_workspace_bytes(args: mt_paged_attn_args, groups) -> int:
    arr, n = _groups_array(groups)
    return int(lib().mt_paged_attn_cascade_workspace_bytes(ctypes.byref(args), arr, n))


def mt_paged_attn_decode_cascade(args: mt_paged_attn_args, groups, workspace,
                                 stream=None) -> None:
    """Decode where the sequences of each group (seq_begin, seq_end,
    n_prefix_blocks) share their first n_prefix_blocks block-table entries:
    each shared block is read once per KV head for the whole group."""
    arr, n = _groups_array(groups)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().mt_paged_attn_decode_cascade(ctypes.byref(args), arr, n, _ptr(workspace),
                                              nbytes, _stream(stream)),
           "mt_paged_attn_decode_cascade")


def mt_paged_attn_decode_cascade_append(args: mt_paged_attn_args, groups, k_new, v_new,
                                        workspace, stream=None) -> None:
    """Cascade decode with each sequence's new K/V row stored at position
    context_lens[s]-1 in the same call."""
    arr, n = _groups_array(groups)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().mt_paged_attn_decode_cascade_append(ctypes.byref(args), arr, n, _ptr(k_new),
                                                     _ptr(v_new), _ptr(workspace), nbytes,
                                                     _stream(stream)),
           "mt_paged_attn_decode_cascade_append")


MT_STATIC_SCRATCH_BYTES = 8 << 20


def mt_paged_attn_decode_static(args: mt_paged_attn_args, status=None, stream=None) -> None:
    """Decode with the library's built-in scratch array instead of a workspace
    (for callers that cannot allocate device memory when they decode)."""
    _check(lib().mt_paged_attn_decode_static(ctypes.byref(args), _ptr(status), _stream(stream)),
           "mt_paged_attn_decode_static")


def _moves_array(moves):
    """mt_move array for `moves`: (src, dst, len) triples, or an int64 numpy
    array of shape (n, 3), which is passed without copying."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(moves, dtype=np.int64).reshape(-1, 3))
    if a.shape[0] == 0:
        a = np.zeros((1, 3), dtype=np.int64)
    ptr = a.ctypes.data_as(ctypes.POINTER(mt_move))
    ptr._keep = a  # the array must outlive the call
    return ptr


def mt_order_moves(moves):
    arr = _moves_array(moves)
    n_out = ctypes.c_int(0)
    _check(lib().mt_order_moves(arr, len(moves), ctypes.byref(n_out)), "mt_order_moves")
    return [tuple(int(v) for v in r) for r in arr._keep[:n_out.value]]


def mt_check_moves(moves, n_cells: int):
    """Returns (status, first_bad) without raising."""
    arr = _moves_array(moves)
    bad = ctypes.c_int(-1)
    st = lib().mt_check_moves(arr, len(moves), int(n_cells), ctypes.byref(bad))
    return st, bad.value


def mt_copy_cells(pools, row_bytes: int, n_cells: int, moves, status=None,
                  stream=None) -> None:
    ptrs = (ctypes.c_void_p * max(1, len(pools)))(*[_ptr(p) for p in pools])
    arr = _moves_array(moves)
    _check(lib().mt_copy_cells(ptrs, len(pools), int(row_bytes), int(n_cells), arr, len(moves),
                               _ptr(status), _stream(stream)), "mt_copy_cells")


def mt_kv_quant_int4(fmt, pool, block_size, n_kv_heads, head_dim, n_phys_blocks, blocks,
                     scales, nibbles, status=None, stream=None) -> None:
    _check(lib().mt_kv_quant_int4(_fmt(fmt), _ptr(pool), block_size, n_kv_heads, head_dim,
                                  int(n_phys_blocks), _ptr(blocks), int(blocks.numel()),
                                  _ptr(scales), _ptr(nibbles), _ptr(status), _stream(stream)),
           "mt_kv_quant_int4")


def mt_kv_dequant_int4(fmt, pool, block_size, n_kv_heads, head_dim, n_phys_blocks, dst_blocks,
                       scales, nibbles, status=None, stream=None) -> None:
    _check(lib().mt_kv_dequant_int4(_fmt(fmt), _ptr(pool), block_size, n_kv_heads, head_dim,
                                    int(n_phys_blocks), _ptr(dst_blocks),
                                    int(dst_blocks.numel()), _ptr(scales), _ptr(nibbles),
                                    _ptr(status), _stream(stream)), "mt_kv_dequant_int4")


def mt_kv_relayout(src, dst, n_layers: int, old_cap: int, new_cap: int, row_bytes: int,
                   stream=None) -> None:
    _check(lib().mt_kv_relayout(_ptr(src), _ptr(dst), n_layers, old_cap, new_cap, row_bytes,
                                _stream(stream)), "mt_kv_relayout")


def mt_kv_grow_capacity(cap: int, need: int, max_ctx: int) -> int:
    return int(lib().mt_kv_grow_capacity(cap, need, max_ctx))


def mt_selftest_bounded_wait(limit_ns: int, status, stream=None) -> None:
    """Run the bounded-wait self-test kernel (sets the timeout bit in `status`)."""
    _check(lib().mt_selftest_bounded_wait(int(limit_ns), _ptr(status), _stream(stream)),
           "mt_selftest_bounded_wait")


def mt_check_device_status(status_word, stream=None) -> int:
    """Synchronise, read and clear a device status word; returns the mt_status."""
    return int(lib().mt_check_device_status(_ptr(status_word), _stream(stream)))
