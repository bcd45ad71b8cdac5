"""CPU oracle for sparse MLA attention (test infrastructure only).

This package is the checker, not the product. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library under
``sparse_mla_attention_top_gb300`` never does, and the two share no code.

The arithmetic lives in ``oracle.cpp`` (plain loops, fp64). This module compiles it with
g++ and wraps each entry point for numpy arrays. Every function cites the passage it
follows in its C++ docstring; see the header comment of ``oracle.cpp`` for the sources.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.cpp"
_LIB_PATH = _HERE / "liboracle.so"
_lib = None

ROW = 576
VDIM = 512
KV_BF16 = 0
KV_FP8_E4M3 = 1
ERR_RANGE = 1
ERR_DUPLICATE = 2


def build(force: bool = False) -> Path:
    """Compile oracle.cpp into liboracle.so next to it (g++, OpenMP, -O2)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared", str(_SRC), "-o", str(tmp)]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB_PATH))
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_e4m3_table.argtypes = [P]
        lib.oracle_resolve.argtypes = [P, i32, i32, P, P, P, i32, P, i32, i64, P]
        lib.oracle_resolve.restype = i32
        lib.oracle_decode.argtypes = [P, i32, i32, P, i32, i64, i64, i32, P, i32, P, P, P, i32, P, f64, P, i32, P, P]
        lib.oracle_decode.restype = i32
        lib.oracle_group_union.argtypes = [P, P, i32, i32, i32, i64, P, P]
        lib.oracle_group_union.restype = i32
        lib.oracle_prefill_grouped.argtypes = [P, i32, i32, i32, P, i32, i64, i64, P, P, i32, f64, P, i32, P, P]
        lib.oracle_prefill_grouped.restype = i32
        lib.oracle_dense_paged.argtypes = [P, i32, P, i32, i64, P, i32, i32, f64, P, P]
        lib.oracle_merge.argtypes = [P, P, i32, i64, P, P]
        lib.oracle_attend_slots.argtypes = [P, i32, P, i32, i64, P, i32, f64, P, P]
        lib.oracle_fetch_rows.argtypes = [P, i32, i64, P, i32, P]
        lib.oracle_topk_select.argtypes = [P, i32, i32, i64, P, i32, P]
        lib.oracle_num_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())


def e4m3_table() -> np.ndarray:
    out = np.empty(256, np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def resolve(topk, topk_len=None, req_of_token=None, block_table=None, seq_lens=None,
            page_size=1, num_pages=0):
    """Slots [T, K] int64 (-1 for dead entries) and the error bits."""
    topk = _c(topk, np.int32)
    T, K = topk.shape
    bt = _c(block_table, np.int32)
    max_blocks = 0 if bt is None else bt.shape[1]
    out = np.empty((T, K), np.int64)
    err = _load().oracle_resolve(_ptr(topk), T, K, _ptr(_c(topk_len, np.int32)), _ptr(_c(req_of_token, np.int32)),
                                 _ptr(bt), max_blocks, _ptr(_c(seq_lens, np.int32)), page_size, num_pages, _ptr(out))
    return out, int(err)


def _kv_args(kv_bytes, kv_dtype, row_stride):
    kv_bytes = np.ascontiguousarray(kv_bytes).view(np.uint8)
    if row_stride is None:
        row_stride = 1152 if kv_dtype == KV_BF16 else 656
    return kv_bytes, int(row_stride)


def decode(q_bits, kv_bytes, kv_dtype, num_pages, page_size, topk, scale, *, block_table=None,
           req_of_token=None, seq_lens=None, topk_len=None, query_ids=None, row_stride=None):
    """Sparse MLA decode for the chosen queries. q_bits: [T, H, 576] bf16 bit patterns (uint16).
    Returns (out [n, H, 512] fp64, lse [n, H] fp64, error bits)."""
    q_bits = _c(q_bits, np.uint16)
    T, H, _ = q_bits.shape
    topk = _c(topk, np.int32)
    K = topk.shape[1]
    ids = np.arange(T, dtype=np.int32) if query_ids is None else _c(query_ids, np.int32)
    kv_bytes, row_stride = _kv_args(kv_bytes, kv_dtype, row_stride)
    bt = _c(block_table, np.int32)
    max_blocks = 0 if bt is None else bt.shape[1]
    out = np.empty((len(ids), H, VDIM), np.float64)
    lse = np.empty((len(ids), H), np.float64)
    err = _load().oracle_decode(_ptr(q_bits), T, H, _ptr(kv_bytes), kv_dtype, row_stride, num_pages, page_size,
                                _ptr(bt), max_blocks, _ptr(_c(req_of_token, np.int32)), _ptr(_c(seq_lens, np.int32)),
                                _ptr(topk), K, _ptr(_c(topk_len, np.int32)), float(scale), _ptr(ids), len(ids),
                                _ptr(out), _ptr(lse))
    return out, lse, int(err)


def group_union(slots, G, num_slots, topk_len=None):
    """(enc [ceil(T/G), G*K] int32, lens [ceil(T/G)] int32, error bits)."""
    slots = _c(slots, np.int32)
    T, K = slots.shape
    groups = (T + G - 1) // G
    enc = np.empty((groups, G * K), np.int32)
    lens = np.empty(groups, np.int32)
    err = _load().oracle_group_union(_ptr(slots), _ptr(_c(topk_len, np.int32)), T, K, G, int(num_slots),
                                     _ptr(enc), _ptr(lens))
    return enc, lens, int(err)


def prefill_grouped(q_bits, G, kv_bytes, kv_dtype, num_slots, enc, lens, K, scale, *, query_ids=None,
                    row_stride=None):
    """Grouped prefill for the chosen queries: (out [n, H, 512], lse [n, H], error bits)."""
    q_bits = _c(q_bits, np.uint16)
    T, H, _ = q_bits.shape
    ids = np.arange(T, dtype=np.int32) if query_ids is None else _c(query_ids, np.int32)
    kv_bytes, row_stride = _kv_args(kv_bytes, kv_dtype, row_stride)
    enc = _c(enc, np.int32)
    lens = _c(lens, np.int32)
    out = np.empty((len(ids), H, VDIM), np.float64)
    lse = np.empty((len(ids), H), np.float64)
    err = _load().oracle_prefill_grouped(_ptr(q_bits), T, H, G, _ptr(kv_bytes), kv_dtype, row_stride,
                                         int(num_slots), _ptr(enc), _ptr(lens), K, float(scale), _ptr(ids),
                                         len(ids), _ptr(out), _ptr(lse))
    return out, lse, int(err)


def dense_paged(q_heads_bits, kv_bytes, kv_dtype, block_table_row, ctx, page_size, scale, row_stride=None):
    """Dense paged attention of one request over all its ctx positions: (out [H,512], lse [H])."""
    q = _c(q_heads_bits, np.uint16)
    H = q.shape[0]
    kv_bytes, row_stride = _kv_args(kv_bytes, kv_dtype, row_stride)
    out = np.empty((H, VDIM), np.float64)
    lse = np.empty(H, np.float64)
    _load().oracle_dense_paged(_ptr(q), H, _ptr(kv_bytes), kv_dtype, row_stride,
                               _ptr(_c(block_table_row, np.int32)), int(ctx), int(page_size), float(scale),
                               _ptr(out), _ptr(lse))
    return out, lse


def merge(o_part, lse_part):
    """Merge split partials: o_part [S, ..., 512] fp32, lse_part [S, ...] fp32 -> (out, lse) fp64."""
    o_part = _c(o_part, np.float32)
    lse_part = _c(lse_part, np.float32)
    S = o_part.shape[0]
    lead = lse_part.shape[1:]
    R = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (VDIM,), np.float64)
    lse = np.empty(lead, np.float64)
    _load().oracle_merge(_ptr(o_part), _ptr(lse_part), S, R, _ptr(out), _ptr(lse))
    return out, lse


def attend_slots(q_rows, kv_bytes, kv_dtype, slots, scale, row_stride=None):
    """Attention of explicit fp64 query rows [n, 576] over explicit slots: (out [n,512], lse [n])."""
    q = _c(np.atleast_2d(q_rows), np.float64)
    slots = _c(slots, np.int64)
    kv_bytes, row_stride = _kv_args(kv_bytes, kv_dtype, row_stride)
    out = np.empty((q.shape[0], VDIM), np.float64)
    lse = np.empty(q.shape[0], np.float64)
    _load().oracle_attend_slots(_ptr(q), q.shape[0], _ptr(kv_bytes), kv_dtype, row_stride, _ptr(slots),
                                len(slots), float(scale), _ptr(out), _ptr(lse))
    return out, lse


def fetch_rows(kv_bytes, kv_dtype, slots, row_stride=None):
    """The oracle's fp64 view of cache rows [n, 576]."""
    slots = _c(slots, np.int64)
    kv_bytes, row_stride = _kv_args(kv_bytes, kv_dtype, row_stride)
    rows = np.empty((len(slots), ROW), np.float64)
    _load().oracle_fetch_rows(_ptr(kv_bytes), kv_dtype, row_stride, _ptr(slots), len(slots), _ptr(rows))
    return rows


def topk_select(scores, K, lens=None):
    """Top-k positions per query row of `scores` [T, N] fp32 (ascending, -1 padded) -> [T, K] int32."""
    scores = _c(scores, np.float32)
    T, N = scores.shape
    out = np.empty((T, K), np.int32)
    _load().oracle_topk_select(_ptr(scores), T, N, N, _ptr(_c(lens, np.int32)), int(K), _ptr(out))
    return out
