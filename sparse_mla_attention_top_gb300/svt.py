"""Thin Python binding of libsvt.so (ctypes).

Argument marshalling only: every function takes torch tensors on the current CUDA device,
checks dtypes and shapes, passes raw pointers and the current stream to the C ABI, and
raises SvtError on a non-OK status. All computation happens in the library's kernels; there
is no fallback. The names follow the C entry points in include/svt.h.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path
from typing import Optional

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libsvt.so"
_lib = None

SVT_OK, SVT_ERR_INVALID_ARG, SVT_ERR_UNSUPPORTED, SVT_ERR_WORKSPACE, SVT_ERR_CUDA = range(5)
STATUS_NAMES = {0: "SVT_OK", 1: "SVT_ERR_INVALID_ARG", 2: "SVT_ERR_UNSUPPORTED", 3: "SVT_ERR_WORKSPACE",
                4: "SVT_ERR_CUDA"}
DEV_ERR_INDEX_RANGE = 0x1
DEV_ERR_TIMEOUT = 0x2
DEV_ERR_FP8_RANGE = 0x4
KV_BF16 = 0
KV_FP8_E4M3 = 1
ROW_BYTES = {KV_BF16: 1152, KV_FP8_E4M3: 656}

EXPORTED = [
    "svt_last_error_string", "svt_workspace_init", "svt_read_status", "svt_resolve_workspace_size",
    "svt_resolve_topk_slots", "svt_sparse_mla_decode_workspace_size", "svt_sparse_mla_decode",
    "svt_build_group_union_workspace_size", "svt_build_group_union",
    "svt_sparse_mla_prefill_grouped_workspace_size", "svt_sparse_mla_prefill_grouped",
    "svt_sparse_mla_prefill_grouped_union_tile", "svt_merge_splits",
    "svt_topk_select",
    "svt_sparse_mla_decode_noalloc", "svt_debug_pipeline_fault", "svt_gather_probe", "svt_tensor_probe",
]


class SvtError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _KV(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("num_pages", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("row_stride_bytes", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def library_path() -> Path:
    return _LIB_PATH


def use_library(path) -> None:
    """Loads the library from `path` instead of libsvt.so (the phase-trace build, for
    profiling); must come before the first call into the library."""
    global _LIB_PATH
    if _lib is not None:
        raise RuntimeError("the library is already loaded")
    _LIB_PATH = Path(path)


def lib():
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH} is missing: build it first (sparse_mla_attention_top_gb300.build)")
        L = ctypes.CDLL(str(_LIB_PATH))
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        L.svt_last_error_string.restype = ctypes.c_char_p
        L.svt_workspace_init.argtypes = [P, sz, P]
        L.svt_read_status.argtypes = [P, P, P]
        L.svt_resolve_workspace_size.restype = sz
        L.svt_resolve_topk_slots.argtypes = [P, i32, i32, P, P, P, i32, i32, P, i32, i64, P, P, sz, P]
        L.svt_sparse_mla_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        L.svt_sparse_mla_decode_workspace_size.restype = sz
        L.svt_sparse_mla_decode.argtypes = [P, i32, i32, ctypes.POINTER(_KV), P, i32, i32, P, P, P, i32, P, f32, P, P,
                                            i32, P, sz, P]
        L.svt_build_group_union_workspace_size.argtypes = [i32, i32, i32]
        L.svt_build_group_union_workspace_size.restype = sz
        L.svt_build_group_union.argtypes = [P, P, i32, i32, i32, i64, P, P, P, sz, P]
        L.svt_sparse_mla_prefill_grouped_workspace_size.argtypes = [i32, i32, i32]
        L.svt_sparse_mla_prefill_grouped_workspace_size.restype = sz
        L.svt_sparse_mla_prefill_grouped.argtypes = [P, i32, i32, i32, ctypes.POINTER(_KV), P, P, i32, f32, P, P, P,
                                                     sz, P]
        L.svt_sparse_mla_prefill_grouped_union_tile.argtypes = L.svt_sparse_mla_prefill_grouped.argtypes
        L.svt_merge_splits.argtypes = [P, P, i32, i32, i32, P, P, P]
        L.svt_topk_select.argtypes = [P, i32, i32, i64, P, i32, P, P]
        L.svt_sparse_mla_decode_noalloc.argtypes = [P, i32, i32, ctypes.POINTER(_KV), P, i32, i32, P, P, P, i32, P, f32,
                                                    P, P, i32, P, P]
        L.svt_debug_pipeline_fault.argtypes = [i32, i64]
        L.svt_gather_probe.argtypes = [ctypes.POINTER(_KV), P, i64, i32, P, P, sz, P]
        L.svt_tensor_probe.argtypes = [P, P, P, i32, i32, P, P, P, P, sz, P]
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != SVT_OK:
        msg = lib().svt_last_error_string()
        raise SvtError(status, where, msg.decode() if msg else "")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _i32(t: Optional[torch.Tensor], name: str) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


@dataclass
class KVCache:
    """A paged latent cache in device memory: `data` is uint8 [num_pages * page_size, row_bytes]
    (or any contiguous tensor with those bytes); dtype KV_BF16 or KV_FP8_E4M3."""
    data: torch.Tensor
    num_pages: int
    page_size: int
    dtype: int = KV_BF16
    row_stride_bytes: int = 0

    def _c(self) -> _KV:
        if not self.data.is_cuda or not self.data.is_contiguous():
            raise TypeError("kv data must be a contiguous CUDA tensor")
        return _KV(self.data.data_ptr(), int(self.num_pages), int(self.page_size), int(self.row_stride_bytes),
                   int(self.dtype))

    @property
    def num_slots(self) -> int:
        return int(self.num_pages) * int(self.page_size)


class Workspace:
    """Caller-owned scratch for one stream: a 256-byte status header plus per-call space.
    Grows on demand (allocation happens here, in torch, never inside the library)."""

    def __init__(self, device=None, nbytes: int = 256):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.buf = torch.zeros(max(256, nbytes), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> "Workspace":
        if nbytes > self.buf.numel():
            old = self.buf
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
            self.buf[:256].copy_(old[:256])  # keep pending status bits
        return self

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    def read_status(self, stream=None) -> int:
        out = ctypes.c_int32(0)
        _check(lib().svt_read_status(self.ptr, _stream(stream), ctypes.byref(out)), "svt_read_status")
        return int(out.value)


_default_ws = {}


def default_workspace() -> Workspace:
    dev = torch.cuda.current_device()
    if dev not in _default_ws:
        _default_ws[dev] = Workspace()
    return _default_ws[dev]


def resolve_topk_slots(topk_pos, *, block_table=None, seq_lens=None, req_of_token=None, topk_len=None,
                       page_size: int = 1, num_pages: int, out=None, ws: Optional[Workspace] = None):
    """svt_resolve_topk_slots: [T, K] positions -> [T, K] int32 slots (-1 for dead entries)."""
    topk_pos = _i32(topk_pos, "topk_pos")
    T, K = topk_pos.shape
    bt = _i32(block_table, "block_table")
    out = torch.empty((T, K), dtype=torch.int32, device=topk_pos.device) if out is None else out
    ws = (ws or default_workspace()).ensure(lib().svt_resolve_workspace_size())
    _check(lib().svt_resolve_topk_slots(_ptr(topk_pos), T, K, _ptr(_i32(topk_len, "topk_len")),
                                        _ptr(_i32(req_of_token, "req_of_token")), _ptr(bt),
                                        0 if bt is None else bt.shape[0], 0 if bt is None else bt.shape[1],
                                        _ptr(_i32(seq_lens, "seq_lens")), int(page_size), int(num_pages), _ptr(out),
                                        ws.ptr, ws.nbytes, _stream()), "svt_resolve_topk_slots")
    return out


def sparse_mla_decode(q, kv: KVCache, topk, softmax_scale: float, *, block_table=None, seq_lens=None,
                      req_of_token=None, topk_len=None, num_splits: int = 0, out=None, lse=None,
                      return_lse: bool = True, ws: Optional[Workspace] = None):
    """svt_sparse_mla_decode. q [T, H, 576] bf16; topk [T, K] int32 positions (slots when
    block_table is None). Returns (out [T, H, 512] bf16, lse [T, H] fp32 or None)."""
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != 576 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bf16 [T, H, 576] tensor")
    T, H, _ = q.shape
    topk = _i32(topk, "topk")
    K = topk.shape[1]
    bt = _i32(block_table, "block_table")
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    ws = (ws or default_workspace()).ensure(lib().svt_sparse_mla_decode_workspace_size(T, H, K, num_splits))
    kvc = kv._c()
    _check(lib().svt_sparse_mla_decode(_ptr(q), T, H, ctypes.byref(kvc), _ptr(bt), 0 if bt is None else bt.shape[0],
                                       0 if bt is None else bt.shape[1], _ptr(_i32(req_of_token, "req_of_token")),
                                       _ptr(_i32(seq_lens, "seq_lens")), _ptr(topk), K,
                                       _ptr(_i32(topk_len, "topk_len")), float(softmax_scale), _ptr(out), _ptr(lse),
                                       int(num_splits), ws.ptr, ws.nbytes, _stream()), "svt_sparse_mla_decode")
    return out, lse


def build_group_union(slots, G: int, num_slots: int, *, topk_len=None, enc=None, lens=None,
                      ws: Optional[Workspace] = None):
    """svt_build_group_union: slots [T, K] int32 -> (enc [ceil(T/G), G*K] int32, lens [ceil(T/G)] int32)."""
    slots = _i32(slots, "slots")
    T, K = slots.shape
    groups = (T + G - 1) // G
    if enc is None:
        enc = torch.empty((groups, G * K), dtype=torch.int32, device=slots.device)
    if lens is None:
        lens = torch.empty((groups,), dtype=torch.int32, device=slots.device)
    ws = (ws or default_workspace()).ensure(lib().svt_build_group_union_workspace_size(T, K, G))
    _check(lib().svt_build_group_union(_ptr(slots), _ptr(_i32(topk_len, "topk_len")), T, K, int(G), int(num_slots),
                                       _ptr(enc), _ptr(lens), ws.ptr, ws.nbytes, _stream()), "svt_build_group_union")
    return enc, lens


def sparse_mla_prefill_grouped(q, G: int, kv: KVCache, enc, lens, K: int, softmax_scale: float, *, out=None,
                               lse=None, return_lse: bool = True, ws: Optional[Workspace] = None,
                               union_tile: bool = False):
    """svt_sparse_mla_prefill_grouped (or, with union_tile, svt_sparse_mla_prefill_grouped_union_tile).
    q [T, H, 576] bf16 token-major, H * G = 128."""
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != 576 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bf16 [T, H, 576] tensor")
    T, H, _ = q.shape
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    ws = (ws or default_workspace()).ensure(lib().svt_sparse_mla_prefill_grouped_workspace_size(T, H, G))
    kvc = kv._c()
    name = "svt_sparse_mla_prefill_grouped_union_tile" if union_tile else "svt_sparse_mla_prefill_grouped"
    _check(getattr(lib(), name)(_ptr(q), T, H, int(G), ctypes.byref(kvc), _ptr(_i32(enc, "enc")),
                                _ptr(_i32(lens, "lens")), int(K), float(softmax_scale), _ptr(out), _ptr(lse), ws.ptr,
                                ws.nbytes, _stream()), name)
    return out, lse


def merge_splits(o_part, lse_part, *, out=None, lse=None, return_lse: bool = True):
    """svt_merge_splits: o_part [S, T, H, 512] fp32, lse_part [S, T, H] fp32 -> (out bf16, lse fp32)."""
    if o_part.dtype != torch.float32 or lse_part.dtype != torch.float32:
        raise TypeError("partials must be fp32")
    S, T, H, _ = o_part.shape
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=o_part.device)
    if lse is None and return_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=o_part.device)
    if not (o_part.is_contiguous() and lse_part.is_contiguous()):
        raise TypeError("partials must be contiguous")
    _check(lib().svt_merge_splits(_ptr(o_part), _ptr(lse_part), S, T, H, _ptr(out),
                                  _ptr(lse), _stream()), "svt_merge_splits")
    return out, lse


def topk_select(scores, K: int, *, lens=None, out=None):
    """svt_topk_select: scores [T, N] fp32 (rows may be strided) -> [T, K] int32 positions,
    ascending, -1 padded."""
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise TypeError("scores must be a [T, N] fp32 tensor with unit column stride")
    T, N = scores.shape
    if lens is not None:
        lens = _i32(lens, "lens")
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=scores.device)
    stride = scores.stride(0) if T > 1 else N  # a single row's stride is meaningless (can be 0)
    _check(lib().svt_topk_select(_ptr(scores), T, N, stride, _ptr(lens), int(K), _ptr(out), _stream()),
           "svt_topk_select")
    return out


def debug_pipeline_fault(fault: int = 0, wait_limit_ns: int = 0) -> None:
    """Failure-detection hook for tests (svt_debug_pipeline_fault): plant a withheld arrival
    in the attention kernels launched afterwards and/or shorten their wait limit; (0, 0)
    restores ordinary behaviour."""
    _check(lib().svt_debug_pipeline_fault(int(fault), int(wait_limit_ns)), "svt_debug_pipeline_fault")


def gather_probe(kv: KVCache, slots, mode: int = 0, *, out=None, ws: Optional[Workspace] = None):
    """Reads the cache rows of `slots` ([n] int32) the way the decode's gather does, with no
    arithmetic (svt_gather_probe); returns each row's XOR of 32-bit words as int32 [n]."""
    slots = _i32(slots, "slots")
    n = slots.numel()
    if out is None:
        out = torch.empty((n,), dtype=torch.int32, device=slots.device)
    ws = default_workspace() if ws is None else ws
    kvc = kv._c()
    _check(lib().svt_gather_probe(ctypes.byref(kvc), _ptr(slots), n, int(mode), _ptr(out), ws.ptr, ws.nbytes,
                                  _stream()), "svt_gather_probe")
    return out


def tensor_probe(k_rows, q, pt, reps: int = 1, grid: int = 1, *, ws: Optional[Workspace] = None):
    """Issues one half-tile's S^T and PV MMA group of the attention kernels `reps` times on
    `grid` CTAs (svt_tensor_probe). k_rows, q: [64, 576] bf16; pt: [64, 64] bf16 (P^T).
    Returns (S^T [64, 64] fp32, O^T [512, 64] fp32 = reps * V^T P^T, cycles [grid] int64)."""
    for name, t, shape in (("k_rows", k_rows, (64, 576)), ("q", q, (64, 576)), ("pt", pt, (64, 64))):
        if t.dtype != torch.bfloat16 or tuple(t.shape) != shape or not t.is_contiguous() or not t.is_cuda:
            raise SvtError(f"{name} must be a contiguous CUDA bf16 tensor of shape {shape}")
    dev = k_rows.device
    s_out = torch.empty((64, 64), dtype=torch.float32, device=dev)
    o_out = torch.empty((512, 64), dtype=torch.float32, device=dev)
    cycles = torch.empty((int(grid),), dtype=torch.int64, device=dev)
    ws = default_workspace() if ws is None else ws
    _check(lib().svt_tensor_probe(_ptr(k_rows), _ptr(q), _ptr(pt), int(reps), int(grid), _ptr(s_out), _ptr(o_out),
                                  _ptr(cycles), ws.ptr, ws.nbytes, _stream()), "svt_tensor_probe")
    return s_out, o_out, cycles
