"""The C-ABI library builds, loads and exports every entry point include/svt.h declares, and
its host-side argument checks reject bad calls before anything reaches a GPU. No GPU is used:
every call below fails its checks before the library touches the device."""

import ctypes
import os
import re

import pytest

from sparse_mla_attention_top_gb300 import build as B
from sparse_mla_attention_top_gb300 import svt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "svt.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return svt.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SVT_API\s+[\w\s\*]+?\b(svt_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("svt_sparse_mla_decode", "svt_sparse_mla_prefill_grouped", "svt_build_group_union",
                     "svt_merge_splits", "svt_resolve_topk_slots"):
        assert required in names
    assert names == sorted(svt.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    nm_names = set()
    for name in declared_functions():
        assert hasattr(L, name), name
        nm_names.add(name)
    assert nm_names == set(svt.EXPORTED)


def _kv(dtype=0, pages=4, page_size=64, stride=0, data=0x10000):
    return svt._KV(data, pages, page_size, stride, dtype)


WS = ctypes.c_void_p(0x100000)  # a 256-aligned fake address; never dereferenced by failing calls


def _err(L):
    return L.svt_last_error_string().decode()


def test_decode_rejects_bad_arguments(L):
    kv = _kv()
    q = ctypes.c_void_p(0x20000)
    out = ctypes.c_void_p(0x30000)
    topk = ctypes.c_void_p(0x40000)
    call = lambda **kw: L.svt_sparse_mla_decode(  # noqa: E731
        kw.get("q", q), kw.get("T", 2), kw.get("H", 64), ctypes.byref(kw.get("kv", kv)), None, 0, 0, None, None,
        kw.get("topk", topk), kw.get("K", 128), None, ctypes.c_float(kw.get("scale", 0.04)), out, None,
        kw.get("splits", 1), kw.get("ws", WS), kw.get("ws_bytes", 1 << 30), None)
    assert call(H=129) == svt.SVT_ERR_UNSUPPORTED and "128" in _err(L)
    assert call(H=0) == svt.SVT_ERR_INVALID_ARG
    assert call(T=-1) == svt.SVT_ERR_INVALID_ARG
    assert call(splits=-2) == svt.SVT_ERR_INVALID_ARG
    assert call(scale=float("nan")) == svt.SVT_ERR_INVALID_ARG
    assert call(kv=_kv(dtype=7)) == svt.SVT_ERR_UNSUPPORTED
    assert call(kv=_kv(stride=1160)) == svt.SVT_ERR_INVALID_ARG  # not a multiple of 16
    assert call(kv=_kv(stride=1024)) == svt.SVT_ERR_INVALID_ARG  # shorter than a bf16 row
    assert call(kv=_kv(data=0x10008)) == svt.SVT_ERR_INVALID_ARG  # misaligned cache
    assert call(kv=_kv(pages=1 << 26, page_size=64)) == svt.SVT_ERR_UNSUPPORTED  # >= 2^31 rows
    assert call(ws=ctypes.c_void_p(0x100010)) == svt.SVT_ERR_INVALID_ARG  # misaligned workspace
    assert call(ws_bytes=16) == svt.SVT_ERR_WORKSPACE
    assert call(q=ctypes.c_void_p(0x20008)) == svt.SVT_ERR_INVALID_ARG
    assert call(topk=None) == svt.SVT_ERR_INVALID_ARG


def test_decode_with_block_table_needs_its_shape(L):
    kv = _kv()
    st = L.svt_sparse_mla_decode(ctypes.c_void_p(0x20000), 1, 8, ctypes.byref(kv), ctypes.c_void_p(0x50000), 0, 4,
                                 None, None, ctypes.c_void_p(0x40000), 64, None, ctypes.c_float(0.1),
                                 ctypes.c_void_p(0x30000), None, 1, WS, 1 << 20, None)
    assert st == svt.SVT_ERR_INVALID_ARG and "num_reqs" in _err(L)


def test_prefill_rejects_unsupported_shapes(L):
    kv = _kv()
    call = lambda H, G, kvd=kv: L.svt_sparse_mla_prefill_grouped(  # noqa: E731
        ctypes.c_void_p(0x20000), 8, H, G, ctypes.byref(kvd), ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000),
        2048, ctypes.c_float(0.04), ctypes.c_void_p(0x30000), None, WS, 1 << 20, None)
    assert call(64, 4) == svt.SVT_ERR_UNSUPPORTED and "128" in _err(L)
    assert call(48, 3) == svt.SVT_ERR_UNSUPPORTED
    assert call(128, 1) == svt.SVT_ERR_UNSUPPORTED  # the pages keep H = 128 per rank on the old kernel
    # 2^24 - 1 rows or more: the 24-bit slot field cannot address them
    assert call(64, 2, _kv(pages=(1 << 24) // 64, page_size=64)) == svt.SVT_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["svt_sparse_mla_prefill_grouped", "svt_sparse_mla_prefill_grouped_union_tile"])
def test_both_prefill_entry_points_check_arguments_before_enqueueing(L, entry):
    # The same host checks run for the row-set and the union-tile kernel; a failed one returns
    # before anything is enqueued (no device here: any launch would fail differently).
    kv = _kv()
    fn = getattr(L, entry)
    call = lambda H=64, G=2, kvd=kv, ws_bytes=1 << 20, q=0x20000, scale=0.04: fn(  # noqa: E731
        ctypes.c_void_p(q) if q else None, 8, H, G, ctypes.byref(kvd), ctypes.c_void_p(0x40000),
        ctypes.c_void_p(0x50000), 2048, ctypes.c_float(scale), ctypes.c_void_p(0x30000), None, WS, ws_bytes, None)
    assert call(H=64, G=4) == svt.SVT_ERR_UNSUPPORTED
    assert call(ws_bytes=8) == svt.SVT_ERR_WORKSPACE
    assert call(q=0) == svt.SVT_ERR_INVALID_ARG
    assert call(scale=float("inf")) == svt.SVT_ERR_INVALID_ARG


def test_union_tile_prefill_takes_a_bf16_cache(L):
    kv = _kv(dtype=svt.KV_FP8_E4M3)
    st = L.svt_sparse_mla_prefill_grouped_union_tile(
        ctypes.c_void_p(0x20000), 8, 64, 2, ctypes.byref(kv), ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000),
        2048, ctypes.c_float(0.04), ctypes.c_void_p(0x30000), None, WS, 1 << 20, None)
    assert st == svt.SVT_ERR_UNSUPPORTED and "bf16" in _err(L)


def test_union_rejects_unsupported_arguments(L):
    call = lambda T=8, K=16, G=2, ns=1000, ws_bytes=1 << 20: L.svt_build_group_union(  # noqa: E731
        ctypes.c_void_p(0x20000), None, T, K, G, ns, ctypes.c_void_p(0x30000), ctypes.c_void_p(0x40000), WS,
        ws_bytes, None)
    assert call(G=3) == svt.SVT_ERR_UNSUPPORTED
    assert call(G=8, K=8192) == svt.SVT_ERR_UNSUPPORTED  # G*K beyond the shared-memory sort
    assert call(ns=0xFFFFFF) == svt.SVT_ERR_UNSUPPORTED
    assert call(ns=0) == svt.SVT_ERR_INVALID_ARG
    assert call(K=0) == svt.SVT_ERR_INVALID_ARG
    assert call(ws_bytes=8) == svt.SVT_ERR_WORKSPACE


def test_resolve_and_merge_reject_bad_arguments(L):
    st = L.svt_resolve_topk_slots(ctypes.c_void_p(0x20000), 4, 8, None, None, None, 0, 0, None, 0, 10,
                                  ctypes.c_void_p(0x30000), WS, 1 << 20, None)
    assert st == svt.SVT_ERR_INVALID_ARG  # page_size 0
    st = L.svt_resolve_topk_slots(None, 4, 8, None, None, None, 0, 0, None, 1, 10, ctypes.c_void_p(0x30000), WS,
                                  1 << 20, None)
    assert st == svt.SVT_ERR_INVALID_ARG
    st = L.svt_merge_splits(ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000), 0, 4, 8, ctypes.c_void_p(0x40000),
                            None, None)
    assert st == svt.SVT_ERR_INVALID_ARG
    st = L.svt_merge_splits(ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000), 65, 4, 8, ctypes.c_void_p(0x40000),
                            None, None)
    assert st == svt.SVT_ERR_INVALID_ARG


def test_topk_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    assert L.svt_topk_select(P(0x20000), 4, 100, 100, None, 0, P(0x30000), None) == svt.SVT_ERR_INVALID_ARG  # K 0
    assert L.svt_topk_select(P(0x20000), 4, 100, 99, None, 8, P(0x30000), None) == svt.SVT_ERR_INVALID_ARG  # stride
    assert L.svt_topk_select(None, 4, 100, 100, None, 8, P(0x30000), None) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_topk_select(P(0x20000), -1, 100, 100, None, 8, P(0x30000), None) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_topk_select(None, 0, 100, 100, None, 8, None, None) == svt.SVT_OK  # nothing to do


def test_workspace_sizes(L):
    assert L.svt_resolve_workspace_size() == 256
    assert L.svt_build_group_union_workspace_size(8192, 2048, 2) >= 256
    assert L.svt_sparse_mla_prefill_grouped_workspace_size(8192, 64, 2) >= 256
    # one CTA per query needs no partial buffers
    assert L.svt_sparse_mla_decode_workspace_size(64, 64, 2048, 1) == 256
    # lists split 3 ways are merged by a second kernel and need room for the partials: 2
    # slots per CTA of 64 rows x 512 fp16 + 64 fp32 lse
    n_cta = 64 * 3
    need = L.svt_sparse_mla_decode_workspace_size(64, 64, 2048, 3)
    assert need >= 256 + 2 * n_cta * 64 * (512 * 2 + 4)
    # 2, 4 or 8 slices per list merge inside a thread-block cluster: nothing beyond the header
    for s in (2, 4, 8):
        assert L.svt_sparse_mla_decode_workspace_size(64, 64, 2048, s) == 256


def test_product_path_has_no_oracle_or_fallback():
    # The library package never imports the oracle, and the binding has no CPU path.
    pkg = os.path.join(ROOT, "sparse_mla_attention_top_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn


def test_debug_pipeline_fault_checks_its_arguments(L):
    assert L.svt_debug_pipeline_fault(7, 0) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_debug_pipeline_fault(0, -1) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_debug_pipeline_fault(1, 1000) == svt.SVT_OK
    assert L.svt_debug_pipeline_fault(0, 0) == svt.SVT_OK  # back to ordinary behaviour


def test_tensor_probe_checks_its_arguments(L):
    P = ctypes.c_void_p
    a, b, c, s, o, cyc = (P(0x20000 + 0x10000 * i) for i in range(6))
    assert L.svt_tensor_probe(a, b, c, 0, 1, s, o, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG  # reps 0
    assert L.svt_tensor_probe(a, b, c, 1, 0, s, o, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG  # grid 0
    assert L.svt_tensor_probe(a, b, c, 1, 1025, s, o, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_tensor_probe(a, b, c, 100001, 1, s, o, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_tensor_probe(None, b, c, 1, 1, s, o, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_tensor_probe(a, b, c, 1, 1, s, None, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG
    assert L.svt_tensor_probe(P(0x20008), b, c, 1, 1, s, o, cyc, WS, 256, None) == svt.SVT_ERR_INVALID_ARG
    assert "aligned" in _err(L)
    assert L.svt_tensor_probe(a, b, c, 1, 1, s, o, cyc, WS, 16, None) != svt.SVT_OK  # workspace too small
