"""The allocation-free decode entry point, for callers that cannot call cudaMalloc (a plugin
inside a host application that owns all device memory, or code that must never trigger the
device-wide synchronisation a cudaMalloc can cause). It keeps its scratch in an array inside
the library instead of a caller workspace; its results must match the oracle and the
ordinary decode's, call after call, although every call reuses the same array.

This file is named to be collected last, so that a run which stops at the first failure has
already run every other test."""

import ctypes

import numpy as np
import pytest

import oracle
from sparse_mla_attention_top_gb300 import workloads as W
from tests._dev import BF16_OUT_TOL, LSE_TOL, compare, kv_of, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mla_attention_top_gb300 as S
    from sparse_mla_attention_top_gb300 import build

    build.build()
    return S


def _args(S, w, dev):
    t = dict(q=to_dev(w.q_bits, dev), topk=to_dev(w.topk, dev), bt=to_dev(w.block_table, dev),
             seq=to_dev(w.seq_lens, dev), kv=kv_of(w, dev))
    t["kvc"] = t["kv"]._c()
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(S, w, t, splits, out, lse, status, H=None):
    L = S.svt.lib()
    return L.svt_sparse_mla_decode_noalloc(
        _ptr(t["q"]), w.T, w.H if H is None else H, ctypes.byref(t["kvc"]), _ptr(t["bt"]), w.block_table.shape[0],
        w.block_table.shape[1], None, _ptr(t["seq"]), _ptr(t["topk"]), w.K, None, ctypes.c_float(w.scale), _ptr(out),
        _ptr(lse), splits, _ptr(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle(w):
    ref, ref_lse, err = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                                      block_table=w.block_table, seq_lens=w.seq_lens)
    assert err == 0
    return ref, ref_lse


# splits 3 cuts each query's 11 half-tiles between 3 CTAs that leave partial results in the
# array for the merge kernel (24 CTAs, about 3.2 MiB); 2 merges inside a cluster; 1 is one CTA
# per query; 0 is the automatic plan, on a batch (32 queries: clusters of 4) that fits the array
@pytest.mark.parametrize("splits", [3, 2, 1, 0])
def test_noalloc_decode_matches_oracle_and_workspace_decode_on_two_calls(S, splits):
    dev = torch.device("cuda", 0)
    T = 32 if splits == 0 else 8
    w = W.make_decode(90, T=T, H=64, K=700, ctx_lo=800, ctx_hi=4000, page_size=64)
    t = _args(S, w, dev)
    ref, ref_lse = _oracle(w)
    ws_out, ws_lse = S.sparse_mla_decode(t["q"], t["kv"], t["topk"], w.scale, block_table=t["bt"],
                                         seq_lens=t["seq"], num_splits=splits, ws=S.Workspace(dev))
    # an earlier call on other inputs leaves its partial results and status in the array
    w_other = W.make_decode(93, T=T, H=64, K=700, ctx_lo=800, ctx_hi=4000, page_size=64)
    t_other = _args(S, w_other, dev)
    junk_out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    junk_lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    assert _noalloc(S, w_other, t_other, splits, junk_out, junk_lse, None) == S.svt.SVT_OK
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for _ in range(2):  # the array keeps the last call's bytes; the next call must not see them
        out = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device=dev)
        st = _noalloc(S, w, t, splits, out, lse, status)
        assert st == S.svt.SVT_OK, S.svt.lib().svt_last_error_string()
        torch.cuda.synchronize()
        compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
        assert float((out.float() - ws_out.float()).abs().max()) <= BF16_OUT_TOL
        assert float((lse - ws_lse).abs().max()) <= LSE_TOL
        assert int(status.item()) == 0


def test_noalloc_reports_range_errors_of_its_own_call_only(S):
    dev = torch.device("cuda", 0)
    w = W.make_decode(94, T=4, H=16, K=200, ctx_lo=300, ctx_hi=600, page_size=64)
    bad = w.topk.copy()
    bad[1, 5] = int(w.seq_lens[1]) + 3  # past its request: dead, and flagged
    t = _args(S, w, dev)
    t_bad = dict(t, topk=to_dev(bad, dev))
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    assert _noalloc(S, w, t_bad, 1, out, lse, status) == S.svt.SVT_OK
    torch.cuda.synchronize()
    assert int(status.item()) == S.svt.DEV_ERR_INDEX_RANGE
    assert _noalloc(S, w, t, 1, out, lse, status) == S.svt.SVT_OK  # the next call starts clean
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = _oracle(w)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)


def test_noalloc_rejects_a_decode_beyond_its_scratch_and_enqueues_nothing(S):
    dev = torch.device("cuda", 0)
    w = W.make_decode(91, T=64, H=64, K=300, ctx_lo=400, ctx_hi=900, page_size=64)
    t = _args(S, w, dev)
    out = torch.full((w.T, w.H, 512), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.T, w.H), 7.0, dtype=torch.float32, device=dev)
    status = torch.full((1,), 12345, dtype=torch.int32, device=dev)
    # 64 queries cut into 3 slices: 192 CTAs with partial results, more than 8 MiB of scratch
    st = _noalloc(S, w, t, 3, out, lse, status)
    assert st == S.svt.SVT_ERR_WORKSPACE
    assert b"8388608" in S.svt.lib().svt_last_error_string()
    # a bad argument is refused the same way, before anything reaches the stream
    assert _noalloc(S, w, t, 1, out, lse, status, H=0) == S.svt.SVT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == 12345
    assert bool((out.float() == 7.0).all()) and bool((lse == 7.0).all())
