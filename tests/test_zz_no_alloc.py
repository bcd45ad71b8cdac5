"""The allocation-free decode entry point, for callers that cannot call cudaMalloc (a plugin
inside a host application that owns all device memory, or code that must never trigger the
device-wide synchronisation a cudaMalloc can cause). It keeps its scratch in an array inside
the library instead of a caller workspace; its results must match the ordinary decode's.

This file is named to be collected last, so that a run which stops at the first failure has
already run every other test."""

import ctypes

import numpy as np
import pytest

from sparse_mla_attention_top_gb300 import workloads as W
from tests._dev import BF16_OUT_TOL, LSE_TOL, kv_of, to_dev

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
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(S, w, t, splits, out, lse, status):
    L = S.svt.lib()
    return L.svt_sparse_mla_decode_noalloc(
        _ptr(t["q"]), w.T, w.H, ctypes.byref(t["kvc"]), _ptr(t["bt"]), w.block_table.shape[0],
        w.block_table.shape[1], None, _ptr(t["seq"]), _ptr(t["topk"]), w.K, None, ctypes.c_float(w.scale), _ptr(out),
        _ptr(lse), splits, _ptr(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("splits", [2, 1])
def test_noalloc_decode_matches_the_workspace_decode_on_two_calls(S, splits):
    dev = torch.device("cuda", 0)
    w = W.make_decode(90, T=8, H=64, K=700, ctx_lo=800, ctx_hi=4000, page_size=64)
    t = _args(S, w, dev)
    ref_out, ref_lse = S.sparse_mla_decode(t["q"], t["kv"], t["topk"], w.scale, block_table=t["bt"],
                                           seq_lens=t["seq"], num_splits=splits, ws=S.Workspace(dev))
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for _ in range(2):  # the array keeps the last call's bytes; the second call must not see them
        out = torch.full((w.T, w.H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device=dev)
        st = _noalloc(S, w, t, splits, out, lse, status)
        assert st == S.svt.SVT_OK, S.svt.lib().svt_last_error_string()
        torch.cuda.synchronize()
        assert float((out.float() - ref_out.float()).abs().max()) <= BF16_OUT_TOL
        assert float((lse - ref_lse).abs().max()) <= LSE_TOL
        assert int(status.item()) == 0


def test_noalloc_rejects_a_decode_beyond_its_scratch(S):
    dev = torch.device("cuda", 0)
    w = W.make_decode(91, T=64, H=64, K=300, ctx_lo=400, ctx_hi=900, page_size=64)
    t = _args(S, w, dev)
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    # 64 queries cut into 3 slices: 192 CTAs with partial results, more than 8 MiB of scratch
    st = _noalloc(S, w, t, 3, out, lse, status)
    assert st == S.svt.SVT_ERR_WORKSPACE
    assert b"8388608" in S.svt.lib().svt_last_error_string()
