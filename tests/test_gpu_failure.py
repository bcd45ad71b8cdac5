"""Failure detection on the GPU without a GPU fault, and the e4m3 path's range check.

A pipeline wait that cannot complete must give up after its limit, set the timeout bit in
the status word and let the kernel run to its end, so that the call returns and the context
stays usable; the next ordinary call on the same stream must then be correct ("The Assertion
That Changed Everything": report a device-side failure instead of asserting). The test hook
withholds the arrival that announces the first KV tile (nothing else ever completes that
wait) and shortens the limit to 1 ms.

The e4m3 path contracts in f16: block scales up to 65504 / 448 and q / rope magnitudes below
65536 are exact to the oracle's tolerances at any scale; beyond that the range bit is set."""

import numpy as np
import pytest

import oracle
from sparse_mla_attention_top_gb300 import workloads as W
from tests._dev import BF16_OUT_TOL, FP8_OUT_TOL, LSE_TOL, compare, kv_of, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

WAIT_LIMIT_NS = 1_000_000  # 1 ms


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mla_attention_top_gb300 as S
    from sparse_mla_attention_top_gb300 import build

    build.build()
    return S


@pytest.fixture(scope="module")
def dev(S):
    return torch.device("cuda", 0)


def gpu_decode(S, w, dev, ws, num_splits=0):
    return S.sparse_mla_decode(to_dev(w.q_bits, dev), kv_of(w, dev), to_dev(w.topk, dev), w.scale,
                               block_table=to_dev(w.block_table, dev), seq_lens=to_dev(w.seq_lens, dev),
                               req_of_token=to_dev(w.req_of_token, dev), num_splits=num_splits, ws=ws)


def oracle_decode(w):
    ref, ref_lse, err = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                                      block_table=w.block_table, seq_lens=w.seq_lens, req_of_token=w.req_of_token)
    assert err == 0
    return ref, ref_lse


def gpu_prefill(S, w, dev, ws, union_tile=False):
    slots = S.resolve_topk_slots(to_dev(w.topk, dev), block_table=to_dev(w.block_table, dev),
                                 seq_lens=to_dev(w.seq_lens, dev), req_of_token=to_dev(w.req_of_token, dev),
                                 page_size=w.page_size, num_pages=w.num_pages, ws=ws)
    enc, lens = S.build_group_union(slots, w.G, w.num_slots, ws=ws)
    out, lse = S.sparse_mla_prefill_grouped(to_dev(w.q_bits, dev), w.G, kv_of(w, dev), enc, lens, w.K, w.scale, ws=ws,
                                            union_tile=union_tile)
    return enc, lens, out, lse


class planted_fault:
    def __init__(self, S):
        self.S = S

    def __enter__(self):
        self.S.svt.debug_pipeline_fault(1, WAIT_LIMIT_NS)

    def __exit__(self, *exc):
        self.S.svt.debug_pipeline_fault(0, 0)


# ------------------------------------------------------------------ a wait that runs out

# 1: one CTA per query; 2: slices merged in a thread-block cluster; 3: slices merged by the
# second kernel (partial results in the workspace)
@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3])
@pytest.mark.parametrize("splits", [1, 2, 3])
def test_decode_wait_that_runs_out_is_reported_and_the_next_call_is_correct(S, dev, splits, kv_dtype):
    w = W.make_decode(150 + splits, T=3, H=64, K=400, ctx_lo=500, ctx_hi=2000, page_size=64, kv_dtype=kv_dtype)
    ws = S.Workspace(dev)
    with planted_fault(S):
        gpu_decode(S, w, dev, ws, num_splits=splits)
        torch.cuda.synchronize()  # the call returns: every wait gave up after its limit
    status = ws.read_status()
    assert status & S.svt.DEV_ERR_TIMEOUT, status
    out, lse = gpu_decode(S, w, dev, ws, num_splits=splits)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_decode(w)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL if kv_dtype == W.KV_BF16 else FP8_OUT_TOL)
    assert ws.read_status() == 0


@pytest.mark.parametrize("union_tile", [False, True], ids=["rowsets", "union_tile"])
def test_prefill_wait_that_runs_out_is_reported_and_the_next_call_is_correct(S, dev, union_tile):
    # the union tile: every CTA of every two-CTA cluster times out on its first rows, the
    # peers then on the messages that never come; the cluster still ends and the next call
    # on the stream is correct
    w = W.make_prefill(155, n_new=12, n_cached=150, H=64, G=2, K=160, page_size=16)
    ws = S.Workspace(dev)
    with planted_fault(S):
        gpu_prefill(S, w, dev, ws, union_tile)
        torch.cuda.synchronize()
    status = ws.read_status()
    assert status & S.svt.DEV_ERR_TIMEOUT, status
    enc, lens, out, lse = gpu_prefill(S, w, dev, ws, union_tile)
    torch.cuda.synchronize()
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, w.G, w.kv, w.kv_dtype, w.num_slots, enc.cpu().numpy(),
                                               lens.cpu().numpy(), w.K, w.scale)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


def test_ordinary_calls_never_report_a_timeout(S, dev):
    # the hook is off: the default 2 s limit is never reached by a normal call
    w = W.make_decode(157, T=2, H=64, K=300, ctx_lo=400, ctx_hi=900, page_size=64)
    ws = S.Workspace(dev)
    for splits in (0, 1, 2, 3):
        gpu_decode(S, w, dev, ws, num_splits=splits)
    torch.cuda.synchronize()
    assert ws.read_status() == 0


# ------------------------------------------------------------------ e4m3 range

ROW = W.ROW


def with_block_scale(w, scale: float, q_factor: float):
    """The workload with every block scale set to `scale` and q multiplied by q_factor (so
    that the scores stay those of unit scales and only the magnitudes move)."""
    kv = w.kv.copy()
    kv[:, 512:528] = np.frombuffer(np.full(4, scale, np.float32).tobytes(), np.uint8)[None, :]
    q = W.bf16_bits_to_f32(w.q_bits) * np.float32(q_factor)
    w.kv = kv
    w.q_bits = W.f32_to_bf16_bits(q).reshape(w.q_bits.shape)
    return w


# out = scale x (the unit-scale output): the tolerance scales with the values
@pytest.mark.parametrize("scale", [100.0, 1e-3])
def test_decode_fp8_extreme_block_scales_match_oracle(S, dev, scale):
    w = with_block_scale(W.make_decode(160, T=3, H=64, K=300, ctx_lo=400, ctx_hi=1500, page_size=64,
                                       kv_dtype=W.KV_FP8_E4M3), scale, 1.0 / scale)
    ws = S.Workspace(dev)
    out, lse = gpu_decode(S, w, dev, ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    ref, ref_lse = oracle_decode(w)
    compare(out.float() / scale, lse, ref / scale, ref_lse, FP8_OUT_TOL, LSE_TOL)


def test_decode_fp8_block_scale_beyond_f16_sets_the_range_bit(S, dev):
    w = with_block_scale(W.make_decode(161, T=2, H=64, K=200, ctx_lo=300, ctx_hi=900, page_size=64,
                                       kv_dtype=W.KV_FP8_E4M3), 200.0, 1.0 / 200.0)
    ws = S.Workspace(dev)
    gpu_decode(S, w, dev, ws)
    torch.cuda.synchronize()
    assert ws.read_status() == S.svt.DEV_ERR_FP8_RANGE


def test_fp8_query_beyond_f16_sets_the_range_bit(S, dev):
    w = W.make_decode(162, T=2, H=64, K=200, ctx_lo=300, ctx_hi=900, page_size=64, kv_dtype=W.KV_FP8_E4M3)
    q = W.bf16_bits_to_f32(w.q_bits).copy()
    q[1, 7, 100] = 70000.0
    w.q_bits = W.f32_to_bf16_bits(q).reshape(w.q_bits.shape)
    ws = S.Workspace(dev)
    gpu_decode(S, w, dev, ws)
    torch.cuda.synchronize()
    assert ws.read_status() == S.svt.DEV_ERR_FP8_RANGE
    # the same query on a bf16 cache is in range: no bit
    wb = W.make_decode(162, T=2, H=64, K=200, ctx_lo=300, ctx_hi=900, page_size=64)
    wb.q_bits = w.q_bits
    gpu_decode(S, wb, dev, ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0


def test_prefill_fp8_block_scale_beyond_f16_sets_the_range_bit(S, dev):
    w = W.make_prefill(163, n_new=9, n_cached=100, H=16, G=8, K=90, page_size=16, kv_dtype=W.KV_FP8_E4M3)
    w = with_block_scale(w, 150.0, 1.0 / 150.0)  # 448 x 150 = 67200 > 65504
    ws = S.Workspace(dev)
    gpu_prefill(S, w, dev, ws)
    torch.cuda.synchronize()
    assert ws.read_status() == S.svt.DEV_ERR_FP8_RANGE
