"""Parity of the top-k selection kernel with the CPU oracle: positions must match exactly
(the selection rule makes the kept set unique: ties go to the lower position)."""

import numpy as np
import pytest

import oracle
from sparse_mla_attention_top_gb300 import workloads as W
from tests import _golden
from tests._dev import BF16_OUT_TOL, compare, kv_of, to_dev

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


@pytest.fixture(scope="module")
def dev(S):
    return torch.device("cuda", 0)


def gpu_topk(S, scores, K, dev, lens=None):
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).to(dev)
    ln = None if lens is None else torch.from_numpy(np.ascontiguousarray(lens, np.int32)).to(dev)
    out = S.topk_select(s, K, lens=ln)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("case", _golden.topk_cases(), ids=lambda c: c["name"])
def test_topk_hand_worked_cases(S, dev, case):
    lens = None if case["len"] is None else np.array([case["len"]], np.int32)
    got = gpu_topk(S, case["scores"][None, :], case["K"], dev, lens)[0]
    assert np.array_equal(got, case["expect"]), (got, case["expect"])


def test_topk_tie_heavy_rows_match_oracle(S, dev):
    rng = np.random.default_rng(21)
    pool = np.array([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan, 1e-30, -1e30], np.float32)
    for N, K in [(1, 1), (7, 3), (130, 64), (1025, 1024), (3000, 2048), (5000, 17)]:
        T = 9
        scores = rng.choice(pool, size=(T, N)).astype(np.float32)
        lens = np.concatenate([[0, 1, N, K, K + 1, max(0, K - 1)], rng.integers(0, N + 1, size=T - 6)]).clip(0, N)
        lens = lens.astype(np.int32)
        ref = oracle.topk_select(scores, K, lens=lens)
        got = gpu_topk(S, scores, K, dev, lens)
        assert np.array_equal(got, ref), (N, K)


def test_topk_continuous_scores_span_chunks(S, dev):
    rng = np.random.default_rng(22)
    for N, K in [(2047, 2048), (2049, 2048), (4096 + 37, 2048), (20000, 512)]:
        scores = rng.standard_normal((5, N)).astype(np.float32)
        ref = oracle.topk_select(scores, K)
        assert np.array_equal(gpu_topk(S, scores, K, dev), ref), (N, K)


def test_topk_long_rows_and_strided_rows(S, dev):
    rng = np.random.default_rng(23)
    # rows whose half is longer than the shared-memory key buffer are read from global memory
    N, K = 100000, 2048
    scores = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((3, N), dtype=np.float32)))
    lens = np.array([N, 90000, 40000], np.int32)
    assert np.array_equal(gpu_topk(S, scores, K, dev, lens), oracle.topk_select(scores, K, lens=lens))
    # a [T, N] view of a wider buffer
    wide = torch.from_numpy(rng.standard_normal((4, 900)).astype(np.float32)).to(dev)
    view = wide[:, :700]
    got = S.topk_select(view, 100).cpu().numpy()
    assert np.array_equal(got, oracle.topk_select(view.cpu().numpy(), 100))


def test_topk_many_rows_one_cta_each(S, dev):
    # more rows than half the SMs: each row gets one CTA (smaller batches split a row between
    # a pair of CTAs); tie-heavy rows, then rows longer than the shared-memory key buffer
    rng = np.random.default_rng(26)
    pool = np.array([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan, 1e-30, -1e30], np.float32)
    T, N, K = 100, 3000, 1000
    scores = rng.choice(pool, size=(T, N)).astype(np.float32)
    lens = rng.integers(0, N + 1, size=T).astype(np.int32)
    assert np.array_equal(gpu_topk(S, scores, K, dev, lens), oracle.topk_select(scores, K, lens=lens))
    T, N, K = 100, 50000, 2048
    scores = rng.standard_normal((T, N)).astype(np.float32)
    lens = rng.integers(K, N + 1, size=T).astype(np.int32)
    assert np.array_equal(gpu_topk(S, scores, K, dev, lens), oracle.topk_select(scores, K, lens=lens))


def test_topk_full_size_batch(S, dev):
    w = W.topk_batch()
    got = gpu_topk(S, w.scores, w.K, dev, w.lens)
    assert np.array_equal(got, oracle.topk_select(w.scores, w.K, lens=w.lens))


def test_topk_feeds_decode(S, dev):
    # scores -> top-k positions -> sparse decode, against the oracle's own chain
    w = W.make_decode(24, T=5, H=64, K=256, ctx_lo=300, ctx_hi=3000, page_size=16)
    rng = np.random.default_rng(25)
    N = int(w.seq_lens.max())
    scores = rng.standard_normal((w.T, N)).astype(np.float32)
    lens = w.seq_lens[w.req_of_token]
    topk_dev = S.topk_select(torch.from_numpy(scores).to(dev), w.K, lens=torch.from_numpy(lens).to(dev))
    topk_ref = oracle.topk_select(scores, w.K, lens=lens)
    assert np.array_equal(topk_dev.cpu().numpy(), topk_ref)
    out, lse = S.sparse_mla_decode(to_dev(w.q_bits, dev), kv_of(w, dev), topk_dev, w.scale,
                                   block_table=to_dev(w.block_table, dev), seq_lens=to_dev(w.seq_lens, dev),
                                   req_of_token=to_dev(w.req_of_token, dev))
    ref, ref_lse, err = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, topk_ref, w.scale,
                                      block_table=w.block_table, seq_lens=w.seq_lens, req_of_token=w.req_of_token)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
