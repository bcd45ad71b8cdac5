"""The five benchmark workloads at full size, in the launch configuration bench.py times
(automatic split for decode), checked against the oracle: integer outputs (slots, unions)
in full and bit-exact; attention outputs of every query of the decode workloads and of a
stratified sample of more than 256 prefill queries (every member of groups spread over the
run and of the groups where the lists change shape), every head of each, within the
tolerances. Workloads: tiny decode (8 heads, 64 of 256); bf16 decode batch (64 x 64
heads, top-k 2048, contexts 8K-32K); e4m3 decode batch (128 x 64 heads, contexts 4K-46K);
grouped prefill (8192 new tokens, 64 heads, groups of 2); mixed step (16 heads, groups of 8,
8192 new on 24K cached, 128 decodes at 16K-46K, top-k = all dense check at 4K)."""

import numpy as np
import pytest

import oracle
from sparse_mla_attention_top_gb300 import workloads as W
from tests._dev import BF16_OUT_TOL, compare, kv_of, out_tol, to_dev

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


def run_decode(S, w, dev, ws):
    out, lse = S.sparse_mla_decode(to_dev(w.q_bits, dev), kv_of(w, dev), to_dev(w.topk, dev), w.scale,
                                   block_table=to_dev(w.block_table, dev), seq_lens=to_dev(w.seq_lens, dev),
                                   req_of_token=to_dev(w.req_of_token, dev), ws=ws)
    torch.cuda.synchronize()
    return out, lse


def check_decode_sampled(S, w, dev, ids):
    ws = S.Workspace(dev)
    out, lse = run_decode(S, w, dev, ws)
    assert ws.read_status() == 0
    ref, ref_lse, err = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                                      block_table=w.block_table, seq_lens=w.seq_lens, req_of_token=w.req_of_token,
                                      query_ids=ids)
    assert err == 0
    return compare(out, lse, ref, ref_lse, out_tol(w), rows=ids)


def test_tiny_decode_full(S, dev):
    w = W.tiny_decode()
    check_decode_sampled(S, w, dev, np.arange(w.T))


def test_decode_bf16_batch_every_query(S, dev):
    w = W.decode_bf16_batch()
    check_decode_sampled(S, w, dev, np.arange(w.T))


def test_decode_fp8_batch_every_query(S, dev):
    w = W.decode_fp8_batch()
    check_decode_sampled(S, w, dev, np.arange(w.T))


def run_prefill_and_check(S, w, dev, ids, union_tile=False):
    ws = S.Workspace(dev)
    slots = S.resolve_topk_slots(to_dev(w.topk, dev), block_table=to_dev(w.block_table, dev),
                                 seq_lens=to_dev(w.seq_lens, dev), req_of_token=to_dev(w.req_of_token, dev),
                                 page_size=w.page_size, num_pages=w.num_pages, ws=ws)
    enc, lens = S.build_group_union(slots, w.G, w.num_slots, ws=ws)
    out, lse = S.sparse_mla_prefill_grouped(to_dev(w.q_bits, dev), w.G, kv_of(w, dev), enc, lens, w.K, w.scale, ws=ws,
                                            union_tile=union_tile)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    ref_slots, err = oracle.resolve(w.topk, req_of_token=w.req_of_token, block_table=w.block_table,
                                    seq_lens=w.seq_lens, page_size=w.page_size, num_pages=w.num_pages)
    assert err == 0
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    ref_enc, ref_lens, err = oracle.group_union(ref_slots.astype(np.int32), w.G, w.num_slots)
    assert err == 0
    assert np.array_equal(lens.cpu().numpy(), ref_lens)
    assert np.array_equal(enc.cpu().numpy(), ref_enc)
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, w.G, w.kv, w.kv_dtype, w.num_slots, ref_enc, ref_lens, w.K,
                                               w.scale, query_ids=ids)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL, rows=ids)
    live = np.count_nonzero(w.topk >= 0, axis=1)
    return float(ref_lens.mean() / live.mean())


def stratified_groups(w, n_spread: int) -> np.ndarray:
    """Every member of n_spread groups spread evenly over the run, plus every group whose
    members' lists change from the whole causal prefix to the 70 % neighbour lists (the
    queries whose prefix first exceeds K) and the first and last groups."""
    groups = (w.T + w.G - 1) // w.G
    gs = set(np.linspace(0, groups - 1, n_spread).round().astype(int).tolist())
    n_cached = int(w.seq_lens[0]) - w.T
    first_full = max(0, w.K - n_cached - 1)  # first query with at least K candidates
    for q in (first_full - 1, first_full, first_full + 1):
        if 0 <= q < w.T:
            gs.add(q // w.G)
    gs.update({0, groups - 1})
    ids = [g * w.G + m for g in sorted(gs) for m in range(w.G) if g * w.G + m < w.T]
    return np.array(ids, np.int64)


@pytest.mark.parametrize("union_tile", [False, True], ids=["rowsets", "union_tile"])
def test_grouped_prefill_stratified(S, dev, union_tile):
    # both members of more than 128 groups (over 256 queries), every head of each; both kernels
    w = W.grouped_prefill()
    ids = stratified_groups(w, 130)
    assert len(ids) >= 256
    union_lists = run_prefill_and_check(S, w, dev, ids, union_tile)
    assert 1.0 < union_lists < 2.0


def test_mixed_prefill_stratified(S, dev):
    # all 8 members of 40 groups (320 queries)
    w = W.mixed_prefill()
    ids = stratified_groups(w, 40)
    assert len(ids) >= 256
    union_lists = run_prefill_and_check(S, w, dev, ids)
    assert 1.0 < union_lists < 8.0


def test_mixed_decode_every_query(S, dev):
    w = W.mixed_decode()
    check_decode_sampled(S, w, dev, np.arange(w.T))


def test_dense_check_topk_all_equals_dense_paged(S, dev):
    w = W.dense_check()
    ws = S.Workspace(dev)
    out, lse = run_decode(S, w, dev, ws)
    ref, ref_lse = oracle.dense_paged(w.q_bits[0], w.kv, w.kv_dtype, w.block_table[0], int(w.seq_lens[0]),
                                      w.page_size, w.scale)
    compare(out, lse, ref[None], ref_lse[None], BF16_OUT_TOL)
