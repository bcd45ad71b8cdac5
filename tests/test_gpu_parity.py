"""Parity of the CUDA path with the CPU oracle on small seeded inputs that still span
several tiles and a ragged tail. Integer outputs (slots, unions) must be bit-exact; float
outputs must stay within the stated tolerances (out 2e-2 bf16 / 5e-2 fp8, lse 1e-3)."""

import numpy as np
import pytest

import oracle
from sparse_mla_attention_top_gb300 import workloads as W
from tests import _golden
from tests._dev import BF16_OUT_TOL, FP8_OUT_TOL, LSE_TOL, compare, kv_of, out_tol, to_dev

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


@pytest.fixture()
def ws(S, dev):
    return S.Workspace(dev)


def gpu_decode(S, w, dev, ws, topk=None, topk_len=None, num_splits=0, use_table=True):
    topk = w.topk if topk is None else topk
    return S.sparse_mla_decode(to_dev(w.q_bits, dev), kv_of(w, dev), to_dev(topk, dev), w.scale,
                               block_table=to_dev(w.block_table, dev) if use_table else None,
                               seq_lens=to_dev(w.seq_lens, dev) if use_table else None,
                               req_of_token=to_dev(w.req_of_token, dev) if use_table else None,
                               topk_len=to_dev(topk_len, dev), num_splits=num_splits, ws=ws)


def oracle_decode(w, topk=None, topk_len=None, query_ids=None):
    topk = w.topk if topk is None else topk
    return oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, topk, w.scale,
                         block_table=w.block_table, seq_lens=w.seq_lens, req_of_token=w.req_of_token,
                         topk_len=topk_len, query_ids=query_ids)


# ------------------------------------------------------------------------ slot resolution

def test_resolve_hand_worked_example(S, dev, ws):
    c = _golden.resolve_case()
    slots = S.resolve_topk_slots(to_dev(c["topk"], dev), block_table=to_dev(c["block_table"], dev),
                                 seq_lens=to_dev(c["seq_lens"], dev), req_of_token=to_dev(c["req_of_token"], dev),
                                 topk_len=to_dev(c["topk_len"], dev), page_size=c["page_size"],
                                 num_pages=c["num_pages"], ws=ws)
    assert np.array_equal(slots.cpu().numpy(), c["slots"])
    assert ws.read_status() == S.svt.DEV_ERR_INDEX_RANGE


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_resolve_matches_oracle_bit_exact(S, dev, ws, page_size):
    w = W.make_decode(21, T=9, H=1, K=333, ctx_lo=100, ctx_hi=5000, page_size=page_size)
    topk = w.topk.copy()
    rng = np.random.default_rng(page_size)
    topk[rng.random(topk.shape) < 0.05] = -1
    topk[0, 5] = w.seq_lens[0] + 3  # past the request: range error
    topk_len = rng.integers(0, w.K + 1, size=w.T).astype(np.int32)
    slots = S.resolve_topk_slots(to_dev(topk, dev), block_table=to_dev(w.block_table, dev),
                                 seq_lens=to_dev(w.seq_lens, dev), topk_len=to_dev(topk_len, dev),
                                 page_size=w.page_size, num_pages=w.num_pages, ws=ws)
    ref, err = oracle.resolve(topk, topk_len, None, w.block_table, w.seq_lens, w.page_size, w.num_pages)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), ref)
    assert ws.read_status() == (S.svt.DEV_ERR_INDEX_RANGE if err & 1 else 0)


# ---------------------------------------------------------------------------------- union

def test_union_hand_worked_cases(S, dev, ws):
    for c in _golden.union_cases():
        slots = np.array(c["rows"], np.int32)
        ln = np.array(c["lens_rows"], np.int32)
        enc, lens = S.build_group_union(to_dev(slots, dev), c["G"], c["num_slots"], topk_len=to_dev(ln, dev), ws=ws)
        ref_enc, ref_lens, _ = oracle.group_union(slots, c["G"], c["num_slots"], topk_len=ln)
        assert np.array_equal(lens.cpu().numpy(), ref_lens), c["name"]
        assert np.array_equal(enc.cpu().numpy(), ref_enc), c["name"]
        for g, (n, pairs) in c["groups"].items():
            assert enc[g, :n].cpu().tolist() == [_golden.encode(m, s) for m, s in pairs]
    assert ws.read_status() == 0


@pytest.mark.parametrize("G,K,T", [(2, 64, 17), (4, 100, 22), (8, 33, 70), (2, 2048, 9), (8, 2048, 11)])
def test_union_matches_oracle_bit_exact(S, dev, ws, G, K, T):
    rng = np.random.default_rng(G * 1000 + K)
    num_slots = 5000
    slots = np.full((T, K), -1, np.int32)
    for t in range(T):
        n = int(rng.integers(0, K + 1))
        base = rng.choice(num_slots, size=n, replace=False).astype(np.int32)
        if t > 0 and n:  # neighbours overlap
            prev = slots[t - 1][slots[t - 1] >= 0]
            k = min(len(prev), n // 2)
            base[:k] = prev[:k]
            base = np.unique(base)
            rng.shuffle(base)
        slots[t, :len(base)] = base
        slots[t] = slots[t][rng.permutation(K)]
    ln = rng.integers(0, K + 1, size=T).astype(np.int32)
    enc, lens = S.build_group_union(to_dev(slots, dev), G, num_slots, topk_len=to_dev(ln, dev), ws=ws)
    ref_enc, ref_lens, err = oracle.group_union(slots, G, num_slots, topk_len=ln)
    assert err == 0
    assert np.array_equal(lens.cpu().numpy(), ref_lens)
    assert np.array_equal(enc.cpu().numpy(), ref_enc)


def test_union_out_of_range_slot_is_dropped_and_flagged(S, dev, ws):
    slots = np.array([[3, 900, 5], [5, -1, 7]], np.int32)
    enc, lens = S.build_group_union(to_dev(slots, dev), 2, 100, ws=ws)
    ref_enc, ref_lens, err = oracle.group_union(slots, 2, 100)
    assert err == 1 and np.array_equal(enc.cpu().numpy(), ref_enc) and lens.item() == 3
    assert ws.read_status() == S.svt.DEV_ERR_INDEX_RANGE


# --------------------------------------------------------------------------------- decode

def test_tiny_decode(S, dev, ws):
    w = W.tiny_decode()
    out, lse = gpu_decode(S, w, dev, ws)
    ref, ref_lse, err = oracle_decode(w)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


@pytest.mark.parametrize("num_splits", [0, 1, 2, 3])
def test_decode_ragged_tail_and_splits(S, dev, ws, num_splits):
    # K = 300: two full 128-row tiles and a tail of 44
    w = W.make_decode(31, T=7, H=64, K=300, ctx_lo=250, ctx_hi=4000, page_size=64)
    out, lse = gpu_decode(S, w, dev, ws, num_splits=num_splits)
    ref, ref_lse, err = oracle_decode(w)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


@pytest.mark.parametrize("H", [1, 8, 16, 33, 64, 100, 128])
def test_decode_head_counts(S, dev, ws, H):
    w = W.make_decode(40 + H, T=3, H=H, K=200, ctx_lo=300, ctx_hi=900, page_size=16)
    out, lse = gpu_decode(S, w, dev, ws)
    ref, ref_lse, _ = oracle_decode(w)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)


def test_decode_fp8_cache(S, dev, ws):
    w = W.make_decode(51, T=5, H=64, K=260, ctx_lo=300, ctx_hi=3000, page_size=64, kv_dtype=W.KV_FP8_E4M3)
    out, lse = gpu_decode(S, w, dev, ws)
    ref, ref_lse, err = oracle_decode(w)
    assert err == 0
    compare(out, lse, ref, ref_lse, FP8_OUT_TOL)
    assert ws.read_status() == 0


def test_decode_virtual_block_table_equals_paged(S, dev, ws):
    # slots passed directly (no table, page_size-1 view) give the same result as positions
    w = W.make_decode(52, T=4, H=32, K=190, ctx_lo=200, ctx_hi=2000, page_size=64)
    out, lse = gpu_decode(S, w, dev, ws)
    slots, _ = oracle.resolve(w.topk, block_table=w.block_table, seq_lens=w.seq_lens, page_size=w.page_size,
                              num_pages=w.num_pages)
    out2, lse2 = gpu_decode(S, w, dev, ws, topk=slots.astype(np.int32), use_table=False)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_decode_padding_and_live_counts(S, dev, ws):
    w = W.make_decode(53, T=4, H=16, K=256, ctx_lo=400, ctx_hi=900, page_size=8)
    rng = np.random.default_rng(1)
    padded = np.full((w.T, 400), -1, np.int32)
    for t in range(w.T):
        where = np.sort(rng.choice(400, w.K, replace=False))
        padded[t, where] = w.topk[t]
    out, lse = gpu_decode(S, w, dev, ws, topk=padded)
    ref, ref_lse, _ = oracle_decode(w)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    lens = np.array([0, 1, 129, 256], np.int32)
    out, lse = gpu_decode(S, w, dev, ws, topk_len=lens)
    ref, ref_lse, _ = oracle_decode(w, topk_len=lens)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))  # empty query


def test_decode_single_index_returns_v_row(S, dev, ws):
    w = W.make_decode(54, T=3, H=64, K=5, ctx_lo=100, ctx_hi=100, page_size=4)
    topk = np.full((3, 5), -1, np.int32)
    topk[:, 2] = [7, 50, 99]
    out, lse = gpu_decode(S, w, dev, ws, topk=topk)
    slots, _ = oracle.resolve(topk, block_table=w.block_table, seq_lens=w.seq_lens, page_size=w.page_size,
                              num_pages=w.num_pages)
    rows = oracle.fetch_rows(w.kv, w.kv_dtype, slots[:, 2])
    o = out.float().cpu().numpy()
    for t in range(3):  # exactly the bf16 V row (P = 1, l = 1)
        assert np.array_equal(o[t], np.broadcast_to(rows[t, :512], (64, 512)))
    ref, ref_lse, _ = oracle_decode(w, topk=topk)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_TOL


def test_decode_zero_query_gives_mean_and_log_count(S, dev, ws):
    w = W.make_decode(55, T=2, H=8, K=300, ctx_lo=1000, ctx_hi=1000, page_size=64)
    w.q_bits[:] = 0
    out, lse = gpu_decode(S, w, dev, ws)
    slots, _ = oracle.resolve(w.topk, block_table=w.block_table, seq_lens=w.seq_lens, page_size=w.page_size,
                              num_pages=w.num_pages)
    for t in range(2):
        mean = oracle.fetch_rows(w.kv, w.kv_dtype, slots[t])[:, :512].mean(axis=0)
        assert np.max(np.abs(out[t].float().cpu().numpy() - mean)) <= BF16_OUT_TOL
    assert np.allclose(lse.cpu().numpy(), np.log(300), atol=LSE_TOL)


def test_decode_order_invariance(S, dev, ws):
    w = W.make_decode(56, T=3, H=64, K=384, ctx_lo=500, ctx_hi=3000, page_size=64)
    out, lse = gpu_decode(S, w, dev, ws)
    perm = np.random.default_rng(2).permutation(w.K)
    out2, lse2 = gpu_decode(S, w, dev, ws, topk=np.ascontiguousarray(w.topk[:, perm]))
    assert float((out.float() - out2.float()).abs().max()) <= BF16_OUT_TOL
    assert float((lse - lse2).abs().max()) <= LSE_TOL


def test_decode_out_of_range_entries_are_dead_and_flagged(S, dev, ws):
    w = W.make_decode(57, T=2, H=16, K=130, ctx_lo=500, ctx_hi=600, page_size=64)
    bad = w.topk.copy()
    bad[1, 7] = 10 ** 6
    out, lse = gpu_decode(S, w, dev, ws, topk=bad)
    ref, ref_lse, err = oracle_decode(w, topk=bad)
    assert err == 1
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == S.svt.DEV_ERR_INDEX_RANGE


def test_decode_large_scores_rescale(S, dev, ws):
    # Scores that grow tile after tile force the reference maximum to move (rescale path).
    w = W.make_decode(58, T=2, H=64, K=512, ctx_lo=600, ctx_hi=600, page_size=64)
    scale = 0.5  # wide score spread
    out, lse = S.sparse_mla_decode(to_dev(w.q_bits, dev), kv_of(w, dev), to_dev(w.topk, dev), scale,
                                   block_table=to_dev(w.block_table, dev), seq_lens=to_dev(w.seq_lens, dev), ws=ws)
    ref, ref_lse, _ = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, scale,
                                    block_table=w.block_table, seq_lens=w.seq_lens)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)


# ------------------------------------------------------------------ cluster-merged slices

@pytest.mark.parametrize("splits", [2, 4, 8])
@pytest.mark.parametrize("H", [1, 33, 64, 100, 128])
def test_decode_cluster_slices_match_oracle(S, dev, ws, splits, H):
    # Each query's list cut into 2, 4 or 8 slices whose CTAs form a thread-block cluster and
    # merge in distributed shared memory. K = 700 leaves a ragged last half-tile; the live
    # counts leave whole slices with nothing (an empty query, a single entry, 65 entries).
    w = W.make_decode(90 + H, T=5, H=H, K=700, ctx_lo=400, ctx_hi=3000, page_size=64)
    lens = np.array([700, 0, 1, 65, 430], np.int32)
    out, lse = gpu_decode(S, w, dev, ws, topk_len=lens, num_splits=splits)
    ref, ref_lse, err = oracle_decode(w, topk_len=lens)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    assert ws.read_status() == 0


@pytest.mark.parametrize("T,K", [(32, 1024), (64, 512), (120, 256), (100, 512)])
def test_decode_automatic_plan_matches_oracle(S, dev, ws, T, K):
    # The automatic plan over batch sizes that take each of its branches on a 152-SM GPU:
    # 32 queries -> clusters of 4, 64 -> clusters of 2, 120 -> one CTA per query, 100 ->
    # stream-K with the merge kernel. Every query is checked.
    w = W.make_decode(130 + T, T=T, H=64, K=K, ctx_lo=K // 2, ctx_hi=3 * K, page_size=64)
    out, lse = gpu_decode(S, w, dev, ws)
    ref, ref_lse, err = oracle_decode(w)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


def test_decode_fp8_cache_cluster_slices(S, dev, ws):
    w = W.make_decode(97, T=6, H=64, K=520, ctx_lo=300, ctx_hi=5000, page_size=64, kv_dtype=W.KV_FP8_E4M3)
    ref, ref_lse, err = oracle_decode(w)
    assert err == 0
    for splits in (2, 4, 8):
        out, lse = gpu_decode(S, w, dev, ws, num_splits=splits)
        compare(out, lse, ref, ref_lse, FP8_OUT_TOL)
    assert ws.read_status() == 0


def test_decode_cluster_slices_equal_unsplit(S, dev, ws):
    # The same lists computed whole (one CTA per query) and in clustered slices agree within
    # rounding, and the slices' merged LSE is the whole list's.
    w = W.make_decode(98, T=4, H=64, K=1024, ctx_lo=2000, ctx_hi=6000, page_size=64)
    out1, lse1 = gpu_decode(S, w, dev, ws, num_splits=1)
    for splits in (2, 4, 8):
        out, lse = gpu_decode(S, w, dev, ws, num_splits=splits)
        assert float((out.float() - out1.float()).abs().max()) <= 1e-2
        assert float((lse - lse1).abs().max()) <= 1e-4


# ---------------------------------------------------------------------------------- merge

def test_merge_splits_matches_oracle(S, dev):
    rng = np.random.default_rng(3)
    Sn, T, H = 5, 3, 7
    o = rng.standard_normal((Sn, T, H, 512)).astype(np.float32)
    l = rng.standard_normal((Sn, T, H)).astype(np.float32) * 3
    l[1, 0, :] = -np.inf
    l[:, 2, 3] = -np.inf  # an all-empty row
    out, lse = S.merge_splits(to_dev(o, dev), to_dev(l, dev))
    ref, ref_lse = oracle.merge(o, l)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert torch.all(out[2, 3] == 0)


# -------------------------------------------------------------------------- grouped prefill

def gpu_prefill(S, w, dev, ws, union_tile=False):
    slots = S.resolve_topk_slots(to_dev(w.topk, dev), block_table=to_dev(w.block_table, dev),
                                 seq_lens=to_dev(w.seq_lens, dev), req_of_token=to_dev(w.req_of_token, dev),
                                 page_size=w.page_size, num_pages=w.num_pages, ws=ws)
    enc, lens = S.build_group_union(slots, w.G, w.num_slots, ws=ws)
    out, lse = S.sparse_mla_prefill_grouped(to_dev(w.q_bits, dev), w.G, kv_of(w, dev), enc, lens, w.K, w.scale, ws=ws,
                                            union_tile=union_tile)
    return slots, enc, lens, out, lse


# Both grouped-prefill kernels (bf16 cache): row-sets of 64 rows that walk their members'
# entries (svt_sparse_mla_prefill_grouped) and one union tile for all 128 rows on a pair of
# CTAs (svt_sparse_mla_prefill_grouped_union_tile).
TILES = pytest.mark.parametrize("union_tile", [False, True], ids=["rowsets", "union_tile"])


@TILES
@pytest.mark.parametrize("H,G,T", [(64, 2, 13), (32, 4, 22), (16, 8, 37)])
def test_prefill_matches_oracle(S, dev, ws, H, G, T, union_tile):
    w = W.make_prefill(60 + G, n_new=T, n_cached=150, H=H, G=G, K=160, page_size=16)
    slots, enc, lens, out, lse = gpu_prefill(S, w, dev, ws, union_tile)
    ref_slots, _ = oracle.resolve(w.topk, req_of_token=w.req_of_token, block_table=w.block_table,
                                  seq_lens=w.seq_lens, page_size=w.page_size, num_pages=w.num_pages)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    ref_enc, ref_lens, _ = oracle.group_union(ref_slots.astype(np.int32), G, w.num_slots)
    assert np.array_equal(enc.cpu().numpy(), ref_enc) and np.array_equal(lens.cpu().numpy(), ref_lens)
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, G, w.kv, w.kv_dtype, w.num_slots, ref_enc, ref_lens, w.K,
                                               w.scale)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


@TILES
@pytest.mark.parametrize("H,G", [(64, 2), (32, 4), (16, 8)])
def test_prefill_row_sets_keep_only_their_members_entries(S, dev, ws, H, G, union_tile):
    # Each 64-row half of a group walks only the union entries live for one of its members.
    # Odd tokens select nothing (a half may keep no entry at all), and tokens 4 apart share
    # their lists, so some entries are live for several members and others for one.
    w = W.make_prefill(110 + G, n_new=3 * G + 1, n_cached=700, H=H, G=G, K=200, page_size=16)
    topk = w.topk.copy()
    for t in range(w.T):
        if t % 2 == 1:
            topk[t] = -1
        elif t >= 4:
            topk[t] = topk[t - 4]
    slots = S.resolve_topk_slots(to_dev(topk, dev), block_table=to_dev(w.block_table, dev),
                                 seq_lens=to_dev(w.seq_lens, dev), req_of_token=to_dev(w.req_of_token, dev),
                                 page_size=w.page_size, num_pages=w.num_pages, ws=ws)
    enc, lens = S.build_group_union(slots, G, w.num_slots, ws=ws)
    out, lse = S.sparse_mla_prefill_grouped(to_dev(w.q_bits, dev), G, kv_of(w, dev), enc, lens, w.K, w.scale, ws=ws,
                                            union_tile=union_tile)
    ref_enc, ref_lens, _ = oracle.group_union(slots.cpu().numpy(), G, w.num_slots)
    assert np.array_equal(enc.cpu().numpy(), ref_enc)
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, G, w.kv, w.kv_dtype, w.num_slots, ref_enc, ref_lens, w.K,
                                               w.scale)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert torch.all(out[1::2] == 0) and torch.all(torch.isneginf(lse[1::2]))
    assert ws.read_status() == 0


@TILES
@pytest.mark.parametrize("H,G", [(64, 2), (16, 8)])
def test_prefill_rescales_and_empty_groups(S, dev, ws, H, G, union_tile):
    # A wide score spread (softmax scale 0.5) moves the reference maximum in the middle of the
    # lists (in the union tile, both the CTA that runs the softmax of a row and the one holding
    # the other half of its channels rescale their O); the second group's members all select
    # nothing (a group with no tile between groups with several), and the unions span several
    # tiles with a ragged last one.
    w = W.make_prefill(140 + G, n_new=3 * G, n_cached=700, H=H, G=G, K=300, page_size=16)
    topk = w.topk.copy()
    topk[G:2 * G] = -1
    scale = 0.5
    slots = S.resolve_topk_slots(to_dev(topk, dev), block_table=to_dev(w.block_table, dev),
                                 seq_lens=to_dev(w.seq_lens, dev), req_of_token=to_dev(w.req_of_token, dev),
                                 page_size=w.page_size, num_pages=w.num_pages, ws=ws)
    enc, lens = S.build_group_union(slots, G, w.num_slots, ws=ws)
    out, lse = S.sparse_mla_prefill_grouped(to_dev(w.q_bits, dev), G, kv_of(w, dev), enc, lens, w.K, scale, ws=ws,
                                            union_tile=union_tile)
    ref_enc, ref_lens, _ = oracle.group_union(slots.cpu().numpy(), G, w.num_slots)
    assert np.array_equal(enc.cpu().numpy(), ref_enc)
    assert ref_lens[1] == 0 and ref_lens[0] > 4 * 64 and ref_lens[0] % 64 != 0
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, G, w.kv, w.kv_dtype, w.num_slots, ref_enc, ref_lens, w.K,
                                               scale)
    assert err == 0
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert torch.all(out[G:2 * G] == 0) and torch.all(torch.isneginf(lse[G:2 * G]))
    assert ws.read_status() == 0


@pytest.mark.parametrize("H,G,T", [(64, 2, 37), (32, 4, 41), (16, 8, 45)])
def test_prefill_row_set_counts_bit_exact(S, dev, H, G, T):
    # The count kernel's per-half kept entries (left in the workspace after the header) equal
    # a plain recount from the oracle's union: entries with a membership bit of one of the
    # members whose rows the half holds.
    w = W.make_prefill(120 + G, n_new=T, n_cached=900, H=H, G=G, K=96, page_size=16)
    ws = S.Workspace(dev)
    slots, enc, lens, out, lse = gpu_prefill(S, w, dev, ws)
    torch.cuda.synchronize()
    ref_enc, ref_lens, _ = oracle.group_union(slots.cpu().numpy(), G, w.num_slots)
    groups = ref_lens.shape[0]
    got = ws.buf[256:256 + 8 * groups].cpu().view(torch.int32).numpy()
    want = []
    for g in range(groups):
        masks = (ref_enc[g, :ref_lens[g]].astype(np.int64) & 0xFFFFFFFF) >> 24
        for half in range(2):
            members = {(half * 64 + r) // H for r in range(64)}
            bits = sum(1 << m for m in members)
            want.append(int(np.count_nonzero(masks & bits)))
    assert np.array_equal(got, np.array(want, np.int32))
    assert ws.read_status() == 0


@TILES
def test_prefill_equals_per_query_decode_on_gpu(S, dev, ws, union_tile):
    w = W.make_prefill(70, n_new=9, n_cached=300, H=64, G=2, K=200, page_size=64)
    _, _, _, out, lse = gpu_prefill(S, w, dev, ws, union_tile)
    out_d, lse_d = gpu_decode(S, w, dev, ws)
    assert float((out.float() - out_d.float()).abs().max()) <= BF16_OUT_TOL
    assert float((lse - lse_d).abs().max()) <= LSE_TOL


@TILES
def test_prefill_membership_bit_negative_control(S, dev, ws, union_tile):
    # A flipped membership bit must change that member's rows: the parity check has teeth.
    w = W.make_prefill(71, n_new=4, n_cached=400, H=64, G=2, K=128, page_size=64)
    slots, enc, lens, out, lse = gpu_prefill(S, w, dev, ws, union_tile)
    e = enc.clone()
    row = e[0, : int(lens[0])]
    has1 = ((row.view(torch.int32) >> 24) & 2) != 0
    idx = int(torch.nonzero(~has1)[0])
    e[0, idx] = row[idx] | (2 << 24)
    out2, lse2 = S.sparse_mla_prefill_grouped(to_dev(w.q_bits, dev), w.G, kv_of(w, dev), e, lens, w.K, w.scale, ws=ws,
                                              union_tile=union_tile)
    assert float((lse2[1] - lse[1]).abs().max()) > LSE_TOL
    assert torch.equal(out2[0], out[0])


def test_workspace_reuse_across_shapes_and_repeats(S, dev):
    # One workspace serves calls of different shapes back to back (split and unsplit), so a
    # call never depends on bytes an earlier call left in it.
    ws = S.Workspace(dev)
    big = W.make_decode(80, T=5, H=64, K=700, ctx_lo=800, ctx_hi=3000, page_size=64)
    small = W.make_decode(81, T=4, H=16, K=256, ctx_lo=300, ctx_hi=900, page_size=16)
    ref_b, ref_lse_b, _ = oracle_decode(big)
    ref_s, ref_lse_s, _ = oracle_decode(small)
    for w, ref, ref_lse in [(big, ref_b, ref_lse_b), (small, ref_s, ref_lse_s), (big, ref_b, ref_lse_b),
                            (small, ref_s, ref_lse_s)]:
        for splits in (0, 2, 3):
            out, lse = gpu_decode(S, w, dev, ws, num_splits=splits)
            compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


# ------------------------------------------------------------- e4m3 grouped prefill

@pytest.mark.parametrize("H,G,T", [(64, 2, 11), (16, 8, 29)])
def test_prefill_fp8_cache_matches_oracle(S, dev, ws, H, G, T):
    w = W.make_prefill(100 + G, n_new=T, n_cached=200, H=H, G=G, K=150, page_size=16, kv_dtype=W.KV_FP8_E4M3)
    slots, enc, lens, out, lse = gpu_prefill(S, w, dev, ws)
    ref_enc, ref_lens, _ = oracle.group_union(slots.cpu().numpy(), G, w.num_slots)
    assert np.array_equal(enc.cpu().numpy(), ref_enc)
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, G, w.kv, w.kv_dtype, w.num_slots, ref_enc, ref_lens, w.K,
                                               w.scale)
    assert err == 0
    compare(out, lse, ref, ref_lse, FP8_OUT_TOL)
    assert ws.read_status() == 0


# ------------------------------------------------------------------ CUDA graph replay

def test_decode_and_prefill_replay_from_a_cuda_graph(S, dev):
    # The grids depend only on the arguments, so a captured step replays with new inputs.
    w = W.make_decode(110, T=6, H=64, K=400, ctx_lo=500, ctx_hi=3000, page_size=64)
    ws = S.Workspace(dev).ensure(1 << 24)
    q = to_dev(w.q_bits, dev)
    kv = kv_of(w, dev)
    topk = to_dev(w.topk, dev)
    bt, seq = to_dev(w.block_table, dev), to_dev(w.seq_lens, dev)
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    S.sparse_mla_decode(q, kv, topk, w.scale, block_table=bt, seq_lens=seq, out=out, lse=lse, ws=ws)  # warm
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            S.sparse_mla_decode(q, kv, topk, w.scale, block_table=bt, seq_lens=seq, out=out, lse=lse, ws=ws)
    w2 = W.make_decode(111, T=6, H=64, K=400, ctx_lo=500, ctx_hi=3000, page_size=64)
    q.copy_(to_dev(w2.q_bits, dev))  # new queries, same cache and lists
    g.replay()
    torch.cuda.synchronize()
    w2.kv, w2.block_table, w2.seq_lens, w2.topk, w2.num_pages = w.kv, w.block_table, w.seq_lens, w.topk, w.num_pages
    ref, ref_lse, _ = oracle_decode(w2)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    g.replay()
    torch.cuda.synchronize()
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert ws.read_status() == 0


# --------------------------------------------------------- zigzag-sharded prefill

def test_zigzag_sharded_prefill_reproduces_the_whole_step(S, dev, ws):
    from sparse_mla_attention_top_gb300.shard import zigzag_split

    w = W.make_prefill(120, n_new=37, n_cached=400, H=64, G=2, K=180, page_size=16)
    _, _, _, out_all, lse_all = gpu_prefill(S, w, dev, ws)
    out = torch.zeros_like(out_all)
    lse = torch.zeros_like(lse_all)
    for ids in zigzag_split(w.T, 4):  # each rank runs its own rows, no exchange
        idx = torch.from_numpy(ids).to(dev)
        qr = to_dev(w.q_bits, dev)[idx].contiguous()
        tk = to_dev(w.topk, dev)[idx].contiguous()
        slots = S.resolve_topk_slots(tk, block_table=to_dev(w.block_table, dev), seq_lens=to_dev(w.seq_lens, dev),
                                     req_of_token=torch.zeros(len(ids), dtype=torch.int32, device=dev),
                                     page_size=w.page_size, num_pages=w.num_pages, ws=ws)
        enc, lens = S.build_group_union(slots, w.G, w.num_slots, ws=ws)
        o, l = S.sparse_mla_prefill_grouped(qr, w.G, kv_of(w, dev), enc, lens, w.K, w.scale, ws=ws)
        out[idx] = o
        lse[idx] = l
    ref, ref_lse, _ = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                                    block_table=w.block_table, seq_lens=w.seq_lens, req_of_token=w.req_of_token)
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    assert float((out.float() - out_all.float()).abs().max()) <= BF16_OUT_TOL
    assert ws.read_status() == 0
