"""Pins of the CPU oracle to facts fixed outside it.

Every test here checks the oracle against something it does not compute itself: values
worked out by hand (tests/golden/), closed forms for constructed inputs whose scores are
known exactly, invariants of the definition, a library conversion (torch's e4m3 cast), or
brute force on tiny inputs. Together they are chosen so that a plausible slip in the oracle
(a dropped rope or latent term, V taking the rope columns, a wrong scale or sign, a
transposed head/channel index, a wrong log base, a mask bit on the wrong member, a merge
weight off by one split) fails at least one of them. No GPU is used.
"""

import math

import numpy as np
import pytest

import oracle
from sparse_mla_attention_top_gb300 import workloads as W
from tests import _golden

ROW, VDIM = 576, 512


# --------------------------------------------------------------------------------- helpers

def bf16_cache(rows_f32: np.ndarray) -> np.ndarray:
    """bf16 cache bytes from float32 rows that are exactly representable in bf16."""
    bits = W.f32_to_bf16_bits(rows_f32)
    assert np.array_equal(W.bf16_bits_to_f32(bits), rows_f32.astype(np.float32)), "not bf16-exact"
    return bits.view(np.uint8).reshape(rows_f32.shape[0], ROW * 2)


def one_hot_q(channel: int, value: float = 1.0) -> np.ndarray:
    q = np.zeros(ROW)
    q[channel] = value
    return q


def random_bf16_rows(rng, n):
    return W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((n, ROW)).astype(np.float32)))


# ------------------------------------------------------------------------------ e4m3 codes

def test_e4m3_table_matches_hand_worked_codes():
    table = oracle.e4m3_table()
    for code, val in _golden.e4m3_cases():
        if math.isnan(val):
            assert math.isnan(table[code]), hex(code)
        else:
            assert table[code] == val and math.copysign(1, table[code]) == math.copysign(1, val), hex(code)


def test_e4m3_table_matches_torch_cast_for_all_codes():
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    table = oracle.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(table))
    assert np.array_equal(ref[~nan], table[~nan])
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}


# --------------------------------------------------------------------------- slot resolution

def test_resolve_hand_worked_example():
    c = _golden.resolve_case()
    slots, err = oracle.resolve(c["topk"], c["topk_len"], c["req_of_token"], c["block_table"], c["seq_lens"],
                                c["page_size"], c["num_pages"])
    assert np.array_equal(slots, c["slots"])
    assert err == c["error"]


def test_resolve_page_id_outside_cache_is_an_error():
    bt = np.array([[1, 9]], np.int32)  # page 9 does not exist in a 4-page cache
    slots, err = oracle.resolve(np.array([[0, 5]], np.int32), block_table=bt, seq_lens=np.array([8], np.int32),
                                page_size=4, num_pages=4)
    assert slots.tolist() == [[4, -1]] and err == 1


def test_resolve_page_size_one_is_table_lookup():
    # The Virtual Block Table, Assumptions and Reasoning, assumption 1: with P = 1,
    # table[req, pos // 1] * 1 + pos % 1 = table[req, pos].
    rng = np.random.default_rng(3)
    bt = np.stack([rng.permutation(500)[:300] for _ in range(3)]).astype(np.int32)
    topk = np.stack([rng.choice(300, 50, replace=False) for _ in range(3)]).astype(np.int32)
    slots, err = oracle.resolve(topk, block_table=bt, seq_lens=np.full(3, 300, np.int32), page_size=1,
                                num_pages=500)
    assert err == 0
    assert np.array_equal(slots, np.take_along_axis(bt, topk, axis=1))


def test_resolve_is_a_bijection_onto_the_requests_slots():
    # Over all positions of a request, resolution hits each slot of its pages exactly once
    # (a shuffled page table only permutes whole pages).
    rng = np.random.default_rng(4)
    P, ctx = 16, 16 * 7 + 5
    bt = rng.permutation(20)[:8].astype(np.int32)[None, :]
    slots, err = oracle.resolve(np.arange(ctx, dtype=np.int32)[None, :], block_table=bt,
                                seq_lens=np.array([ctx], np.int32), page_size=P, num_pages=20)
    assert err == 0
    expect = sorted(int(b) * P + o for i, b in enumerate(bt[0]) for o in range(P) if i * P + o < ctx)
    assert sorted(slots[0].tolist()) == expect
    # contiguous positions inside one page stay contiguous slots
    assert all(slots[0, i + 1] - slots[0, i] == 1 for i in range(ctx - 1) if (i + 1) % P)


def test_resolve_without_table_passes_slots_through_with_range_check():
    topk = np.array([[3, -1, 7, 8]], np.int32)
    slots, err = oracle.resolve(topk, page_size=1, num_pages=8)
    assert slots.tolist() == [[3, -1, 7, -1]] and err == 1


# -------------------------------------------------------------- attention: closed forms

SCALE = 576 ** -0.5


def test_single_index_returns_that_v_row_and_its_score():
    rng = np.random.default_rng(0)
    rows = random_bf16_rows(rng, 6)
    rows[4, 512 + 5] = 1.5
    kv = bf16_cache(rows)
    q = one_hot_q(512 + 5, 2.0)  # a rope channel
    out, lse = oracle.attend_slots(q, kv, oracle.KV_BF16, [4], SCALE)
    assert np.array_equal(out[0], rows[4, :VDIM].astype(np.float64))  # V = first 512 columns only
    assert lse[0] == pytest.approx(SCALE * 2.0 * 1.5, abs=1e-15)


def test_zero_query_gives_mean_of_rows_and_log_count():
    rng = np.random.default_rng(1)
    rows = random_bf16_rows(rng, 10)
    kv = bf16_cache(rows)
    sel = [0, 3, 4, 9, 7]
    out, lse = oracle.attend_slots(np.zeros(ROW), kv, oracle.KV_BF16, sel, SCALE)
    assert np.allclose(out[0], rows[sel, :VDIM].astype(np.float64).mean(axis=0), atol=1e-14)
    assert lse[0] == pytest.approx(math.log(len(sel)), abs=1e-14)


@pytest.mark.parametrize("channel", [7, 300, 511, 512, 575])
def test_two_rows_with_known_scores(channel):
    # q is one-hot on `channel`; the two rows differ there, so s_i = scale * x_i exactly.
    # Latent and rope channels both take part in K; the output only has the 512 latent columns.
    rng = np.random.default_rng(channel)
    rows = random_bf16_rows(rng, 3)
    rows[0, channel], rows[2, channel] = 3.0, -1.25
    kv = bf16_cache(rows)
    s1, s2 = 0.5 * 3.0, 0.5 * -1.25
    out, lse = oracle.attend_slots(one_hot_q(channel), kv, oracle.KV_BF16, [0, 2], 0.5)
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    expect = w1 * rows[0, :VDIM].astype(np.float64) + (1 - w1) * rows[2, :VDIM].astype(np.float64)
    assert np.allclose(out[0], expect, atol=1e-14)
    assert lse[0] == pytest.approx(np.logaddexp(s1, s2), abs=1e-14)  # natural log


def test_each_head_uses_its_own_query_row():
    # Head 0 looks at channel 10, head 1 at rope channel 520: different weights per head.
    rows = np.zeros((2, ROW), np.float32)
    rows[0, 10], rows[1, 10] = 2.0, 0.0
    rows[0, 520], rows[1, 520] = 0.0, 2.0
    rows[0, :VDIM] += 0.0
    rows[0, 100], rows[1, 100] = 1.0, -1.0   # V column 100 tells which row won
    kv = bf16_cache(rows)
    q = np.stack([one_hot_q(10, 4.0), one_hot_q(520, 4.0)])
    out, lse = oracle.attend_slots(q, kv, oracle.KV_BF16, [0, 1], 1.0)
    w = 1.0 / (1.0 + math.exp(-8.0))
    assert out[0, 100] == pytest.approx(w - (1 - w), abs=1e-14)
    assert out[1, 100] == pytest.approx((1 - w) - w, abs=1e-14)
    assert lse[0] == pytest.approx(np.logaddexp(8.0, 0.0), abs=1e-14)


def test_large_scores_do_not_overflow():
    rows = np.zeros((2, ROW), np.float32)
    rows[0, 0], rows[1, 0] = 1000.0, 996.0
    rows[0, 1], rows[1, 1] = 1.0, 3.0
    kv = bf16_cache(rows)
    out, lse = oracle.attend_slots(one_hot_q(0), kv, oracle.KV_BF16, [0, 1], 1.0)
    w0 = 1.0 / (1.0 + math.exp(-4.0))
    assert out[0, 1] == pytest.approx(w0 * 1.0 + (1 - w0) * 3.0, abs=1e-13)
    assert lse[0] == pytest.approx(1000.0 + math.log1p(math.exp(-4.0)), abs=1e-12)


def test_empty_selection():
    kv = bf16_cache(np.zeros((2, ROW), np.float32))
    out, lse = oracle.attend_slots(one_hot_q(0), kv, oracle.KV_BF16, [-1, -1], 1.0)
    assert np.all(out == 0) and lse[0] == -math.inf


# -------------------------------------------------------------- attention: invariants

@pytest.fixture(scope="module")
def small_decode():
    return W.make_decode(11, T=3, H=4, K=96, ctx_lo=150, ctx_hi=400, page_size=8)


def _dec(w, topk, topk_len=None):
    return oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, topk, w.scale,
                         block_table=w.block_table, seq_lens=w.seq_lens, topk_len=topk_len)


def test_index_order_does_not_matter(small_decode):
    w = small_decode
    out, lse, err = _dec(w, w.topk)
    perm = np.random.default_rng(5).permutation(w.K)
    out2, lse2, err2 = _dec(w, w.topk[:, perm])
    assert err == err2 == 0
    assert np.allclose(out, out2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)


def test_minus_one_padding_anywhere_is_ignored(small_decode):
    w = small_decode
    out, lse, _ = _dec(w, w.topk)
    rng = np.random.default_rng(6)
    padded = np.full((w.T, w.K + 40), -1, np.int32)
    for t in range(w.T):
        where = np.sort(rng.choice(w.K + 40, w.K, replace=False))
        padded[t, where] = w.topk[t]
    out2, lse2, err = _dec(w, padded)
    assert err == 0
    assert np.allclose(out, out2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)


def test_entries_past_the_live_count_are_ignored(small_decode):
    w = small_decode
    n = np.array([5, 96, 40], np.int32)
    out, lse, _ = _dec(w, w.topk, topk_len=n)
    cut = w.topk.copy()
    for t in range(w.T):
        cut[t, n[t]:] = -1
    out2, lse2, _ = _dec(w, cut)
    assert np.allclose(out, out2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)


def test_topk_all_equals_dense_paged_attention():
    # The Virtual Block Table, The Breakthrough: the sparse list through a page_size-1 view and
    # the dense walk over the request's pages are the same attention when the list holds
    # every position.
    w = W.make_decode(12, T=2, H=3, K=205, ctx_lo=205, ctx_hi=205, page_size=16)
    rng = np.random.default_rng(7)
    topk = np.stack([rng.permutation(205) for _ in range(2)]).astype(np.int32)
    out, lse, err = _dec(w, topk)
    assert err == 0
    for t in range(2):
        d_out, d_lse = oracle.dense_paged(w.q_bits[t], w.kv, w.kv_dtype, w.block_table[t], 205, w.page_size, w.scale)
        assert np.allclose(out[t], d_out, atol=1e-12) and np.allclose(lse[t], d_lse, atol=1e-12)


def test_slots_through_virtual_table_match_positions_through_pages(small_decode):
    # Resolving first and passing slots with no table (page_size 1 view) changes nothing.
    w = small_decode
    out, lse, _ = _dec(w, w.topk)
    slots, err = oracle.resolve(w.topk, block_table=w.block_table, seq_lens=w.seq_lens, page_size=w.page_size,
                                num_pages=w.num_pages)
    out2, lse2, err2 = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_slots, 1, slots.astype(np.int32), w.scale)
    assert err == err2 == 0
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_out_of_range_position_is_flagged_and_skipped(small_decode):
    w = small_decode
    bad = w.topk.copy()
    bad[1, 3] = w.seq_lens[1] + 5
    out, lse, err = _dec(w, bad)
    dropped = bad.copy()
    dropped[1, 3] = -1
    out2, lse2, _ = _dec(w, dropped)
    assert err == 1 and np.array_equal(out, out2)


def test_duplicate_index_is_flagged(small_decode):
    w = small_decode
    dup = w.topk.copy()
    dup[0, 1] = dup[0, 0]
    assert _dec(w, dup)[2] == 2


# ------------------------------------------------------------------------------ fp8 cache

def _fp8_rows(codes, scales, rope_bits):
    n = codes.shape[0]
    out = np.empty((n, 656), np.uint8)
    out[:, :512] = codes
    out[:, 512:528] = scales.astype(np.float32).view(np.uint8).reshape(n, 16)
    out[:, 528:] = rope_bits.view(np.uint8).reshape(n, 128)
    return out


def test_fp8_with_unit_scales_equals_bf16_cache_of_the_same_values():
    rng = np.random.default_rng(8)
    n = 40
    codes = rng.integers(0, 256, size=(n, 512), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    rope = W.f32_to_bf16_bits(rng.standard_normal((n, 64)).astype(np.float32))
    fp8 = _fp8_rows(codes, np.ones((n, 4)), rope)
    vals = oracle.e4m3_table()[codes].astype(np.float32)  # e4m3 values are exact in bf16
    bf = bf16_cache(np.concatenate([vals, W.bf16_bits_to_f32(rope)], axis=1))
    q = rng.standard_normal((3, ROW))
    sel = rng.choice(n, 25, replace=False)
    o8, l8 = oracle.attend_slots(q, fp8, oracle.KV_FP8_E4M3, sel, 0.05)
    ob, lb = oracle.attend_slots(q, bf, oracle.KV_BF16, sel, 0.05)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_fp8_block_scale_applies_to_its_128_channels_only():
    # code 0x40 (2.0) with scale 0.5 in block 1 equals code 0x38 (1.0) with scale 1.0.
    n = 2
    codes = np.full((n, 512), 0x38, np.uint8)
    rope = np.zeros((n, 64), np.uint16)
    a = _fp8_rows(codes, np.ones((n, 4)), rope)
    codes_b = codes.copy()
    codes_b[:, 128:256] = 0x40
    scales_b = np.ones((n, 4))
    scales_b[:, 1] = 0.5
    b = _fp8_rows(codes_b, scales_b, rope)
    ra = oracle.fetch_rows(a, oracle.KV_FP8_E4M3, [0, 1])
    rb = oracle.fetch_rows(b, oracle.KV_FP8_E4M3, [0, 1])
    assert np.array_equal(ra, rb) and np.all(ra[:, :512] == 1.0) and np.all(ra[:, 512:] == 0.0)
    scales_c = np.ones((n, 4))
    scales_c[:, 2] = 3.0
    rc = oracle.fetch_rows(_fp8_rows(codes, scales_c, rope), oracle.KV_FP8_E4M3, [0])
    assert np.all(rc[0, 256:384] == 3.0) and np.all(rc[0, :256] == 1.0) and np.all(rc[0, 384:512] == 1.0)


# ---------------------------------------------------------------------------------- union

def test_union_hand_worked_cases():
    for c in _golden.union_cases():
        slots = np.array(c["rows"], np.int32)
        lens_rows = np.array(c["lens_rows"], np.int32)
        enc, lens, err = oracle.group_union(slots, c["G"], c["num_slots"], topk_len=lens_rows)
        assert err == 0, c["name"]
        for g, (n, pairs) in c["groups"].items():
            assert lens[g] == n, c["name"]
            expect = [_golden.encode(m, s) for m, s in pairs] + [-1] * (c["G"] * c["K"] - n)
            assert enc[g].tolist() == expect, c["name"]


def test_union_brute_force_on_random_tiny_groups():
    rng = np.random.default_rng(9)
    for G in (2, 4, 8):
        for trial in range(20):
            T, K = int(rng.integers(1, 3 * G)), int(rng.integers(1, 12))
            slots = rng.integers(-3, 30, size=(T, K)).astype(np.int32)
            for t in range(T):  # distinct live entries per query
                live = slots[t][slots[t] >= 0]
                u, idx = np.unique(live, return_index=True)
                keep = np.zeros(len(live), bool)
                keep[idx] = True
                slots[t][np.nonzero(slots[t] >= 0)[0][~keep]] = -1
            lens_rows = rng.integers(0, K + 1, size=T).astype(np.int32)
            enc, lens, err = oracle.group_union(slots, G, 30, topk_len=lens_rows)
            assert err == 0
            for g in range(enc.shape[0]):
                members = {}
                for m in range(G):
                    t = g * G + m
                    if t < T:
                        members[m] = {int(s) for s in slots[t, :lens_rows[t]] if s >= 0}
                union = sorted(set().union(*members.values())) if members else []
                assert lens[g] == len(union)
                got = enc[g].view(np.uint32)
                assert [int(x) & 0xFFFFFF for x in got[:lens[g]]] == union
                for i, s in enumerate(union):
                    mask = int(got[i]) >> 24
                    for m in range(G):
                        assert bool((mask >> m) & 1) == (m in members and s in members[m])
                assert np.all(enc[g, lens[g]:] == -1)


def test_union_flags_out_of_range_and_duplicates():
    enc, lens, err = oracle.group_union(np.array([[1, 40], [2, 2]], np.int32), 2, 30)
    assert err == 3 and lens[0] == 2


# ---------------------------------------------------------------------------------- merge

def test_merge_of_one_split_is_identity():
    rng = np.random.default_rng(10)
    o = rng.standard_normal((1, 3, 512)).astype(np.float32)
    l = rng.standard_normal((1, 3)).astype(np.float32)
    out, lse = oracle.merge(o, l)
    assert np.array_equal(out, o[0].astype(np.float64)) and np.array_equal(lse, l[0].astype(np.float64))


def test_merge_of_halves_equals_unsplit_attention():
    rng = np.random.default_rng(11)
    rows = random_bf16_rows(rng, 200)
    kv = bf16_cache(rows)
    q = rng.standard_normal((2, ROW))
    sel = rng.choice(200, 150, replace=False)
    parts = [sel[:37], sel[37:100], sel[100:]]
    o_part, l_part = [], []
    for p in parts:
        o, l = oracle.attend_slots(q, kv, oracle.KV_BF16, p, 0.1)
        o_part.append(o)
        l_part.append(l)
    # an empty split weighs nothing
    o_part.append(np.zeros((2, 512)))
    l_part.append(np.full(2, -np.inf))
    out, lse = oracle.merge(np.array(o_part, np.float32), np.array(l_part, np.float32))
    ref, ref_lse = oracle.attend_slots(q, kv, oracle.KV_BF16, sel, 0.1)
    assert np.allclose(out, ref, atol=2e-6) and np.allclose(lse, ref_lse, atol=2e-6)


def test_merge_all_empty():
    out, lse = oracle.merge(np.zeros((2, 1, 512), np.float32), np.full((2, 1), -np.inf, np.float32))
    assert np.all(out == 0) and lse[0] == -np.inf


# ------------------------------------------------------------------------ grouped prefill

@pytest.fixture(scope="module")
def small_prefill():
    return W.make_prefill(13, n_new=21, n_cached=90, H=4, G=4, K=64, page_size=16)


def _union_of(w):
    slots, err = oracle.resolve(w.topk, req_of_token=w.req_of_token, block_table=w.block_table,
                                seq_lens=w.seq_lens, page_size=w.page_size, num_pages=w.num_pages)
    assert err == 0
    enc, lens, err = oracle.group_union(slots.astype(np.int32), w.G, w.num_slots)
    assert err == 0
    return slots, enc, lens


def test_grouped_prefill_equals_per_query_decode(small_prefill):
    w = small_prefill
    _, enc, lens = _union_of(w)
    out, lse, err = oracle.prefill_grouped(w.q_bits, w.G, w.kv, w.kv_dtype, w.num_slots, enc, lens, w.K, w.scale)
    assert err == 0
    ref, ref_lse, err = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                                      block_table=w.block_table, req_of_token=w.req_of_token, seq_lens=w.seq_lens)
    assert err == 0
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, ref_lse, atol=1e-12)
    # the tail group (21 = 5 * 4 + 1) has one member; its union is that member's list
    assert lens[-1] == np.count_nonzero(w.topk[20] >= 0)


def test_flipping_a_membership_bit_breaks_the_invariant(small_prefill):
    # Negative control: a mask bit on the wrong member must change that member's output.
    w = small_prefill
    _, enc, lens = _union_of(w)
    bad = enc.copy()
    g = 3
    e = int(np.nonzero((bad[g, :lens[g]].view(np.uint32) >> 24) & 2 == 0)[0][0])  # member 1 lacks it
    bad[g, e] = int(np.array([bad[g, e]], np.int32).view(np.uint32)[0] | (2 << 24))
    out, lse, _ = oracle.prefill_grouped(w.q_bits, w.G, w.kv, w.kv_dtype, w.num_slots, bad, lens, w.K, w.scale,
                                         query_ids=[g * w.G + 1])
    ref, ref_lse, _ = oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                                    block_table=w.block_table, req_of_token=w.req_of_token, seq_lens=w.seq_lens,
                                    query_ids=[g * w.G + 1])
    assert not np.allclose(lse, ref_lse, atol=1e-3)


def test_dropping_the_tail_groups_output_fails_the_parity_check(small_prefill):
    # Negative control for the parity harness (vLLM PR #63104, Tests: dropping the tail's
    # output must fail): the oracle's own result, rounded as the GPU returns it, passes the
    # comparison the GPU tests use; the same result with the short last group's rows zeroed
    # (a kernel that skipped the tail) does not.
    torch = pytest.importorskip("torch")
    from tests._dev import BF16_OUT_TOL, compare

    w = small_prefill
    _, enc, lens = _union_of(w)
    ref, ref_lse, err = oracle.prefill_grouped(w.q_bits, w.G, w.kv, w.kv_dtype, w.num_slots, enc, lens, w.K, w.scale)
    assert err == 0
    out = torch.from_numpy(ref).to(torch.bfloat16)
    lse = torch.from_numpy(ref_lse.astype(np.float32))
    compare(out, lse, ref, ref_lse, BF16_OUT_TOL)
    tail = (w.T // w.G) * w.G  # 21 queries in groups of 4: query 20 is the tail group
    dropped_out, dropped_lse = out.clone(), lse.clone()
    dropped_out[tail:] = 0
    dropped_lse[tail:] = -math.inf
    with pytest.raises(AssertionError):
        compare(dropped_out, dropped_lse, ref, ref_lse, BF16_OUT_TOL)


def test_generators_hold_their_stated_shapes():
    w = W.make_prefill(14, n_new=40, n_cached=2100, H=2, G=2, K=64, page_size=64)
    live = [set(int(x) for x in row if x >= 0) for row in w.topk]
    assert all(len(s) == 64 for s in live)
    assert all(max(s) <= 2100 + i for i, s in enumerate(live))  # causal prefix only
    overlap = np.mean([len(live[i] & live[i - 1]) / 64 for i in range(1, 40)])
    assert 0.65 <= overlap <= 0.8


# ----------------------------------------------------------------------------- top-k selection


@pytest.mark.parametrize("case", _golden.topk_cases(), ids=lambda c: c["name"])
def test_topk_hand_worked_cases(case):
    lens = None if case["len"] is None else np.array([case["len"]], np.int32)
    got = oracle.topk_select(case["scores"][None, :], case["K"], lens=lens)[0]
    assert np.array_equal(got, case["expect"]), (got, case["expect"])


def _topk_by_rank_count(row, K, length):
    """Position j is kept iff fewer than K candidates outrank it (greater score, or an equal
    score at a lower position; NaN below every number): a quadratic count, written apart
    from the oracle's sorts."""
    def beats(a, b):
        xa, xb = row[a], row[b]
        if np.isnan(xa) or np.isnan(xb):
            if np.isnan(xa) and np.isnan(xb):
                return a < b
            return np.isnan(xb)
        return xa > xb or (xa == xb and a < b)
    kept = [j for j in range(length) if sum(beats(i, j) for i in range(length) if i != j) < K]
    return np.array(kept + [-1] * (K - len(kept)), np.int32)


def test_topk_matches_rank_counting_on_random_rows_with_ties():
    rng = np.random.default_rng(11)
    for trial in range(60):
        n = int(rng.integers(1, 40))
        K = int(rng.integers(1, 20))
        # few distinct values, some NaN / infinities / signed zeros, so ties are common
        pool = np.array([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan], np.float32)
        row = rng.choice(pool, size=n).astype(np.float32)
        length = int(rng.integers(0, n + 1))
        got = oracle.topk_select(row[None, :], K, lens=np.array([length], np.int32))[0]
        assert np.array_equal(got, _topk_by_rank_count(row, K, length)), (trial, row, K, length, got)


def test_topk_output_invariants():
    rng = np.random.default_rng(12)
    T, N, K = 6, 300, 64
    scores = rng.standard_normal((T, N)).astype(np.float32)
    lens = np.array([0, 1, 63, 64, 65, 300], np.int32)
    out = oracle.topk_select(scores, K, lens=lens)
    for t in range(T):
        m = min(K, int(lens[t]))
        kept = out[t, :m]
        assert np.all(out[t, m:] == -1)
        assert np.all(np.diff(kept) > 0) and (m == 0 or (kept[0] >= 0 and kept[-1] < lens[t]))
        if 0 < m < lens[t]:
            # every kept score is at least every dropped one
            dropped = np.setdiff1d(np.arange(lens[t]), kept)
            assert scores[t, kept].min() >= scores[t, dropped].max()
