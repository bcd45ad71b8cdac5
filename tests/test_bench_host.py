"""Host-side accounting of bench.py: the kept-entry counts behind the executed-flop figure of
grouped prefill, against a brute-force count over the union's membership masks, and the
phase-trace analyses on synthetic stamps with known answers."""

import numpy as np
import pytest

import bench


@pytest.mark.parametrize("H,G", [(64, 2), (32, 4), (16, 8)])
def test_rowset_kept_counts_brute_force(H, G):
    rng = np.random.default_rng(H)
    groups, width = 5, 40
    enc = np.full((groups, width), -1, np.int32)
    lens = rng.integers(0, width + 1, size=groups)
    for g in range(groups):
        masks = rng.integers(1, 1 << G, size=lens[g])
        slots = np.sort(rng.choice(1 << 20, size=lens[g], replace=False))
        enc[g, : lens[g]] = ((masks.astype(np.int64) << 24) | slots).astype(np.uint32).view(np.int32)
    got = bench.rowset_kept_counts(enc, lens.astype(np.int64), H)
    want = []
    for g in range(groups):
        for half in range(2):
            members = {(half * 64 + r) // H for r in range(64)}
            n = 0
            for i in range(lens[g]):
                m = (int(enc[g, i]) & 0xFFFFFFFF) >> 24
                n += any((m >> b) & 1 for b in members)
            want.append(n)
    assert got.tolist() == want


def test_phase_trace_analysis_on_a_synthetic_launch():
    # two CTAs at 2 GHz (2 cycles per ns): set-up 1000 cycles, half-tiles every 4000 cycles,
    # rows landing 1500 cycles after their fill is issued, S^T done 800 cycles after issue
    slots = bench.TRACE_HEAD + bench.TRACE_G * bench.TRACE_EV
    tr = np.zeros((4, slots), np.uint64)
    for c in range(2):
        c0, gt0 = 10_000 + 37 * c, 5_000_000 + 100 * c
        n = 10
        ev = np.zeros((bench.TRACE_G, bench.TRACE_EV), np.int64)
        for g in range(n):
            issue = c0 + 6000 + 4000 * g
            ev[g, :8] = [issue - 500, issue - 100, issue, issue + 800, issue + 1400, issue + 1500, issue - 3000,
                         issue - 1600]
            ev[g, 8:11] = [issue + 900, issue + 1000, issue + 1300]
        end = c0 + 6000 + 4000 * n + 3000
        tr[c, 0], tr[c, 1], tr[c, 2], tr[c, 3], tr[c, 4] = gt0, c0, c0 + 1000, c0 + 1200, c0 + 2000
        tr[c, 5], tr[c, 6], tr[c, 7], tr[c, 9] = end - 2000, end - 1000, end - 500, end
        tr[c, 14], tr[c, 15] = n, gt0 + (end - c0) // 2
        tr[c, bench.TRACE_HEAD:] = ev.reshape(-1).astype(np.uint64)
    out = bench.analyse_trace(tr)
    assert out["ctas"] == 2 and abs(out["sm_ghz"] - 2.0) < 1e-6
    assert out["half_tile_period_us"] == pytest.approx(2.0)      # 4000 cycles
    assert out["fill_issue_to_landed_us"] == pytest.approx(0.75)  # 1500 cycles
    assert out["s_issue_to_done_us"] == pytest.approx(0.4)
    assert out["softmax_us"] == pytest.approx(0.3)
    assert out["setup_us"] == pytest.approx(0.5)
    assert out["first_s_issued_us"] == pytest.approx(3.0)
    assert out["s_issuer_wait_rows_us"] == pytest.approx(0.2)     # buffer free at -500, rows at -100
    assert out["softmax_tmem_load_us"] == pytest.approx(0.05)
    assert out["softmax_fence_arrive_us"] == pytest.approx(0.05)
    assert out["cluster_merge_us"] is None and "cluster_merge_steps_us" not in out


def test_phase_trace_merge_steps():
    # one clustered CTA: merge stamps 1000 cycles apart from "roles done" (slot 7) on
    slots = bench.TRACE_HEAD + bench.TRACE_G * bench.TRACE_EV
    tr = np.zeros((1, slots), np.uint64)
    c0, gt0 = 50_000, 9_000_000
    tr[0, 0], tr[0, 1], tr[0, 7] = gt0, c0, c0 + 10_000
    order = [24, 25, 26, 27, 16, 17, 21, 22, 18, 8]
    for k, slot in enumerate(order):
        tr[0, slot] = c0 + 10_000 + 1000 * (k + 1)
    tr[0, 9] = c0 + 30_000
    tr[0, 15] = gt0 + 15_000  # 2 cycles per ns
    out = bench.analyse_trace(tr)
    assert out["cluster_merge_us"] == pytest.approx(5.0)
    steps = out["cluster_merge_steps_us"]
    assert list(steps) == ["lse_headers", "o_from_tmem", "pack", "cluster_barrier", "issue_copies", "copies_land",
                           "weights", "weights_barrier", "combine_and_store", "final_barrier"]
    assert all(v == pytest.approx(0.5) for v in steps.values())


def test_row_set_switch_analysis_on_a_synthetic_window():
    # one CTA at 2 GHz; traced half-tiles 0..11 of a mid-launch window: the last six of a
    # 32-half-tile row-set (index 27..32), then a new row-set (index 1..6). S^T issues every
    # 4000 cycles except into the new row-set (8000); the new row-set's Q^T is issued 2600
    # cycles after the last S^T and seen 1800 later; the epilogue ends 5000 cycles after the
    # old row-set's last P^T.
    slots = bench.TRACE_HEAD + bench.TRACE_G * bench.TRACE_EV
    tr = np.zeros((1, slots), np.uint64)
    c0, gt0 = 100_000, 7_000_000
    ev = np.zeros((bench.TRACE_G, bench.TRACE_EV), np.int64)
    issue = c0 + 50_000
    for k in range(12):
        if k > 0:
            issue += 8000 if k == 6 else 4000
        ev[k, 0], ev[k, 1], ev[k, 11], ev[k, 2] = issue - 3000, issue - 2900, issue - 2800, issue
        ev[k, 3], ev[k, 4], ev[k, 5] = issue + 300, issue + 1900, issue + 3500
        ev[k, 12] = 27 + k if k < 6 else k - 5
    ev[6, 14] = ev[5, 2] + 2600
    ev[6, 15] = ev[6, 14] + 1800
    ev[6, 13] = ev[5, 4] + 5000
    tr[0, 0], tr[0, 1], tr[0, 7], tr[0, 9] = gt0, c0, c0 + 3_000_000, c0 + 3_000_100
    tr[0, 14], tr[0, 23], tr[0, 15] = 1500, 50, gt0 + 3_000_100 // 2
    tr[0, bench.TRACE_HEAD:] = ev.reshape(-1).astype(np.uint64)
    out = bench.analyse_boundaries(tr)
    assert out["switches"] == 1
    assert out["steady_period_us"] == pytest.approx(2.0)
    assert out["period_into_us"] == pytest.approx(4.0)
    assert out["switch_extra_us"] == pytest.approx(2.0)           # 20000 cycles against 4 x 4000
    assert out["prev_s_issued_to_q_issued_us"] == pytest.approx(1.3)
    assert out["q_issued_to_q_seen_us"] == pytest.approx(0.9)
    assert out["epilogue_us"] == pytest.approx(2.5)
    assert out["previous_segment_half_tiles_median"] == 32
    assert out["segments_per_cta_median"] == 50
    assert out["roles_done_per_half_tile_us"] == pytest.approx(1.0)  # 3e6 cycles / 1500 at 2 GHz
    # the window analysis of the same stamps reports the mid-launch period and no first-tile times
    w = bench.analyse_trace(tr, window=True)
    assert w["half_tile_period_us"] == pytest.approx(2.0) and "first_s_issued_us" not in w
