"""Host-side accounting of bench.py: the kept-entry counts behind the executed-flop figure of
grouped prefill, against a brute-force count over the union's membership masks."""

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
