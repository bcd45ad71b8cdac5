"""The gather probe (svt_gather_probe) really reads every row it is given: each row's XOR of
32-bit words, for both cache layouts and all three ways of moving the rows, against numpy on
the same bytes; skipped slots (negative or past the cache) give 0. The slot count leaves a
ragged last stage of 64 rows."""

import numpy as np
import pytest

from sparse_mla_attention_top_gb300 import workloads as W
from tests._dev import kv_of, to_dev

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


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_gather_probe_reads_every_row(S, mode, kv_dtype):
    dev = torch.device("cuda", 0)
    w = W.make_decode(170, T=3, H=8, K=64, ctx_lo=900, ctx_hi=1500, page_size=16, kv_dtype=kv_dtype)
    rng = np.random.default_rng(mode)
    n = 64 * 37 + 23
    slots = rng.integers(0, w.num_slots, size=n).astype(np.int32)
    slots[5] = -1
    slots[77] = w.num_slots + 4  # past the cache
    slots[n - 1] = -7
    ws = S.Workspace(dev)
    got = S.gather_probe(kv_of(w, dev), to_dev(slots, dev), mode, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    words = w.kv.view(np.uint32)
    want = np.zeros(n, np.uint32)
    live = (slots >= 0) & (slots < w.num_slots)
    want[live] = np.bitwise_xor.reduce(words[slots[live]], axis=1)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want)
