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


def _bf16_matrix(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("reps,grid", [(1, 1), (3, 1), (5, 4)])
def test_tensor_probe_computes_the_half_tile_contractions(S, reps, grid):
    # S^T = K Q^T over 576 channels and O^T = reps * V^T P^T over the 512 latent channels,
    # against fp64 sums of the same bf16 values (fp32 accumulation in the tensor cores)
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(40 + reps)
    k_rows = _bf16_matrix(rng, (64, 576))
    q = _bf16_matrix(rng, (64, 576))
    pt = torch.from_numpy(rng.random((64, 64)).astype(np.float32)).to(torch.bfloat16)
    ws = S.Workspace(dev)
    s_t, o_t, cycles = S.tensor_probe(k_rows.to(dev), q.to(dev), pt.to(dev), reps=reps, grid=grid, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_status() == 0
    kf, qf, pf = (t.float().double().numpy() for t in (k_rows, q, pt))
    want_s = kf @ qf.T
    want_o = reps * (kf[:, :512].T @ pf)
    assert np.max(np.abs(s_t.cpu().numpy() - want_s)) < 1e-2 + 1e-5 * np.max(np.abs(want_s))
    assert np.max(np.abs(o_t.cpu().numpy() - want_o)) < 1e-2 + 1e-5 * np.max(np.abs(want_o))
    c = cycles.cpu().numpy()
    assert c.shape == (grid,) and np.all(c > 0)
