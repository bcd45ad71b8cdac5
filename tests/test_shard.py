"""Zigzag token split for sharded grouped prefill: host-side partition properties, and the
partition agreed by two gloo ranks on the CPU."""

import os
import socket

import numpy as np
import pytest

from sparse_mla_attention_top_gb300.shard import zigzag_split


@pytest.mark.parametrize("n,world", [(0, 2), (7, 4), (8192, 4), (15000, 8), (3, 1)])
def test_zigzag_covers_every_token_once(n, world):
    parts = zigzag_split(n, world)
    assert len(parts) == world
    allt = np.concatenate(parts) if parts else np.array([], np.int64)
    assert np.array_equal(np.sort(allt), np.arange(n))
    for p in parts:
        assert np.all(np.diff(p) > 0)


def test_zigzag_gives_each_rank_an_early_and_a_late_chunk():
    parts = zigzag_split(8000, 4)
    # chunks of 1000: rank r has [1000 r, 1000 (r+1)) and [1000 (7-r), 1000 (8-r))
    for r, p in enumerate(parts):
        assert p[0] == 1000 * r and p[-1] == 1000 * (8 - r) - 1 and len(p) == 2000


def test_zigzag_balances_causal_work():
    n, world = 32768, 4
    work = [int((p + 1).sum()) for p in zigzag_split(n, world)]  # prefix lengths seen
    assert max(work) / min(work) < 1.01
    contiguous = [int((np.arange(r * n // world, (r + 1) * n // world) + 1).sum()) for r in range(world)]
    assert max(contiguous) / min(contiguous) > 5


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = torch.from_numpy(zigzag_split(1001, world)[rank])
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([len(mine)]))
    out = [torch.zeros(int(s.item()), dtype=torch.int64) for s in sizes]
    # gloo all_gather needs equal sizes: pad to the largest
    m = max(int(s.item()) for s in sizes)
    padded = torch.full((m,), -1, dtype=torch.int64)
    padded[: len(mine)] = mine
    gathered = [torch.zeros(m, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(gathered, padded)
    allt = torch.cat([g[g >= 0] for g in gathered])
    q.put((rank, sorted(allt.tolist()) == list(range(1001))))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_a_partition_of_all_tokens():
    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert all(ok for _, ok in (q.get(timeout=10) for _ in range(2)))
