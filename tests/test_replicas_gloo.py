"""The N > 1 path of bench.py (independent replicas, one per rank, timed by the slowest),
exercised with two gloo ranks on the CPU."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank)
    ms = [1.5, 4.0][rank]  # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms, w)
    bench.barrier(w)
    q.put((rank, ms_max, bench.replica_throughput(64, ms_max, w)))
    dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_and_add_their_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, value in res:
        assert ms_max == 4.0                           # max over ranks
        assert value == pytest.approx(64 * 2 / 4.0e-3)  # both replicas' queries / slowest time


def _reference_rank(rank, q):
    os.environ.update(WORLD_SIZE="2", RANK=str(rank))
    import contextlib
    import io

    import bench

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        if rank == 1:
            bench.run_reference(type("A", (), {"decode_T": 4, "warmup": 0, "steps": 1, "gpus": 2})())
    q.put((rank, buf.getvalue()))


def test_reference_arm_runs_on_rank_zero_only():
    # a non-zero rank of the reference arm exits without work or output
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_reference_rank, args=(1, q))
    p.start()
    p.join(timeout=120)
    assert p.exitcode == 0
    rank, out = q.get(timeout=10)
    assert rank == 1 and out == ""
