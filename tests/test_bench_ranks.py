"""The N > 1 path of bench.py, on CPU: every rank runs its own replica of the workload, the
ranks agree on the slowest rank's time, and the whole-job rate counts all ranks' tokens.
Two gloo ranks in spawned processes (rendezvous on 127.0.0.1)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, 10.0 + 5.0 * rank, "cpu")   # rank 1 is the slow one
        dist.barrier()
        q.put((rank, ms, bench.whole_job_rate(world, 512, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_token():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in out] == [0, 1]
    for _, ms, rate in out:
        assert ms == 15.0
        assert rate == pytest.approx(2 * 512 / 0.015)


def test_single_rank_passes_its_own_time():
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.whole_job_rate(1, 512, 130.0) == pytest.approx(512 / 0.13)
