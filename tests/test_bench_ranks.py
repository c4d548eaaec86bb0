"""The N > 1 path of bench.py, on CPU: every rank runs its own token shard of the batch, the
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


def test_gpus_flag_starts_one_rank_per_gpu_without_a_launcher():
    """`bench.py --gpus 2` with no launcher in the environment starts two local ranks through
    torch.distributed.run (rendezvous on 127.0.0.1); each rank binds the device of its local
    rank.  --show-ranks stops each rank right after the binding, before any device work."""
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    for attempt in range(2):   # the port bench.py picks can be taken before the launcher binds it
        r = subprocess.run([sys.executable, bench.__file__, "--gpus", "2", "--show-ranks"], capture_output=True,
                           text=True, timeout=180, env=env)
        if r.returncode == 0:
            break
    assert r.returncode == 0, r.stderr
    ranks = sorted((json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")), key=lambda d: d["rank"])
    assert [d["rank"] for d in ranks] == [0, 1]
    assert all(d["world"] == 2 for d in ranks)
    assert [d["device"] for d in ranks] == ["cuda:0", "cuda:1"]


def test_launcher_world_must_match_gpus():
    cmd = bench.launcher_command(4, ["--gpus", "4"], 12345)
    assert "--nproc-per-node=4" in cmd and "127.0.0.1" in cmd and cmd[-2:] == ["--gpus", "4"]
    bench.check_world(2, 2)
    with pytest.raises(SystemExit):
        bench.check_world(2, 1)
