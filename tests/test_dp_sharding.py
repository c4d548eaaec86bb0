"""Data parallelism over tokens, checked on the CPU with two gloo ranks.

The stack is independent across tokens except for the loss means, so a rank that holds rows
[b, e) of a global batch of M rows and takes its means over M (token_count = M) owns exactly
its share of the loss and of every dA, dB; the global gradients are the ranks' sum.  Each
rank here runs the oracle on its shard, the ranks all-gather their gradients over gloo and
sum them in rank order -- the same exchange the GPU path performs with NCCL and
lsn_sum_ranks -- and the result must be the single-rank oracle's on the whole batch."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import layer_streamed_nf4_quant_b300 as lsn  # noqa: E402

D, DKV, F, R, L, M = 256, 256, 512, 16, 2, 96


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layers():
    import synth
    from oracle import nf4 as onf4
    from oracle.nf4 import bf16_value
    out = []
    for l in range(L):
        W = synth.layer_weights(l, D, DKV, F)
        A, B = synth.layer_lora(l, R, D, DKV, F)
        out.append(({p: onf4.dequantize(onf4.quantize(w)) for p, w in W.items()},
                    {p: bf16_value(a).astype(np.float64) for p, a in A.items()},
                    {p: bf16_value(b).astype(np.float64) for p, b in B.items()}))
    return out


def _flat(ref):
    parts = []
    for l in range(L):
        for p in sorted(ref["dA"][l]):
            parts += [ref["dA"][l][p].ravel(), ref["dB"][l][p].ravel()]
    return np.concatenate(parts)


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import synth
    from oracle import stack as ostack
    from oracle.nf4 import bf16_value
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b, e = lsn.shard_range(M, world, rank)
        x0 = bf16_value(synth.stack_input(M, D)).astype(np.float64)[b:e]
        ref = ostack.stack_forward_backward(x0, _layers(), 1.0, token_count=M)
        mine = torch.from_numpy(_flat(ref))
        gathered = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)
        total = gathered[0].clone()
        for g in gathered[1:]:          # rank order, as lsn_sum_ranks adds
            total += g
        loss = torch.tensor([ref["loss"]], dtype=torch.float64)
        dist.all_reduce(loss)
        q.put((rank, b, e, total.numpy(), float(loss.item()), ref["dx0"]))
    finally:
        dist.destroy_process_group()


def test_shard_ranges_partition_the_batch():
    for tokens, world in ((96, 2), (97, 3), (512, 8), (8, 8)):
        ranges = [lsn.shard_range(tokens, world, r) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == tokens
        assert all(ranges[i][1] == ranges[i + 1][0] for i in range(world - 1))
        sizes = [e - b for b, e in ranges]
        assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        lsn.shard_range(3, 4, 0)


def test_two_gloo_ranks_sum_to_the_single_rank_gradients():
    import torch.multiprocessing as mp
    import synth
    from oracle import stack as ostack
    from oracle.nf4 import bf16_value
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=300) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    full = ostack.stack_forward_backward(bf16_value(synth.stack_input(M, D)).astype(np.float64), _layers(), 1.0)
    want = _flat(full)
    for rank, b, e, total, loss, dx0 in out:
        np.testing.assert_array_equal(total, out[0][3])                 # every rank holds the same bits
        assert np.linalg.norm(total - want) <= 1e-12 * np.linalg.norm(want)
        assert loss == pytest.approx(full["loss"], rel=1e-12)
        np.testing.assert_allclose(dx0, full["dx0"][b:e], rtol=0, atol=1e-15 * np.abs(full["dx0"]).max())
