"""GPU tests of the data-parallel pieces on one device: the fixed-order rank sum, the step's
global token count and per-layer gradient hook, and DataParallel's exchange.

Ranks are emulated one after another in one process (nothing waits on another rank): each
"rank" runs layer_stack_step on its contiguous token shard with token_count = the global
batch, and the shards' gradients summed in rank order must be the full batch's gradients --
up to the fp32 order of the token contraction and the bf16 roundings it can flip."""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from test_gpu_stack import Stack, _oracle, _grad_views  # noqa: E402

SHARD_TOL = 2e-3     # relative Frobenius, shard sum vs the full batch on the device
GRAD_TOL = 1e-2      # the stated gradient bar, against the oracle


def _lsn():
    import layer_streamed_nf4_quant_b300 as lsn
    return lsn


def _fro(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("n_ranks,n", [(1, 1000), (2, 4096), (3, 1001), (8, 65539)])
def test_sum_ranks_is_the_rank_ordered_fp32_sum(n_ranks, n):
    lsn = _lsn()
    rng = np.random.default_rng(n_ranks * 7 + n)
    g = (rng.standard_normal((n_ranks, n)) * 10.0 ** rng.uniform(-3, 3, (n_ranks, 1))).astype(np.float32)
    want = g[0].copy()
    for r in range(1, n_ranks):
        want = want + g[r]                    # float32 adds, rank order
    gathered = torch.from_numpy(g).cuda().reshape(-1)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    lsn.sum_ranks(gathered, n_ranks, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))
    lsn.sum_ranks(gathered, n_ranks, gathered[:n])     # in place into in[0]
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gathered[:n].cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.fixture(scope="module")
def small():
    lsn = _lsn()
    return Stack(lsn.StackDesc(n_layers=3, d_model=256, d_kv=256, d_ff=512, rank=16), M=300)


def _run_shard(st, b, e, token_count, hook=None, calls=None):
    lsn = _lsn()
    d = st.desc
    x0 = st.x0[b:e].contiguous()
    grads = [torch.full((d.lora_elems,), float("nan"), dtype=torch.float32, device="cuda")
             for _ in range(d.n_layers)]
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    dx0 = torch.empty((e - b, d.d_model), dtype=torch.float32, device="cuda")
    ws = torch.empty(d.workspace_bytes(e - b), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    if hook is None and calls is not None:
        hook = _lsn().lsn_layer_hook(lambda user, layer, ptr, elems, s: calls.append((layer, ptr, elems, s)))
    lsn.layer_stack_step(d, x0, st.lora, grads, loss, ws, resident_store=st.resident, dx0=dx0, stream=stream,
                         token_count=token_count, grads_ready=hook)
    torch.cuda.synchronize()
    assert lsn.device_check() == 0
    return {"grads": grads, "loss": loss, "dx0": dx0, "stream": stream}


@pytest.mark.parametrize("world", [2, 3])
def test_token_shards_sum_to_the_full_batch(small, world):
    lsn = _lsn()
    d, M = small.desc, small.M
    full = small.run()
    shards, calls = [], []
    for r in range(world):
        b, e = lsn.shard_range(M, world, r)
        seen = []
        shards.append((b, e, _run_shard(small, b, e, M, calls=seen)))
        calls.append(seen)
    for (b, e, out), seen in zip(shards, calls):
        # the hook ran once per layer, last layer first, on that layer's gradient blob
        assert [c[0] for c in seen] == list(range(d.n_layers - 1, -1, -1))
        assert [c[1] for c in seen] == [out["grads"][c[0]].data_ptr() for c in seen]
        assert all(c[2] == d.lora_elems for c in seen)
        assert all(c[3] == out["stream"].cuda_stream for c in seen)
        assert _fro(out["dx0"], full["dx0"][b:e]) <= SHARD_TOL
    loss = sum(float(o["loss"].item()) for _, _, o in shards)
    assert abs(loss - full["loss"].item()) <= 1e-4 * full["loss"].item()
    ref = _oracle(small)
    for l in range(d.n_layers):
        gathered = torch.cat([o["grads"][l] for _, _, o in shards])
        total = torch.empty(d.lora_elems, dtype=torch.float32, device="cuda")
        lsn.sum_ranks(gathered, world, total)
        torch.cuda.synchronize()
        assert _fro(total, full["grads"][l]) <= SHARD_TOL, l
        gA, gB = _grad_views(small, total)
        for p in gA:
            for got, want in ((gA[p], ref["dA"][l][p]), (gB[p], ref["dB"][l][p])):
                assert np.linalg.norm(got - want) / np.linalg.norm(want) <= GRAD_TOL, (l, p)


def test_shard_without_global_count_is_not_its_share(small):
    """The same shard with token_count left at 0 takes its means over its own rows: its
    gradients are world times its share (a pin on what token_count changes)."""
    lsn = _lsn()
    b, e = lsn.shard_range(small.M, 2, 0)
    share = _run_shard(small, b, e, small.M)
    local = _run_shard(small, b, e, 0)
    for g, h in zip(share["grads"], local["grads"]):
        assert _fro(h, g * (small.M / (e - b))) <= 1e-6


class _FakeDist:
    """A stand-in for torch.distributed in one process: rank 0 of `world`, whose peers'
    gradients for each layer were computed beforehand (peers[l] = [rank 1, rank 2, ...])."""

    def __init__(self, world, grads, peers):
        self.world, self.peers = world, peers
        self.layer_of = {g.data_ptr(): l for l, g in enumerate(grads)}
        self.gathers = []

    def get_world_size(self, group=None):
        return self.world

    def all_gather_into_tensor(self, out, t, group=None):
        l = self.layer_of[t.data_ptr()]
        self.gathers.append(l)
        n = t.numel()
        out[:n].copy_(t)
        for r, g in enumerate(self.peers[l], start=1):
            out[r * n:(r + 1) * n].copy_(g)


def test_data_parallel_exchange_gives_every_rank_the_summed_bits(small):
    lsn = _lsn()
    d, M, world = small.desc, small.M, 2
    b1, e1 = lsn.shard_range(M, world, 1)
    peer = _run_shard(small, b1, e1, M)
    b0, e0 = lsn.shard_range(M, world, 0)
    lone = _run_shard(small, b0, e0, M)
    want = []
    for l in range(d.n_layers):
        w = torch.empty(d.lora_elems, dtype=torch.float32, device="cuda")
        lsn.sum_ranks(torch.cat([lone["grads"][l], peer["grads"][l]]), world, w)
        want.append(w)
    torch.cuda.synchronize()

    x0 = small.x0[b0:e0].contiguous()
    grads = [torch.full((d.lora_elems,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(d.n_layers)]
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(d.workspace_bytes(e0 - b0), dtype=torch.uint8, device="cuda")
    compute = torch.cuda.Stream()
    fake = _FakeDist(world, grads, [[g] for g in peer["grads"]])
    dp = lsn.DataParallel(fake, d, grads, compute)
    pool = small.pool()
    lsn.layer_stack_step(d, x0, small.lora, grads, loss, ws, pool=pool, stream=compute, token_count=M,
                         grads_ready=dp.hook)
    dp.finish()
    torch.cuda.synchronize()
    assert lsn.device_check() == 0
    pool.close()
    assert fake.gathers == list(range(d.n_layers - 1, -1, -1))
    for l in range(d.n_layers):
        assert torch.equal(grads[l].view(torch.int32), want[l].view(torch.int32)), l
