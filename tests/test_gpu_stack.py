"""GPU tests of layer_stack_step: oracle parity of the small and full-size layer, and the
streamed run bit-identical to the resident run (plus replay, slot parity, copy delays)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FWD_TOL = 2e-2
GRAD_TOL = 1e-2


def _lsn():
    import layer_streamed_nf4_quant_b300 as lsn
    return lsn


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


class Stack:
    """A stack on the device: pinned store, resident copy, LoRA blobs, input, workspace."""

    def __init__(self, desc, M, x_rows_seed=1):
        import synth
        from layer_streamed_nf4_quant_b300 import workload
        self.desc = desc
        self.M = M
        self.store = workload.build_store(desc)
        self.resident = self.store.cuda()
        self.lora = [workload.lora_blob(desc, l) for l in range(desc.n_layers)]
        self.x0_bits = synth.stack_input(M, desc.d_model, seed=x_rows_seed)
        self.x0 = workload.bf16_tensor(self.x0_bits)
        self.ws = torch.empty(desc.workspace_bytes(M), dtype=torch.uint8, device="cuda")
        self.slots = [torch.empty(desc.image_bytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
        self.copy_stream = torch.cuda.Stream()

    def pool(self, first_slot=0, reuse=False, chunked=False):
        lsn = _lsn()
        offs = [l * self.desc.image_bytes for l in range(self.desc.n_layers)]
        pool = lsn.StreamPool(self.store, offs, self.desc.image_bytes, self.slots[0], self.slots[1],
                              self.copy_stream, first_slot=first_slot, reuse_resident=reuse)
        if chunked:
            pool.set_chunks(self.desc.chunk_offsets())
        return pool

    def run(self, pool=None, recompute=False, reference=False, bwd_weights=0):
        lsn = _lsn()
        d = self.desc
        grads = [torch.full((d.lora_elems,), float("nan"), dtype=torch.float32, device="cuda")
                 for _ in range(d.n_layers)]
        loss = torch.zeros(1, dtype=torch.float32, device="cuda")
        x_out = torch.empty((self.M, d.d_model), dtype=torch.bfloat16, device="cuda")
        dx0 = torch.empty((self.M, d.d_model), dtype=torch.float32, device="cuda")
        x_ref = torch.empty((self.M, d.d_model), dtype=torch.bfloat16, device="cuda") if reference else None
        ws = self.ws
        if recompute or reference or bwd_weights:
            ws = torch.empty(d.workspace_bytes(self.M, recompute, reference, bwd_weights), dtype=torch.uint8,
                             device="cuda")
        lsn.layer_stack_step(d, self.x0, self.lora, grads, loss, ws, pool=pool,
                             resident_store=None if pool else self.resident, x_out=x_out, dx0=dx0,
                             recompute=recompute, reference_pass=reference, x_ref_out=x_ref,
                             bwd_weights=bwd_weights)
        torch.cuda.synchronize()
        assert lsn.device_check() == 0
        return {"loss": loss, "x": x_out, "dx0": dx0, "grads": grads, "x_ref": x_ref}


def _same(a, b):
    assert torch.equal(a["loss"].view(torch.int32), b["loss"].view(torch.int32))
    assert torch.equal(a["x"].view(torch.int16), b["x"].view(torch.int16))
    assert torch.equal(a["dx0"].view(torch.int32), b["dx0"].view(torch.int32))
    for g, h in zip(a["grads"], b["grads"]):
        assert torch.equal(g.view(torch.int32), h.view(torch.int32))


def _oracle(st, rows=None):
    """Oracle of the whole stack (on a token slice when `rows` is given)."""
    import synth
    from oracle import nf4 as onf4
    from oracle import stack as ostack
    from oracle.nf4 import bf16_value
    d = st.desc
    layers = []
    for l in range(d.n_layers):
        W = synth.layer_weights(l, d.d_model, d.d_kv, d.d_ff)
        A, B = synth.layer_lora(l, d.rank, d.d_model, d.d_kv, d.d_ff)
        Wh = {p: onf4.dequantize(onf4.quantize(W[p])) for p in W}
        Af = {p: bf16_value(A[p]).astype(np.float64) for p in A}
        Bf = {p: bf16_value(B[p]).astype(np.float64) for p in B}
        layers.append((Wh, Af, Bf))
    x0 = bf16_value(st.x0_bits).astype(np.float64)
    if rows is not None:
        x0 = x0[rows]
    return ostack.stack_forward_backward(x0, layers, d.scale, token_count=st.M)


def _grad_views(st, g):
    A, B = st.desc.lora_views(g)
    return {k: v.double().cpu().numpy() for k, v in A.items()}, {k: v.double().cpu().numpy() for k, v in B.items()}


@pytest.fixture(scope="module")
def small():
    lsn = _lsn()
    desc = lsn.StackDesc(n_layers=3, d_model=256, d_kv=256, d_ff=512, rank=16)
    return Stack(desc, M=300)


def test_small_stack_oracle_parity(small):
    from oracle.nf4 import bf16_value
    out = small.run()
    ref = _oracle(small)
    assert abs(out["loss"].item() - ref["loss"]) / ref["loss"] <= FWD_TOL
    x = bf16_value(_bits(out["x"])).astype(np.float64)
    assert np.max(np.abs(x - ref["x_last"])) / np.max(np.abs(ref["x_last"])) <= FWD_TOL
    for l in range(small.desc.n_layers):
        gA, gB = _grad_views(small, out["grads"][l])
        for p in gA:
            for got, want in ((gA[p], ref["dA"][l][p]), (gB[p], ref["dB"][l][p])):
                assert np.all(np.isfinite(got)) and np.any(got != 0)
                assert np.linalg.norm(got - want) / np.linalg.norm(want) <= GRAD_TOL, (l, p)
    dx0 = out["dx0"].double().cpu().numpy()
    assert np.linalg.norm(dx0 - ref["dx0"]) / np.linalg.norm(ref["dx0"]) <= GRAD_TOL


def test_small_streamed_bit_identical_to_resident(small):
    res = small.run()
    pool = small.pool()
    st = small.run(pool)
    _same(res, st)
    stats = pool.stats()
    assert stats["copies"] == 2 * small.desc.n_layers
    assert stats["bytes_copied"] == 2 * small.desc.n_layers * small.desc.image_bytes
    pool.close()


def test_small_replay_slot_parity_and_delays(small):
    base = small.run()
    _same(base, small.run())                                  # deterministic replay
    pool = small.pool(first_slot=1)                           # start in the other slot
    _same(base, small.run(pool))
    pool.set_copy_delay_us(3000)                              # late copies change nothing
    _same(base, small.run(pool))
    pool.close()
    pool = small.pool(reuse=True)                             # skip the turnaround re-copies
    _same(base, small.run(pool))
    assert pool.stats()["skipped"] == 2
    pool.close()


def test_decoded_weight_backward_bit_identical(small):
    """bwd_weights = 2 decodes each layer's W to bf16 scratch and runs the backward's
    transposed GEMMs on the dense copy; the decode gives the producers' values bit for bit, so
    the step's results equal the NF4-operand run's, resident and streamed."""
    base = small.run(bwd_weights=1)
    _same(base, small.run(bwd_weights=2))
    pool = small.pool()
    _same(base, small.run(pool, bwd_weights=2))
    pool.close()
    _same(base, small.run(recompute=True, bwd_weights=2))


def test_recompute_bit_identical_to_stored_activations(small):
    """The checkpointed backward (only x_l kept, each layer recomputed from its re-streamed
    weights) gives the stored-activation run's bits, resident and streamed."""
    base = small.run()
    _same(base, small.run(recompute=True))
    pool = small.pool()
    _same(base, small.run(pool, recompute=True))
    assert pool.stats()["copies"] == 2 * small.desc.n_layers
    pool.close()


def test_reference_pass_shares_the_stream(small):
    """Preference-pair reuse: the adapter-disabled forward runs on the same streamed slots.
    It matches the oracle's frozen-base forward, leaves the policy branch's bits unchanged,
    and copies no layer more often than the plain step (bytes streamed per step x1.0)."""
    from oracle import nf4 as onf4
    from oracle import stack as ostack
    from oracle.nf4 import bf16_value
    import synth
    base = small.run()
    pool = small.pool()
    out = small.run(pool, reference=True)
    _same(base, out)
    stats = pool.stats()
    assert stats["copies"] == 2 * small.desc.n_layers
    assert stats["bytes_copied"] == 2 * small.desc.n_layers * small.desc.image_bytes
    pool.close()
    d = small.desc
    Ws = []
    for l in range(d.n_layers):
        W = synth.layer_weights(l, d.d_model, d.d_kv, d.d_ff)
        Ws.append({p: onf4.dequantize(onf4.quantize(W[p])) for p in W})
    ref = ostack.frozen_stack_forward(bf16_value(small.x0_bits).astype(np.float64), Ws)
    got = bf16_value(_bits(out["x_ref"])).astype(np.float64)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= FWD_TOL
    x_pol = bf16_value(_bits(out["x"])).astype(np.float64)
    assert np.max(np.abs(got - x_pol)) > 0                   # the adapter does change the output


def test_zero_B_stack_bit_identical_to_reference_pass(small):
    """B = 0 in every layer: the policy stack is the frozen stack, so its output must equal
    the adapter-disabled reference pass (LoRA steps left out of the GEMMs) bit for bit."""
    lsn = _lsn()
    d = small.desc
    saved = small.lora
    try:
        zeroed = []
        for blob in saved:
            z = blob.clone()
            _, B = d.lora_views(z)
            for p in B:
                B[p].zero_()
            zeroed.append(z)
        small.lora = zeroed
        out = small.run(reference=True)
    finally:
        small.lora = saved
    assert torch.equal(out["x"].view(torch.int16), out["x_ref"].view(torch.int16))


def test_host_wait_timeout_then_recovery(small):
    """stream_pool_wait with a host timeout: a copy held back by the injected delay makes the
    bounded poll return LSN_ETIMEOUT; once the copy lands the pool goes on, and a full step
    through it still gives the resident bits."""
    lsn = _lsn()
    base = small.run()
    pool = small.pool()
    pool.set_copy_delay_us(300000)
    pool.prefetch(0)
    with pytest.raises(lsn.LsnError) as e:
        pool.wait(0, timeout_ms=5)
    assert e.value.code == lsn.LSN_ETIMEOUT
    torch.cuda.synchronize()
    pool.stats()                                              # the delayed copy has landed
    pool.release(0)
    pool.set_copy_delay_us(0)
    _same(base, small.run(pool))
    pool.close()


def test_chunked_stream_bit_identical_to_resident(small):
    """Sub-layer streaming: each layer copied as [header, q..up] and [o, down], ascending in
    the forward sweep and descending in the reverse one, each GEMM group waiting only for its
    own chunk.  Same bits as the resident run, plain, recomputed and with the reference pass;
    every chunk of every layer copied once per sweep."""
    d = small.desc
    base = small.run()
    pool = small.pool(chunked=True)
    _same(base, small.run(pool))
    st = pool.stats()
    assert st["copies"] == 2 * d.n_layers and st["bytes_copied"] == 2 * d.n_layers * d.image_bytes
    c0, c1 = pool.chunk_stats(0), pool.chunk_stats(1)
    assert c0["copies"] == c1["copies"] == 2 * d.n_layers
    assert c0["bytes_copied"] == 2 * d.n_layers * d.chunk_offsets()[1]
    assert c0["bytes_copied"] + c1["bytes_copied"] == st["bytes_copied"]
    _same(base, small.run(pool, recompute=True))
    _same(base, small.run(pool, reference=True))
    pool.set_copy_delay_us(2000)                              # late chunks change nothing
    _same(base, small.run(pool))
    pool.close()
    pool = small.pool(first_slot=1, reuse=True, chunked=True)
    _same(base, small.run(pool))
    pool.close()


def test_chunk_validation_and_range_waits(small):
    lsn = _lsn()
    d = small.desc
    pool = small.pool()
    o = d.chunk_offsets()[1]
    for bad in ([0, o + 1], [0, 0], [0, d.image_bytes], [256, o], [0, o, o]):
        with pytest.raises(lsn.LsnError) as e:
            pool.set_chunks(bad)
        assert e.value.code == lsn.LSN_EINVAL
    pool.set_chunks([0, o])
    pool.prefetch(0, reverse=True)
    with pytest.raises(lsn.LsnError) as e:
        pool.set_chunks([0])                                  # a slot holds layer 0
    assert e.value.code == lsn.LSN_ESTATE
    with pytest.raises(lsn.LsnError) as e:
        pool.wait_range(0, o, o)                              # empty range
    assert e.value.code == lsn.LSN_EINVAL
    a = pool.wait_range(0, o, d.image_bytes)                  # the chunk copied first
    b = pool.wait_range(0, 0, 64)                             # the header, copied second
    assert a == b
    torch.cuda.synchronize()
    img = torch.empty(d.image_bytes, dtype=torch.uint8, device="cuda")
    img.copy_(small.slots[0])
    assert torch.equal(img.cpu(), small.store[:d.image_bytes])
    pool.release(0)
    pool.set_chunks([0])                                      # back to whole-layer copies
    pool.close()


def test_pool_misuse_is_reported(small):
    lsn = _lsn()
    pool = small.pool()
    pool.prefetch(0)
    pool.prefetch(1)
    with pytest.raises(lsn.LsnError) as e:
        pool.prefetch(2)                                      # slot of layer 0 not released
    assert e.value.code == lsn.LSN_ESTATE
    with pytest.raises(lsn.LsnError) as e:
        pool.wait(2)
    assert e.value.code == lsn.LSN_ESTATE
    pool.wait(0)
    pool.release(0)
    pool.prefetch(2)
    pool.wait(1)
    pool.release(1)
    pool.wait(2)
    pool.release(2)
    pool.close()
    with pytest.raises(lsn.LsnError) as e:
        lsn.StreamPool(small.store.clone(), [0], small.desc.image_bytes, small.slots[0], small.slots[1],
                       small.copy_stream)                     # clone() is not page-locked
    assert e.value.code == lsn.LSN_EINVAL


def test_layer_tag_mismatch_reported(small):
    lsn = _lsn()
    d = small.desc
    bad = small.resident.clone()
    bad[4:8] = torch.tensor([9, 0, 0, 0], dtype=torch.uint8)  # layer 0 image claims to be layer 9
    grads = [torch.empty(d.lora_elems, dtype=torch.float32, device="cuda") for _ in range(d.n_layers)]
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    lsn.layer_stack_step(d, small.x0, small.lora, grads, loss, small.ws, resident_store=bad)
    with pytest.raises(lsn.LsnError) as e:
        lsn.device_check()
    assert e.value.code == lsn.LSN_ECORRUPT
    assert lsn.device_check() == 0                            # the word was cleared


def test_full_layer_oracle_parity():
    """One Llama-3.1-8B-shaped layer at M = 512 (r = 64, alpha = 16) against the oracle."""
    from oracle.nf4 import bf16_value
    lsn = _lsn()
    desc = lsn.StackDesc(n_layers=1)
    st = Stack(desc, M=512)
    out = st.run()
    ref = _oracle(st)
    x = bf16_value(_bits(out["x"])).astype(np.float64)
    assert np.max(np.abs(x - ref["x_last"])) / np.max(np.abs(ref["x_last"])) <= FWD_TOL
    assert abs(out["loss"].item() - ref["loss"]) / ref["loss"] <= FWD_TOL
    dx0 = out["dx0"].double().cpu().numpy()
    assert np.linalg.norm(dx0 - ref["dx0"]) / np.linalg.norm(ref["dx0"]) <= GRAD_TOL
    gA, gB = _grad_views(st, out["grads"][0])
    for p in gA:
        for got, want in ((gA[p], ref["dA"][0][p]), (gB[p], ref["dB"][0][p])):
            assert np.linalg.norm(got - want) / np.linalg.norm(want) <= GRAD_TOL, p


def test_full_stack_32_layers_streamed_bit_identical():
    """The 32-layer stack at batch 1 x 512 streamed through the two-slot pool equals the
    resident run bit for bit."""
    lsn = _lsn()
    desc = lsn.StackDesc(n_layers=32)
    st = Stack(desc, M=512)
    res = st.run()
    pool = st.pool()
    streamed = st.run(pool)
    _same(res, streamed)
    assert np.isfinite(res["loss"].item())
    pool.close()
