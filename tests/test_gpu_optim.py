"""GPU tests of the AdamW update on the LoRA factors: the standalone step against the fp64
oracle, the update fused into the reverse sweep against separate updates, and a short
training run streamed vs resident (the pages' practical check: a few steps with streaming on
and off must not diverge -- "Fine-Tune an 8B Model on a 4GB Laptop GPU: Hands-On Guide",
section "The gotchas nobody's mentioning yet")."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _lsn():
    import layer_streamed_nf4_quant_b300 as lsn
    return lsn


def test_adamw_step_matches_oracle():
    from oracle import optim
    lsn = _lsn()
    n = 100_003
    rng = np.random.default_rng(0)
    p = rng.standard_normal(n).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    tp, tm, tv = (torch.from_numpy(a.copy()).cuda() for a in (p, m, v))
    tb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    P, Mo, V = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    for t in range(1, 4):
        g = rng.standard_normal(n).astype(np.float32)
        lsn.adamw_step(tp, torch.from_numpy(g).cuda(), tm, tv, t, lr=1e-2, weight_decay=0.1, p_bf16=tb)
        P, Mo, V = optim.adamw_step(P, g, Mo, V, t, lr=1e-2, wd=0.1)
    torch.cuda.synchronize()
    # fp32 against fp64: each of the few fp32 operations per step adds at most 2^-24
    # relative error, amplified by cancellation in b1 m + (1-b1) g, so three steps stay
    # within 1e-4 relative or 1e-6 absolute (the gradients are O(1))
    np.testing.assert_allclose(tp.cpu().numpy(), P, rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(tm.cpu().numpy(), Mo, rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(tv.cpu().numpy(), V, rtol=1e-4, atol=1e-6)
    assert torch.equal(tb.view(torch.int16), tp.bfloat16().view(torch.int16))


def _clone_lora(st):
    return [b.clone() for b in st.lora]


def test_fused_update_equals_separate_updates():
    from test_gpu_stack import Stack
    lsn = _lsn()
    desc = lsn.StackDesc(n_layers=3, d_model=256, d_kv=256, d_ff=512, rank=16)
    st = Stack(desc, M=200)
    orig = _clone_lora(st)
    # plain step, then one separate AdamW update per layer
    plain = st.run()
    sep = lsn.AdamW(_clone_lora(st), lr=1e-3, weight_decay=0.01)
    for l in range(desc.n_layers):
        lsn.adamw_step(sep.master[l], plain["grads"][l], sep.m[l], sep.v[l], 1, lr=1e-3, weight_decay=0.01,
                       p_bf16=sep.blobs[l])
    # the same update fused into the reverse sweep
    st.lora = [b.clone() for b in orig]
    fused = lsn.AdamW(st.lora, lr=1e-3, weight_decay=0.01)
    grads = [torch.empty(desc.lora_elems, dtype=torch.float32, device="cuda") for _ in range(desc.n_layers)]
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(desc.workspace_bytes(200), dtype=torch.uint8, device="cuda")
    lsn.layer_stack_step(desc, st.x0, st.lora, grads, loss, ws, resident_store=st.resident, adamw=fused)
    torch.cuda.synchronize()
    for l in range(desc.n_layers):
        assert torch.equal(grads[l].view(torch.int32), plain["grads"][l].view(torch.int32))
        assert torch.equal(fused.master[l].view(torch.int32), sep.master[l].view(torch.int32))
        assert torch.equal(st.lora[l].view(torch.int16), sep.blobs[l].view(torch.int16))
        assert not torch.equal(st.lora[l].view(torch.int16), orig[l].view(torch.int16))


def test_training_run_streamed_equals_resident():
    from test_gpu_stack import Stack
    lsn = _lsn()
    desc = lsn.StackDesc(n_layers=2, d_model=256, d_kv=256, d_ff=512, rank=16)
    st = Stack(desc, M=128)
    orig = _clone_lora(st)
    losses = {}
    finals = {}
    for mode in ("resident", "streamed"):
        blobs = [b.clone() for b in orig]
        opt = lsn.AdamW(blobs, lr=1e-2)
        pool = st.pool() if mode == "streamed" else None
        ws = torch.empty(desc.workspace_bytes(128), dtype=torch.uint8, device="cuda")
        grads = [torch.empty(desc.lora_elems, dtype=torch.float32, device="cuda") for _ in range(2)]
        seq = []
        for _ in range(3):
            loss = torch.zeros(1, dtype=torch.float32, device="cuda")
            lsn.layer_stack_step(desc, st.x0, blobs, grads, loss, ws, pool=pool,
                                 resident_store=None if pool else st.resident, adamw=opt)
            torch.cuda.synchronize()
            seq.append(loss.item())
        losses[mode] = seq
        finals[mode] = blobs
        if pool:
            pool.close()
    assert losses["resident"] == losses["streamed"]
    assert losses["resident"][2] < losses["resident"][0]          # the adapters do train
    for a, b in zip(finals["resident"], finals["streamed"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
