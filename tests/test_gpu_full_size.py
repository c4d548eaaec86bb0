"""GPU parity at the full token count of the 8 x 2048-token workload (M = 16384), one layer:

* sampled rows: the layer stack is row-independent apart from the normalisation of its
  means, so x_1 and dx0 on 256 sampled rows are compared with the oracle run on those rows
  alone (the oracle divides its means by the full M);
* the LoRA gradients of all 16384 rows against the oracle: the oracle runs the rows in
  eight 2048-row chunks, each with its means taken over the full M, and adds the chunks'
  dA, dB in fp64 -- by linearity of the gradient in the per-row loss terms that sum is the
  full batch's gradient (about two minutes of fp64 CPU work);
* additivity over rows on the GPU: the gradients of the full run equal the sum of the
  gradients of 64 runs over disjoint 256-row slices, each scaled by 256 / M, and the loss
  equals the mean of the slice losses.

The launch configuration (tiles, splits, raster) is the one the 16384-token bench uses.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from test_gpu_stack import FWD_TOL, GRAD_TOL, Stack, _bits, _grad_views, _oracle  # noqa: E402

M_FULL = 16384
SLICE = 256


def _lsn():
    import layer_streamed_nf4_quant_b300 as lsn
    return lsn


@pytest.fixture(scope="module")
def full():
    lsn = _lsn()
    st = Stack(lsn.StackDesc(n_layers=1), M=M_FULL)
    return st, st.run()


def test_decoded_weight_backward_matches_nf4_operands(full):
    """At 16384 tokens, the backward with each layer's W decoded to bf16 first (bwd_weights = 2)
    gives the bits of the default run, whose GEMMs decode NF4 themselves."""
    st, out = full
    nf4 = st.run(bwd_weights=2)
    assert torch.equal(out["dx0"].view(torch.int32), nf4["dx0"].view(torch.int32))
    assert torch.equal(out["grads"][0].view(torch.int32), nf4["grads"][0].view(torch.int32))
    assert torch.equal(out["loss"].view(torch.int32), nf4["loss"].view(torch.int32))


def test_sampled_rows_match_oracle(full):
    from oracle.nf4 import bf16_value
    st, out = full
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, SLICE - 1, SLICE, M_FULL // 2, M_FULL - 1],
                                     rng.choice(M_FULL, SLICE - 6, replace=False)]))
    ref = _oracle(st, rows)
    x = bf16_value(_bits(out["x"])[rows]).astype(np.float64)
    assert np.max(np.abs(x - ref["x_last"])) / np.max(np.abs(ref["x_last"])) <= FWD_TOL
    dx0 = out["dx0"].double().cpu().numpy()[rows]
    assert np.linalg.norm(dx0 - ref["dx0"]) / np.linalg.norm(ref["dx0"]) <= GRAD_TOL


def test_full_batch_gradients_match_oracle(full):
    import synth
    from oracle import nf4 as onf4
    from oracle import stack as ostack
    from oracle.nf4 import bf16_value
    st, out = full
    d = st.desc
    W = synth.layer_weights(0, d.d_model, d.d_kv, d.d_ff)
    A, B = synth.layer_lora(0, d.rank, d.d_model, d.d_kv, d.d_ff)
    layers = [({p: onf4.dequantize(onf4.quantize(W[p])) for p in W},
               {p: bf16_value(A[p]).astype(np.float64) for p in A},
               {p: bf16_value(B[p]).astype(np.float64) for p in B})]
    del W
    x0 = bf16_value(st.x0_bits).astype(np.float64)
    chunk = 2048
    dA = dB = None
    for c0 in range(0, M_FULL, chunk):
        ref = ostack.stack_forward_backward(x0[c0:c0 + chunk], layers, d.scale, token_count=M_FULL)
        if dA is None:
            dA, dB = ref["dA"][0], ref["dB"][0]
        else:
            dA = {p: dA[p] + ref["dA"][0][p] for p in dA}
            dB = {p: dB[p] + ref["dB"][0][p] for p in dB}
        del ref
    gA, gB = _grad_views(st, out["grads"][0])
    for p in gA:
        for got, want in ((gA[p], dA[p]), (gB[p], dB[p])):
            assert np.all(np.isfinite(got))
            assert np.linalg.norm(got - want) / np.linalg.norm(want) <= GRAD_TOL, p


def test_gradients_add_up_over_row_slices(full):
    lsn = _lsn()
    st, out = full
    d = st.desc
    ws = torch.empty(d.workspace_bytes(SLICE), dtype=torch.uint8, device="cuda")
    g_sum = torch.zeros(d.lora_elems, dtype=torch.float64, device="cuda")
    losses = []
    dx0_slices = []
    for j in range(M_FULL // SLICE):
        x0 = st.x0[j * SLICE:(j + 1) * SLICE].contiguous()
        g = [torch.empty(d.lora_elems, dtype=torch.float32, device="cuda")]
        loss = torch.zeros(1, dtype=torch.float32, device="cuda")
        dx0 = torch.empty((SLICE, d.d_model), dtype=torch.float32, device="cuda")
        lsn.layer_stack_step(d, x0, st.lora, g, loss, ws, resident_store=st.resident, dx0=dx0)
        torch.cuda.synchronize()
        g_sum += g[0].double()
        losses.append(loss.item())
        if j in (0, M_FULL // SLICE - 1):
            dx0_slices.append((j, dx0.double()))
    assert lsn.device_check() == 0
    scale = SLICE / M_FULL
    full_g = out["grads"][0].double()
    want = (g_sum * scale)
    gA, gB = _grad_views(st, full_g)
    wA, wB = _grad_views(st, want.float())
    for p in gA:
        for got, ref in ((gA[p], wA[p]), (gB[p], wB[p])):
            assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= GRAD_TOL, p
    assert abs(out["loss"].item() - np.mean(losses)) / out["loss"].item() <= 1e-4
    # dx0 rows: the slice's seed gradient is M / SLICE (a power of two) times the full one
    full_dx0 = out["dx0"].double()
    for j, dxs in dx0_slices:
        got = full_dx0[j * SLICE:(j + 1) * SLICE]
        ref = dxs * scale
        assert (torch.linalg.norm(got - ref) / torch.linalg.norm(ref)).item() <= GRAD_TOL
