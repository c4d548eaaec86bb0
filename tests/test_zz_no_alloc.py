"""The allocation-free forward entry point, lora_nf4_fwd_static_scratch.

Some callers of this library may not allocate device memory: a plug-in that runs inside a
framework which owns all device memory and forbids its plug-ins to call cudaMalloc, or a
serving path that must never enter the driver's allocator.  They cannot hand lora_nf4_fwd
the split-K workspace it wants, so the library offers a variant whose scratch is a static
16 MiB device buffer.  These tests call that variant through the C ABI twice in a row and
check each result against lora_nf4_fwd (identical bits, and within the forward tolerance),
and check that a shape needing more scratch than the static buffer holds is refused.

This file is collected last so that a run stopping at the first failure has already run
everything else; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FWD_TOL = 2e-2


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _max_rel(got, ref):
    g, r = got.double(), ref.double()
    return float((g - r).abs().max() / r.abs().max())


def _inputs(M, N, K, r, seed):
    from synth import random_bf16
    rng = np.random.default_rng(seed)
    W = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    return (W, _bf16(random_bf16((M, K), seed + 1)), _bf16(random_bf16((r, K), seed + 2, std=K ** -0.5)),
            _bf16(random_bf16((N, r), seed + 3, std=0.01)), _bf16(random_bf16((M, N), seed + 4)))


# shapes whose forward the library splits over K (so the static scratch is really used) and
# whose fp32 partial sums still fit in the 16 MiB buffer
@pytest.mark.parametrize("M,N,K,r,residual", [(128, 1024, 16384, 8, False), (200, 2048, 8192, 8, True)])
def test_static_scratch_matches_workspace_entry_point(M, N, K, r, residual):
    import layer_streamed_nf4_quant_b300 as lsn
    plan = lsn.lora_fwd_plan(M, N, K, r)
    assert plan["y_splits"] > 1 and plan["t_splits"] > 1
    assert 0 < plan["y_partial_bytes"] <= 16 << 20 and plan["t_partial_bytes"] <= 16 << 20
    W, X, A, B, R = _inputs(M, N, K, r, seed=M + N)
    packed = torch.from_numpy(lsn.nf4_pack(W)).cuda()
    res = R if residual else None
    scale = 16.0 / r
    Y_ref, T_ref = lsn.lora_nf4_fwd(packed, N, K, X, A, B, r, scale, residual=res)
    for call in range(2):                       # two calls in a row share the static scratch
        Y, T = lsn.lora_nf4_fwd_static_scratch(packed, N, K, X, A, B, r, scale, residual=res,
                                               sync_status=(call == 1))
        torch.cuda.synchronize()
        assert _max_rel(Y, Y_ref) <= FWD_TOL and _max_rel(T, T_ref) <= FWD_TOL
        assert torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16))
        assert torch.equal(T.view(torch.int16), T_ref.view(torch.int16))


def test_static_scratch_refuses_shapes_beyond_its_buffer():
    import layer_streamed_nf4_quant_b300 as lsn
    M, N, K, r = 300, 4096, 16384, 8
    assert lsn.lora_fwd_plan(M, N, K, r)["y_partial_bytes"] > 16 << 20   # 4 splits x 300 x 4096 x 4 B
    W, X, A, B, _ = _inputs(M, N, K, r, seed=1)
    packed = torch.from_numpy(lsn.nf4_pack(W)).cuda()
    with pytest.raises(lsn.LsnError) as e:
        lsn.lora_nf4_fwd_static_scratch(packed, N, K, X, A, B, r, 2.0)
    assert e.value.code == lsn.LSN_ENOMEM
    assert "static" in str(e.value)
