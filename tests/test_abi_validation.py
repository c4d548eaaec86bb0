"""CPU-only checks of the C ABI's argument validation: calls with bad shapes, ranks,
alignments or workspaces are refused with the documented status before any device work,
and every refusal leaves a message in lsn_last_error().  The pointers are never
dereferenced, so fake (aligned or misaligned) addresses serve."""
import ctypes as C

import pytest

import layer_streamed_nf4_quant_b300 as lsn
from layer_streamed_nf4_quant_b300._lib import nf4_view

ALIGNED = 0x10000      # never dereferenced: validation fails before any device work
MISALIGNED = 0x10008


def _view(n_out, k_in, base=ALIGNED):
    return nf4_view(C.c_void_p(base), n_out, k_in)


def _fwd(view, M=64, r=8, X=ALIGNED, A=ALIGNED, B=ALIGNED, Y=ALIGNED, T=ALIGNED, ws=ALIGNED, ws_bytes=1 << 30):
    P = C.c_void_p
    return lsn.lib.lora_nf4_fwd(C.byref(view), P(X), M, P(A), P(B), r, 2.0, None, P(Y), P(T), P(ws), ws_bytes, None)


def _bwd(view, M=64, r=8, dX=ALIGNED, ws=ALIGNED, ws_bytes=1 << 30):
    P = C.c_void_p
    return lsn.lib.lora_nf4_bwd(C.byref(view), P(ALIGNED), P(ALIGNED), P(ALIGNED), M, P(ALIGNED), P(ALIGNED), r, 2.0,
                                P(dX), 0, P(ALIGNED), P(ALIGNED), P(ws), ws_bytes, None)


def _msg():
    return lsn.lib.lsn_last_error().decode()


@pytest.mark.parametrize("n_out,k_in,r,M", [
    (128, 100, 8, 64),      # k_in not a multiple of 64
    (100, 128, 8, 64),      # n_out not a multiple of 8
    (128, 128, 4, 64),      # r below 8
    (128, 128, 12, 64),     # r not a multiple of 8
    (128, 128, 72, 64),     # r above 64
    (128, 128, 8, 0),       # no rows
])
def test_bad_shapes_are_refused(n_out, k_in, r, M):
    assert _fwd(_view(n_out, k_in), M=M, r=r) == lsn.LSN_EINVAL
    assert _msg()
    assert _bwd(_view(n_out, k_in), M=M, r=r) == lsn.LSN_EINVAL


def test_misaligned_pointers_are_refused():
    assert _fwd(_view(128, 128, base=MISALIGNED)) == lsn.LSN_EINVAL
    assert "aligned" in _msg()
    assert _fwd(_view(128, 128), X=MISALIGNED) == lsn.LSN_EINVAL
    assert _fwd(_view(128, 128), Y=MISALIGNED) == lsn.LSN_EINVAL
    assert _bwd(_view(128, 128), dX=MISALIGNED) == lsn.LSN_EINVAL


def test_null_arguments_are_refused():
    P = C.c_void_p
    v = _view(128, 128)
    assert lsn.lib.lora_nf4_fwd(None, P(ALIGNED), 64, P(ALIGNED), P(ALIGNED), 8, 2.0, None, P(ALIGNED), P(ALIGNED),
                                P(ALIGNED), 1 << 20, None) == lsn.LSN_EINVAL
    assert _fwd(v, Y=0) == lsn.LSN_EINVAL
    assert lsn.lib.nf4_dequant(None, P(ALIGNED), None) == lsn.LSN_EINVAL


def test_small_workspace_is_refused_with_enomem():
    # a shape whose forward needs split-K partials: the workspace query says how much
    M, n_out, k_in, r = 256, 256, 8192, 64
    need = lsn.lib.lora_nf4_workspace_bytes(M, n_out, k_in, r)
    assert need > 256
    assert _bwd(_view(n_out, k_in), M=M, r=r, ws_bytes=64) == lsn.LSN_ENOMEM
    assert "workspace" in _msg()


def test_workspace_query_rejects_bad_shapes():
    assert lsn.lib.lora_nf4_workspace_bytes(0, 128, 128, 8) == 0
    assert lsn.lib.lora_nf4_workspace_bytes(64, 128, 32, 8) == 0
    assert lsn.lib.lora_nf4_workspace_bytes(64, 128, 128, 4) == 0
    assert lsn.lib.lora_nf4_workspace_bytes(64, 128, 128, 8) > 0


def _fwd_static(view, M=64, r=8, X=ALIGNED, A=ALIGNED, B=ALIGNED, Y=ALIGNED, T=ALIGNED, residual=None):
    P = C.c_void_p
    return lsn.lib.lora_nf4_fwd_static_scratch(C.byref(view), P(X), M, P(A), P(B), r, 2.0,
                                               None if residual is None else P(residual), P(Y), P(T), None, None)


def test_static_scratch_checks_alignment_like_the_workspace_entry():
    """The allocation-free forward refuses every misaligned operand or output that
    lora_nf4_fwd refuses, instead of handing it to a kernel that stores 16-byte vectors."""
    v = _view(128, 128)
    for kw in ({"residual": MISALIGNED}, {"Y": MISALIGNED}, {"T": MISALIGNED}, {"X": MISALIGNED},
               {"A": MISALIGNED}, {"B": MISALIGNED}):
        assert _fwd_static(v, **kw) == lsn.LSN_EINVAL, kw
        assert "aligned" in _msg()
    assert _fwd_static(_view(128, 128, base=MISALIGNED)) == lsn.LSN_EINVAL
    assert _fwd_static(v, T=0) == lsn.LSN_EINVAL          # no adapter-disabled mode here
    assert "NULL" in _msg()


def test_adapter_disabled_forward_validation():
    """lora_nf4_fwd with A = B = NULL is the frozen linear: T may be NULL then, but a
    half-given adapter (only A or only B) is refused."""
    v = _view(128, 128)
    assert _fwd(v, A=0, B=ALIGNED) == lsn.LSN_EINVAL
    assert _fwd(v, A=ALIGNED, B=0) == lsn.LSN_EINVAL
    assert _fwd(v, A=0, B=0, T=0, X=MISALIGNED) == lsn.LSN_EINVAL   # still validated
    assert "aligned" in _msg()


def test_split_planner_choices_are_consistent():
    """The launch planner's split counts (host only): large problems are not split, deep
    skinny ones are, the counts stay within 1..32, repeated queries agree, and the workspace
    query covers the partial sums of both forward launches."""
    big = lsn.lora_fwd_plan(16384, 14336, 4096, 64)
    assert big["y_splits"] == 1 and big["y_partial_bytes"] == 0
    deep = lsn.lora_fwd_plan(128, 1024, 16384, 8)
    assert 1 < deep["y_splits"] <= 32 and 1 < deep["t_splits"] <= 32
    assert deep["y_partial_bytes"] == deep["y_splits"] * 128 * 1024 * 4
    assert lsn.lora_fwd_plan(128, 1024, 16384, 8) == deep
    need = lsn.lib.lora_nf4_workspace_bytes(128, 1024, 16384, 8)
    assert need >= deep["t_partial_bytes"] + deep["y_partial_bytes"]
    with pytest.raises(lsn.LsnError):
        lsn.lora_fwd_plan(128, 1024, 100, 8)


def _step_ex(opts, M=64, L=2):
    P = C.c_void_p
    desc = lsn.StackDesc(n_layers=L, d_model=256, d_kv=256, d_ff=512, rank=8)
    lora = (P * L)(*[ALIGNED] * L)
    grads = (P * L)(*[ALIGNED] * L)
    return lsn.lib.layer_stack_step_ex(None, P(ALIGNED), C.byref(desc.c), C.byref(opts), P(ALIGNED), M, lora, grads,
                                       P(ALIGNED), None, None, None, P(0x100000), 1 << 40, None)


def test_data_parallel_step_options_are_validated():
    from layer_streamed_nf4_quant_b300._lib import lsn_step_opts, lsn_layer_hook, lsn_adamw_state
    for tc in (-1, 63):                        # negative, or fewer tokens than this rank holds
        o = lsn_step_opts(0, 0)
        o.token_count = tc
        assert _step_ex(o) == lsn.LSN_EINVAL
        assert "token_count" in _msg()
    hook = lsn_layer_hook(lambda *a: None)
    st = lsn_adamw_state()
    o = lsn_step_opts(0, 0)
    o.grads_ready = hook
    o.adamw = C.pointer(st)
    assert _step_ex(o) == lsn.LSN_EINVAL
    assert "hook" in _msg()


def test_backward_weight_mode_is_validated_and_sized():
    from layer_streamed_nf4_quant_b300._lib import lsn_step_opts
    for bad in (-1, 3):
        o = lsn_step_opts(0, 0)
        o.bwd_weights = bad
        assert _step_ex(o) == lsn.LSN_EINVAL
        assert "bwd_weights" in _msg()
    d = lsn.StackDesc(n_layers=2, d_model=256, d_kv=256, d_ff=512, rank=8)
    nf4, dense = d.workspace_bytes(64, bwd_weights=1), d.workspace_bytes(64, bwd_weights=2)
    # the bf16 scratch holds the larger of [W_o, W_down] and [W_q .. W_up]
    assert dense - nf4 >= 2 * 256 * (256 + 256 + 256 + 512 + 512)
    assert d.workspace_bytes(64) == nf4                    # default: NF4 operands, no bf16 W
    assert d.workspace_bytes(8192) == d.workspace_bytes(8192, bwd_weights=1)


def test_sum_ranks_arguments_are_validated():
    P = C.c_void_p
    s = lsn.lib.lsn_sum_ranks
    assert s(None, 2, 64, P(ALIGNED), None) == lsn.LSN_EINVAL
    assert s(P(ALIGNED), 2, 64, None, None) == lsn.LSN_EINVAL
    assert s(P(ALIGNED), 0, 64, P(0x20000), None) == lsn.LSN_EINVAL
    assert s(P(MISALIGNED), 2, 64, P(0x20000), None) == lsn.LSN_EINVAL
    assert s(P(ALIGNED), 2, 64, P(MISALIGNED), None) == lsn.LSN_EINVAL
    # out may be in[0] but no other part of the gathered array
    assert s(P(ALIGNED), 2, 64, P(ALIGNED + 64 * 4), None) == lsn.LSN_EINVAL
    assert "overlaps" in _msg()
