"""Layer-streamed NF4-LoRA for B300 (sm_103a): Python binding of liblsn.so.

The functions here marshal torch tensors (device memory, streams) and numpy arrays into the
C ABI declared in ``include/lsn.h``; every step of the computation runs in the library's
CUDA kernels and host code.  Importing this package fails if the library is not built.

bf16 tensors are ``torch.bfloat16``; packed NF4 matrices and layer images are ``torch.uint8``.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from ._lib import (LSN_ECORRUPT, LSN_EINVAL, LSN_ENOMEM, LSN_ESTATE, LSN_ETIMEOUT, LSN_OK,  # noqa: F401
                   LsnError, check, lib, lsn_adamw_hparams, lsn_adamw_state, lsn_layer_hook, lsn_pool_stats,
                   lsn_profile, lsn_stack_desc, lsn_step_opts, nf4_view)

PROJ = ("q", "k", "v", "gate", "up", "o", "down")   # canonical projection order


def _torch():
    import torch
    return torch


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------------------ NF4

def codebook() -> np.ndarray:
    out = (C.c_float * 16)()
    check(lib.lsn_nf4_codebook(out))
    return np.frombuffer(out, dtype=np.float32).copy()


def nf4_packed_bytes(n_out: int, k_in: int) -> int:
    return int(lib.nf4_packed_bytes(n_out, k_in))


def nf4_pack(W: np.ndarray, n_threads: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """Host quantiser: fp32 [n_out x k_in] -> packed bytes (numpy uint8)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    n, k = W.shape
    nbytes = nf4_packed_bytes(n, k)
    if nbytes == 0:
        raise LsnError(LSN_EINVAL, "k_in must be a positive multiple of 64")
    if out is None:
        out = np.empty(nbytes, dtype=np.uint8)
    check(lib.nf4_pack(W.ctypes.data_as(C.c_void_p), n, k, out.ctypes.data_as(C.c_void_p), out.nbytes, n_threads))
    return out


def view(packed, n_out: int, k_in: int) -> nf4_view:
    return nf4_view(C.c_void_p(packed.data_ptr()), n_out, k_in)


def nf4_dequant(packed, n_out: int, k_in: int, out=None, stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty((n_out, k_in), dtype=torch.bfloat16, device=packed.device)
    v = view(packed, n_out, k_in)
    check(lib.nf4_dequant(C.byref(v), _p(out), _stream(stream)))
    return out


# ------------------------------------------------------------------------ LoRA linear

def lora_workspace(M: int, n_out: int, k_in: int, r: int, device="cuda"):
    torch = _torch()
    n = int(lib.lora_nf4_workspace_bytes(M, n_out, k_in, r))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def lora_nf4_fwd(packed, n_out, k_in, X, A, B, r, scale, residual=None, Y=None, T=None, ws=None, stream=None):
    """Y = bf16(X W^T + s T B^T [+ residual]), T = bf16(X A^T).  Returns (Y, T).

    A = B = None disables the adapter: Y = bf16(X W^T [+ residual]) and T is None."""
    torch = _torch()
    M = X.shape[0]
    adapter = A is not None or B is not None
    if Y is None:
        Y = torch.empty((M, n_out), dtype=torch.bfloat16, device=X.device)
    if T is None and adapter:
        T = torch.empty((M, r), dtype=torch.bfloat16, device=X.device)
    if ws is None:
        ws = lora_workspace(M, n_out, k_in, r, X.device)
    v = view(packed, n_out, k_in)
    check(lib.lora_nf4_fwd(C.byref(v), _p(X), M, _p(A), _p(B), r, float(scale), _p(residual), _p(Y), _p(T),
                           _p(ws), ws.numel(), _stream(stream)))
    return Y, T


def lora_fwd_plan(M: int, n_out: int, k_in: int, r: int) -> dict:
    """Split-K counts and partial-sum bytes of lora_nf4_fwd's two launches for this shape."""
    ts, ys, tb, yb = C.c_int(), C.c_int(), C.c_size_t(), C.c_size_t()
    check(lib.lora_nf4_fwd_plan(M, n_out, k_in, r, C.byref(ts), C.byref(ys), C.byref(tb), C.byref(yb)))
    return {"t_splits": ts.value, "y_splits": ys.value, "t_partial_bytes": tb.value, "y_partial_bytes": yb.value}


def lora_nf4_fwd_static_scratch(packed, n_out, k_in, X, A, B, r, scale, residual=None, Y=None, T=None,
                                sync_status=False, stream=None):
    """lora_nf4_fwd without a workspace or any device allocation, for callers that may not
    allocate: the split-K scratch is a 16 MiB static device buffer shared by all calls on a
    device (calls that overlap on the GPU race).  Returns (Y, T)."""
    torch = _torch()
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, n_out), dtype=torch.bfloat16, device=X.device)
    if T is None:
        T = torch.empty((M, r), dtype=torch.bfloat16, device=X.device)
    v = view(packed, n_out, k_in)
    status = C.c_uint32(0)
    check(lib.lora_nf4_fwd_static_scratch(C.byref(v), _p(X), M, _p(A), _p(B), r, float(scale), _p(residual),
                                          _p(Y), _p(T), C.byref(status) if sync_status else None,
                                          _stream(stream)))
    return Y, T


def lora_nf4_bwd(packed, n_out, k_in, X, T, dY, A, B, r, scale, dX=None, accumulate_dX=False, dA=None,
                 dB=None, ws=None, want_dX=True, stream=None):
    """dX (+)= dY W + dT A, dA = dT^T X, dB = s dY^T T with dT = bf16(s dY B).  Returns (dX, dA, dB)."""
    torch = _torch()
    M = X.shape[0]
    dev = X.device
    if want_dX and dX is None:
        dX = torch.empty((M, k_in), dtype=torch.float32, device=dev)
    if dA is None:
        dA = torch.empty((r, k_in), dtype=torch.float32, device=dev)
    if dB is None:
        dB = torch.empty((n_out, r), dtype=torch.float32, device=dev)
    if ws is None:
        ws = lora_workspace(M, n_out, k_in, r, dev)
    v = view(packed, n_out, k_in)
    check(lib.lora_nf4_bwd(C.byref(v), _p(X), _p(T), _p(dY), M, _p(A), _p(B), r, float(scale),
                           _p(dX if want_dX else None), 1 if accumulate_dX else 0, _p(dA), _p(dB), _p(ws),
                           ws.numel(), _stream(stream)))
    return dX, dA, dB


def adamw_step(p, g, m, v, step: int, lr: float, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, p_bf16=None,
               stream=None):
    """One AdamW step on fp32 device tensors p, m, v (in place) with gradient g; writes
    bf16(p) into p_bf16 when given."""
    hp = lsn_adamw_hparams(lr, beta1, beta2, eps, weight_decay, step)
    check(lib.lsn_adamw_step(C.byref(hp), _p(p), _p(p_bf16), _p(g), _p(m), _p(v), p.numel(), _stream(stream)))


def device_check(stream=None) -> int:
    """Synchronises and returns the device error status (raises LsnError on an error)."""
    detail = C.c_uint32(0)
    check(lib.lsn_check(_stream(stream), C.byref(detail)))
    return detail.value


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib.lsn_launch_count())


def profile_enable(on: bool = True) -> None:
    check(lib.lsn_profile_enable(1 if on else 0))


def profile_read(reset: bool = False) -> dict:
    """GEMM launches timed with CUDA events since the last reset: count, ms, FLOPs."""
    p = lsn_profile()
    check(lib.lsn_profile_read(C.byref(p), 1 if reset else 0))
    return {"gemm_launches": p.gemm_launches, "gemm_ms": p.gemm_ms, "gemm_flops": p.gemm_flops}


# ------------------------------------------------------------------------ stream pool

class StreamPool:
    """Two-slot VRAM pool over a pinned host store (owner of the C handle)."""

    def __init__(self, store, offsets, layer_bytes: int, slot0, slot1, copy_stream, first_slot: int = 0,
                 reuse_resident: bool = False):
        self._keep = (store, slot0, slot1, copy_stream)
        n = len(offsets)
        offs = (C.c_size_t * n)(*[int(o) for o in offsets])
        h = C.c_void_p()
        check(lib.stream_pool_create(C.c_void_p(store.data_ptr()), store.numel() * store.element_size(), offs,
                                     layer_bytes, n, _p(slot0), _p(slot1), C.c_void_p(copy_stream.cuda_stream),
                                     first_slot, 1 if reuse_resident else 0, C.byref(h)))
        self.handle = h

    def prefetch(self, layer: int, reverse: bool = False):
        check(lib.stream_pool_prefetch_ex(self.handle, layer, 1 if reverse else 0))

    def wait(self, layer: int, stream=None, timeout_ms: int = 0) -> int:
        p = C.c_void_p()
        check(lib.stream_pool_wait(self.handle, layer, _stream(stream), C.byref(p), timeout_ms))
        return p.value

    def wait_range(self, layer: int, begin: int, end: int, stream=None, timeout_ms: int = 0) -> int:
        p = C.c_void_p()
        check(lib.stream_pool_wait_range(self.handle, layer, begin, end, _stream(stream), C.byref(p), timeout_ms))
        return p.value

    def set_chunks(self, offsets):
        """Copy every layer as len(offsets) chunks starting at these byte offsets (offsets[0] = 0)."""
        n = len(offsets)
        arr = (C.c_size_t * n)(*[int(o) for o in offsets])
        check(lib.stream_pool_set_chunks(self.handle, n, arr))

    def chunk_stats(self, chunk: int) -> dict:
        s = lsn_pool_stats()
        check(lib.stream_pool_chunk_stats(self.handle, chunk, C.byref(s)))
        return {"bytes_copied": s.bytes_copied, "copies": s.copies, "copy_ms": s.copy_ms}

    def release(self, layer: int, stream=None):
        check(lib.stream_pool_release(self.handle, layer, _stream(stream)))

    def set_copy_delay_us(self, usec: int):
        check(lib.stream_pool_set_copy_delay_us(self.handle, usec))

    def stats(self) -> dict:
        s = lsn_pool_stats()
        check(lib.stream_pool_stats(self.handle, C.byref(s)))
        return {"bytes_copied": s.bytes_copied, "copies": s.copies, "skipped": s.skipped,
                "copy_ms": s.copy_ms, "wait_ms": s.wait_ms}

    def reset_stats(self):
        check(lib.stream_pool_reset_stats(self.handle))

    def close(self):
        if self.handle:
            check(lib.stream_pool_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------------ layer stack

class StackDesc:
    """Shapes of the synthetic decoder-layer stack and the layouts the library derives."""

    def __init__(self, n_layers=32, d_model=4096, d_kv=1024, d_ff=14336, rank=64, lora_alpha=16.0,
                 rms_eps=1e-5, kv_loss_coef=1e-3):
        self.c = lsn_stack_desc(n_layers, d_model, d_kv, d_ff, rank, lora_alpha, rms_eps, kv_loss_coef)
        self.n_layers, self.d_model, self.d_kv, self.d_ff, self.rank = n_layers, d_model, d_kv, d_ff, rank
        self.scale = lora_alpha / rank
        self.image_bytes = int(lib.lsn_layer_image_bytes(C.byref(self.c)))
        if self.image_bytes == 0:
            raise LsnError(LSN_EINVAL, "bad stack descriptor")
        offs = (C.c_size_t * 7)()
        check(lib.lsn_layer_image_offsets(C.byref(self.c), offs))
        self.image_offsets = list(offs)
        self.lora_elems = int(lib.lsn_lora_elems(C.byref(self.c)))
        lo = (C.c_size_t * 14)()
        check(lib.lsn_lora_offsets(C.byref(self.c), lo))
        self.lora_offsets = list(lo)

    def chunk_offsets(self):
        """Byte offsets of the two sub-layer chunks of an image: [header, q, k, v, gate, up]
        and [o, down] (the parts the forward needs first and the backward needs first)."""
        return [0, self.image_offsets[PROJ.index("o")]]

    def shape(self, p: str):
        D, dkv, F = self.d_model, self.d_kv, self.d_ff
        return {"q": (D, D), "k": (dkv, D), "v": (dkv, D), "gate": (F, D), "up": (F, D), "o": (D, D),
                "down": (D, F)}[p]

    def workspace_bytes(self, M: int, recompute: bool = False, reference_pass: bool = False,
                        bwd_weights: int = 0) -> int:
        if not (recompute or reference_pass or bwd_weights):
            return int(lib.lsn_stack_workspace_bytes(C.byref(self.c), M))
        o = lsn_step_opts(1 if recompute else 0, 1 if reference_pass else 0)
        o.bwd_weights = int(bwd_weights)
        return int(lib.lsn_stack_workspace_bytes_ex(C.byref(self.c), M, C.byref(o)))

    def pack_layer(self, layer: int, W: dict, dst: np.ndarray | None = None, n_threads: int = 0) -> np.ndarray:
        """Packs one layer image (header + seven NF4 matrices) from fp32 numpy weights."""
        mats = [np.ascontiguousarray(W[p], dtype=np.float32) for p in PROJ]
        for p, m in zip(PROJ, mats):
            if m.shape != self.shape(p):
                raise LsnError(LSN_EINVAL, f"W[{p}] has shape {m.shape}, expected {self.shape(p)}")
        ptrs = (C.c_void_p * 7)(*[m.ctypes.data for m in mats])
        if dst is None:
            dst = np.empty(self.image_bytes, dtype=np.uint8)
        check(lib.lsn_layer_image_pack(C.byref(self.c), layer, ptrs, dst.ctypes.data_as(C.c_void_p), dst.nbytes,
                                       n_threads))
        return dst

    def lora_views(self, blob):
        """Views of A_p [r x K_p] and B_p [N_p x r] inside one layer's LoRA (or grad) blob."""
        A, B = {}, {}
        r = self.rank
        for i, p in enumerate(PROJ):
            n, k = self.shape(p)
            A[p] = blob[self.lora_offsets[i]: self.lora_offsets[i] + r * k].view(r, k)
            B[p] = blob[self.lora_offsets[7 + i]: self.lora_offsets[7 + i] + n * r].view(n, r)
        return A, B


class AdamW:
    """Per-layer AdamW state for the update fused into the reverse sweep: fp32 master copies
    (initialised from the bf16 LoRA blobs), zero moments, and the blobs it refreshes."""

    def __init__(self, lora_blobs, lr=2e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0):
        torch = _torch()
        self.blobs = lora_blobs
        self.master = [b.float().clone() for b in lora_blobs]
        self.m = [torch.zeros_like(x) for x in self.master]
        self.v = [torch.zeros_like(x) for x in self.master]
        self.hp = lsn_adamw_hparams(lr, beta1, beta2, eps, weight_decay, 0)

    def state(self):
        """The C struct for the next step (advances the step counter)."""
        self.hp.step += 1
        L = len(self.blobs)
        self._arrays = [(C.c_void_p * L)(*[t.data_ptr() for t in ts])
                        for ts in (self.master, self.m, self.v, self.blobs)]
        return lsn_adamw_state(self.hp, *self._arrays)


def shard_range(tokens: int, world: int, rank: int):
    """Rows [begin, end) of a global batch of `tokens` rows that data-parallel rank `rank` of
    `world` holds: contiguous, the first tokens % world ranks one row longer."""
    if world < 1 or not 0 <= rank < world or tokens < world:
        raise ValueError("need 0 <= rank < world <= tokens")
    base, extra = divmod(tokens, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def sum_ranks(gathered, n_ranks: int, out, stream=None):
    """out = gathered[0] + gathered[1] + ... in rank order (fp32), gathered = [n_ranks * n]."""
    n = out.numel()
    check(lib.lsn_sum_ranks(_p(gathered), n_ranks, n, _p(out), _stream(stream)))


class DataParallel:
    """Token-sharded data parallelism over a torch.distributed process group (NCCL).

    Every rank runs layer_stack_step on its own shard of the global batch, streaming the layers
    from its own pinned store, with token_count = the global token count so that its loss and
    gradients are its exact share.  Right after each layer's backward (the step's per-layer
    hook) the layer's gradient blob is all-gathered on a communication stream and summed in rank
    order by lsn_sum_ranks: every rank ends with the same bits, and the exchange of layer l
    overlaps the backward of layer l - 1.  finish() makes the compute stream wait for the last
    exchange."""

    def __init__(self, dist, desc: StackDesc, grad_blobs, compute_stream, group=None):
        torch = _torch()
        self.dist, self.group = dist, group
        self.world = dist.get_world_size(group)
        self.grads = grad_blobs
        self.compute = compute_stream
        self.comm = torch.cuda.Stream(device=compute_stream.device)
        self.gathered = torch.empty(self.world * desc.lora_elems, dtype=torch.float32, device=compute_stream.device)
        self.error = None
        self.hook = lsn_layer_hook(self._on_layer)   # pass as grads_ready; kept alive with the object

    def _on_layer(self, user, layer, grad_ptr, elems, stream_ptr):
        torch = _torch()
        g = self.grads[layer]
        if g.data_ptr() != grad_ptr or g.numel() != elems:
            # an exception cannot cross the C caller: finish() raises it
            self.error = f"DataParallel: layer {layer}'s gradient blob is not the one it was given"
            return
        ready = torch.cuda.Event()
        ready.record(self.compute if stream_ptr is None else
                     torch.cuda.ExternalStream(stream_ptr, device=self.compute.device))
        self.comm.wait_event(ready)
        with torch.cuda.stream(self.comm):
            self.dist.all_gather_into_tensor(self.gathered, g, group=self.group)
        sum_ranks(self.gathered, self.world, g, stream=self.comm)

    def finish(self):
        """The compute stream waits for every exchange of the step."""
        torch = _torch()
        if self.error:
            err, self.error = self.error, None
            raise RuntimeError(err)
        done = torch.cuda.Event()
        done.record(self.comm)
        self.compute.wait_event(done)


def layer_stack_step(desc: StackDesc, x0, lora_blobs, grad_blobs, loss_out, ws, pool: StreamPool | None = None,
                     resident_store=None, x_out=None, dx0=None, stream=None, recompute: bool = False,
                     reference_pass: bool = False, x_ref_out=None, adamw: "AdamW | None" = None,
                     x_layers_out=None, dx_layers_out=None, token_count: int = 0, grads_ready=None,
                     bwd_weights: int = 0):
    """One forward + loss + backward pass over the stack (streamed through `pool`, or resident).

    recompute: keep only x_l per layer and recompute the rest in the reverse sweep.
    reference_pass: also run the adapter-disabled forward on the same streamed slots and write
    it to x_ref_out.
    x_layers_out: bf16 [L, M, d_model] receives every layer's output x_{l+1}.
    dx_layers_out: fp32 [L, M, d_model] receives the gradient w.r.t. every layer's input x_l.
    token_count: the token count the loss means are taken over (0: M; a data-parallel shard
    passes the global batch's).
    grads_ready: a lsn_layer_hook (e.g. DataParallel's) called after each layer's backward.
    bwd_weights: 0 or 1 NF4 decoded inside the backward GEMMs, 2 each layer's weights decoded to
    bf16 scratch first (identical results; size ws with the same value)."""
    L = desc.n_layers
    lo = (C.c_void_p * L)(*[b.data_ptr() for b in lora_blobs])
    gr = (C.c_void_p * L)(*[g.data_ptr() for g in grad_blobs])
    if not (recompute or reference_pass or x_ref_out is not None or adamw is not None or
            x_layers_out is not None or dx_layers_out is not None or token_count or grads_ready is not None or
            bwd_weights):
        check(lib.layer_stack_step(pool.handle if pool is not None else None, _p(resident_store), C.byref(desc.c),
                                   _p(x0), x0.shape[0], lo, gr, _p(loss_out), _p(x_out), _p(dx0), _p(ws),
                                   ws.numel(), _stream(stream)))
        return
    o = lsn_step_opts(1 if recompute else 0, 1 if reference_pass else 0)
    if adamw is not None:
        st = adamw.state()
        o.adamw = C.pointer(st)
    o.x_layers_out = None if x_layers_out is None else x_layers_out.data_ptr()
    o.dx_layers_out = None if dx_layers_out is None else dx_layers_out.data_ptr()
    o.token_count = int(token_count)
    o.bwd_weights = int(bwd_weights)
    if grads_ready is not None:
        o.grads_ready = grads_ready
    check(lib.layer_stack_step_ex(pool.handle if pool is not None else None, _p(resident_store), C.byref(desc.c),
                                  C.byref(o), _p(x0), x0.shape[0], lo, gr, _p(loss_out), _p(x_out), _p(x_ref_out),
                                  _p(dx0), _p(ws), ws.numel(), _stream(stream)))
