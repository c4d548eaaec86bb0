"""ctypes declarations of liblsn.so (argument marshalling only; every computation runs in
the library).  Loading fails loudly if the library has not been built."""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblsn.so")

LSN_OK = 0
LSN_EINVAL = -1
LSN_ENOMEM = -2
LSN_ECUDA = -3
LSN_ETIMEOUT = -4
LSN_ESTATE = -5
LSN_ECORRUPT = -6
STATUS_NAMES = {0: "OK", -1: "EINVAL", -2: "ENOMEM", -3: "ECUDA", -4: "ETIMEOUT", -5: "ESTATE",
                -6: "ECORRUPT"}


class LsnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class nf4_view(C.Structure):
    _fields_ = [("base", C.c_void_p), ("n_out", C.c_int64), ("k_in", C.c_int64)]


class lsn_pool_stats(C.Structure):
    _fields_ = [("bytes_copied", C.c_uint64), ("copies", C.c_uint64), ("skipped", C.c_uint64),
                ("copy_ms", C.c_double), ("wait_ms", C.c_double)]


class lsn_stack_desc(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("d_kv", C.c_int32),
                ("d_ff", C.c_int32), ("rank", C.c_int32), ("lora_alpha", C.c_float),
                ("rms_eps", C.c_float), ("kv_loss_coef", C.c_float)]


class lsn_adamw_hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("step", C.c_int32)]


class lsn_adamw_state(C.Structure):
    _fields_ = [("hp", lsn_adamw_hparams), ("master", C.POINTER(C.c_void_p)), ("m", C.POINTER(C.c_void_p)),
                ("v", C.POINTER(C.c_void_p)), ("lora_out", C.POINTER(C.c_void_p))]


# void (*)(void* user, int32_t layer, float* grad, size_t elems, void* stream)
lsn_layer_hook = C.CFUNCTYPE(None, C.c_void_p, C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p)


class lsn_step_opts(C.Structure):
    _fields_ = [("recompute", C.c_int32), ("reference_pass", C.c_int32), ("bwd_weights", C.c_int32), ("reserved", C.c_int32 * 5),
                ("adamw", C.POINTER(lsn_adamw_state)), ("x_layers_out", C.c_void_p),
                ("dx_layers_out", C.c_void_p), ("token_count", C.c_int64), ("grads_ready", lsn_layer_hook),
                ("hook_user", C.c_void_p)]


class lsn_profile(C.Structure):
    _fields_ = [("gemm_launches", C.c_uint64), ("gemm_ms", C.c_double), ("gemm_flops", C.c_double)]


P = C.c_void_p
I = C.c_int
I64 = C.c_int64
SZ = C.c_size_t
F = C.c_float

# name -> (restype, argtypes); mirrors include/lsn.h
SIGNATURES = {
    "lsn_last_error": (C.c_char_p, []),
    "lsn_abi_version": (I, []),
    "lsn_check": (I, [P, C.POINTER(C.c_uint32)]),
    "lsn_launch_count": (C.c_uint64, []),
    "lsn_profile_enable": (I, [I]),
    "lsn_profile_read": (I, [C.POINTER(lsn_profile), I]),
    "lsn_nf4_codebook": (I, [C.POINTER(F)]),
    "nf4_packed_bytes": (SZ, [I64, I64]),
    "nf4_pack": (I, [P, I64, I64, P, SZ, I]),
    "nf4_dequant": (I, [C.POINTER(nf4_view), P, P]),
    "lora_nf4_workspace_bytes": (SZ, [I64, I64, I64, I]),
    "lora_nf4_fwd": (I, [C.POINTER(nf4_view), P, I64, P, P, I, F, P, P, P, P, SZ, P]),
    "lora_nf4_bwd": (I, [C.POINTER(nf4_view), P, P, P, I64, P, P, I, F, P, I, P, P, P, SZ, P]),
    "lora_nf4_fwd_plan": (I, [I64, I64, I64, I, C.POINTER(I), C.POINTER(I), C.POINTER(SZ), C.POINTER(SZ)]),
    "lora_nf4_fwd_static_scratch": (I, [C.POINTER(nf4_view), P, I64, P, P, I, F, P, P, P, C.POINTER(C.c_uint32),
                                        P]),
    "stream_pool_create": (I, [P, SZ, C.POINTER(SZ), SZ, I, P, P, P, I, I, C.POINTER(P)]),
    "stream_pool_prefetch": (I, [P, I]),
    "stream_pool_wait": (I, [P, I, P, C.POINTER(P), I]),
    "stream_pool_release": (I, [P, I, P]),
    "stream_pool_stats": (I, [P, C.POINTER(lsn_pool_stats)]),
    "stream_pool_reset_stats": (I, [P]),
    "stream_pool_set_copy_delay_us": (I, [P, I]),
    "stream_pool_set_chunks": (I, [P, I, C.POINTER(SZ)]),
    "stream_pool_prefetch_ex": (I, [P, I, I]),
    "stream_pool_wait_range": (I, [P, I, SZ, SZ, P, C.POINTER(P), I]),
    "stream_pool_chunk_stats": (I, [P, I, C.POINTER(lsn_pool_stats)]),
    "stream_pool_destroy": (I, [P]),
    "lsn_layer_image_bytes": (SZ, [C.POINTER(lsn_stack_desc)]),
    "lsn_layer_image_offsets": (I, [C.POINTER(lsn_stack_desc), C.POINTER(SZ)]),
    "lsn_layer_image_pack": (I, [C.POINTER(lsn_stack_desc), I, C.POINTER(P), P, SZ, I]),
    "lsn_lora_elems": (SZ, [C.POINTER(lsn_stack_desc)]),
    "lsn_lora_offsets": (I, [C.POINTER(lsn_stack_desc), C.POINTER(SZ)]),
    "lsn_stack_workspace_bytes": (SZ, [C.POINTER(lsn_stack_desc), I64]),
    "layer_stack_step": (I, [P, P, C.POINTER(lsn_stack_desc), P, I64, C.POINTER(P), C.POINTER(P), P, P, P,
                             P, SZ, P]),
    "lsn_stack_workspace_bytes_ex": (SZ, [C.POINTER(lsn_stack_desc), I64, C.POINTER(lsn_step_opts)]),
    "lsn_adamw_step": (I, [C.POINTER(lsn_adamw_hparams), P, P, P, P, P, SZ, P]),
    "lsn_sum_ranks": (I, [P, I, SZ, P, P]),
    "layer_stack_step_ex": (I, [P, P, C.POINTER(lsn_stack_desc), C.POINTER(lsn_step_opts), P, I64, C.POINTER(P),
                                C.POINTER(P), P, P, P, P, P, SZ, P]),
}


def load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python layer_streamed_nf4_quant_b300/build.py`")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load()


def check(rc: int) -> None:
    if rc != LSN_OK:
        raise LsnError(rc, lib.lsn_last_error().decode(errors="replace"))
