"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

This module only draws random numbers and stores them in the dtypes the workloads name
(fp32 weights, bf16 activations and LoRA factors).  It holds none of the method's
arithmetic: no quantisation, no matrix products, no rounding beyond the plain
fp32 -> bf16 storage conversion of a drawn value.

bf16 tensors are carried as numpy ``uint16`` bit patterns.

Workloads (Llama-3.1-8B-shaped synthetic layers, standing in for the pages' Llama 3.1 8B
Instruct fine-tune on an instruction dataset, whose weights and data are not used):

* single linear: X [128x512] ~N(0,1), W [1024x512] ~N(0,0.02^2) fp32, A [8x512] ~U(+-1/sqrt(512)),
  B [1024x8] ~N(0,0.01^2), dY [128x1024] ~N(0,1), one generator seeded 0, drawn in that order.
* decoder layer l: the seven base weights from a generator seeded 100+l, drawn in the
  projection order q, k, v, o, gate, up, down; the LoRA factors from a generator seeded
  200+l: A_p ~U(+-1/sqrt(K_p)) for all p in order, then B_p ~N(0,0.01^2) for all p in order.
* stack input x0 [M x 4096] ~N(0,1) from a generator seeded 1.
"""
from __future__ import annotations

import numpy as np

PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even) and return the bit patterns."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def layer_shapes(d_model: int = 4096, d_kv: int = 1024, d_ff: int = 14336):
    """(n_out, k_in) of the seven projections of one synthetic decoder layer."""
    return {
        "q": (d_model, d_model),
        "k": (d_kv, d_model),
        "v": (d_kv, d_model),
        "o": (d_model, d_model),
        "gate": (d_ff, d_model),
        "up": (d_ff, d_model),
        "down": (d_model, d_ff),
    }


def single_linear_inputs(seed: int = 0, M: int = 128, K: int = 512, N: int = 1024, r: int = 8):
    """The single frozen NF4 linear + LoRA workload.

    Returns X, A, B, dY as bf16 bit patterns and W as fp32.
    """
    rng = np.random.default_rng(seed)
    X = f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    W = (np.float32(0.02) * rng.standard_normal((N, K), dtype=np.float32)).astype(np.float32)
    bound = np.float32(1.0 / np.sqrt(K))
    A = f32_to_bf16_bits(rng.uniform(-bound, bound, size=(r, K)).astype(np.float32))
    B = f32_to_bf16_bits((np.float32(0.01) * rng.standard_normal((N, r), dtype=np.float32)))
    dY = f32_to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return {"X": X, "W": W, "A": A, "B": B, "dY": dY}


def layer_weights(layer: int, d_model: int = 4096, d_kv: int = 1024, d_ff: int = 14336,
                  seed_base: int = 100, std: float = 0.02):
    """The seven fp32 base weights [n_out x k_in] of decoder layer ``layer``."""
    rng = np.random.default_rng(seed_base + layer)
    out = {}
    for name, (n, k) in layer_shapes(d_model, d_kv, d_ff).items():
        w = rng.standard_normal((n, k), dtype=np.float32)
        w *= np.float32(std)
        out[name] = w
    return out


def layer_lora(layer: int, r: int = 64, d_model: int = 4096, d_kv: int = 1024,
               d_ff: int = 14336, seed_base: int = 200):
    """LoRA factors of decoder layer ``layer``: A_p [r x K_p], B_p [N_p x r], bf16 bits."""
    rng = np.random.default_rng(seed_base + layer)
    shapes = layer_shapes(d_model, d_kv, d_ff)
    A, B = {}, {}
    for name, (n, k) in shapes.items():
        bound = np.float32(1.0 / np.sqrt(k))
        A[name] = f32_to_bf16_bits(rng.uniform(-bound, bound, size=(r, k)).astype(np.float32))
    for name, (n, k) in shapes.items():
        B[name] = f32_to_bf16_bits(np.float32(0.01) * rng.standard_normal((n, r), dtype=np.float32))
    return A, B


def stack_input(M: int, d_model: int = 4096, seed: int = 1):
    """x0 [M x d_model] ~N(0,1) as bf16 bits.  Rows are drawn in order, so the first
    512 rows of a larger M equal the M=512 input."""
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((M, d_model), dtype=np.float32))


def random_bf16(shape, seed: int, std: float = 1.0):
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(np.float32(std) * rng.standard_normal(shape, dtype=np.float32))
