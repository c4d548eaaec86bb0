"""The frozen-base linear with its trainable LoRA branch, forward and backward, in float64.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may use this module.

The method ("Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming
Explained", section "How Soup's layer streaming actually works", step 1 "The base model is
frozen"): the base weight W is frozen and gets no gradient; only the low-rank factors train.
With W [N x K], A [r x K], B [N x r] and s = alpha / r:

    T  = X A^T                      (stored; rounded to bf16 when ``rnd``)
    Y  = X W^T + s T B^T
    dT = s dY B
    dB = s dY^T T
    dA = dT^T X
    dX = dY W + dT A

There is no dW.  Matrix products are numpy float64 matmuls; nothing is blocked, fused or
reordered.
"""
from __future__ import annotations

import numpy as np

from .nf4 import bf16_bits, bf16_value


def bf16_round(x) -> np.ndarray:
    """Round float64 values as a stored bf16 tensor: to fp32 first, then fp32 -> bf16 RNE."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    return bf16_value(bf16_bits(x32)).astype(np.float64)


def lora_forward(X, W, A, B, scale, rnd=True):
    """Returns (Y, T).  All inputs float64 values; Y is left unrounded."""
    X = np.asarray(X, np.float64)
    T = X @ np.asarray(A, np.float64).T
    if rnd:
        T = bf16_round(T)
    Y = X @ np.asarray(W, np.float64).T + scale * (T @ np.asarray(B, np.float64).T)
    return Y, T


def lora_backward(X, W, A, B, T, dY, scale):
    """Returns (dX, dA, dB) for the loss gradient dY of Y; W is frozen (no dW)."""
    X = np.asarray(X, np.float64)
    dY = np.asarray(dY, np.float64)
    B = np.asarray(B, np.float64)
    dT = scale * (dY @ B)
    dB = scale * (dY.T @ np.asarray(T, np.float64))
    dA = dT.T @ X
    dX = dY @ np.asarray(W, np.float64) + dT @ np.asarray(A, np.float64)
    return dX, dA, dB
