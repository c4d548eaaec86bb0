"""The synthetic decoder layer, the layer stack, its loss and the hand-derived backward.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may use this module.

Streaming changes when a layer's weights reach the GPU, never what is computed ("Can You
Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained", section "The
gradient bug also reveals something important about AI benchmarks": the streamed run must
give the resident run's forward output and its LoRA gradients).  So the oracle of the
streamed step is the plain mathematics of the stack on the NF4-dequantised weights:

    h     = rmsnorm(x)  = x * (mean(x^2) + eps)^-1/2             (unit weight; bf16)
    p     = h W_p^T + s (h A_p^T) B_p^T   for p in q, k, v, gate, up   (bf16)
    a     = silu(gate) * up                                          (bf16)
    x'    = x + [q W_o^T + s (q A_o^T) B_o^T] + [a W_d^T + s (a A_d^T) B_d^T]   (bf16)
    loss  = 0.5 mean(x_L^2) + sum_l c (mean(k_l^2) + mean(v_l^2)),   c = 1e-3

The synthetic layer has no attention: o is applied to q directly.  Every tensor that the
GPU path stores in bf16 (h, the T's, q, k, v, gate, up, a, x') is rounded to bf16 here when
``rnd`` is set; everything else stays float64.  The backward is written by hand from the
chain rule; the finite-difference tests check it.
"""
from __future__ import annotations

import numpy as np

from .lora import bf16_round, lora_backward, lora_forward

QKVGU = ("q", "k", "v", "gate", "up")
PROJ = ("q", "k", "v", "o", "gate", "up", "down")


def rmsnorm_forward(x, eps):
    x = np.asarray(x, np.float64)
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)
    return x * rstd[:, None], rstd


def rmsnorm_backward(x, rstd, dh):
    """d/dx of h = x * rstd(x): rstd*dh - rstd^3 * x * mean(dh*x)."""
    x = np.asarray(x, np.float64)
    dot = np.mean(dh * x, axis=1)
    return rstd[:, None] * dh - (rstd ** 3 * dot)[:, None] * x


def sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def silu(g):
    return g * sigmoid(g)


def silu_mul_backward(g, u, da):
    """a = silu(g) * u:  dg = da*u*sig(g)*(1 + g*(1 - sig(g))),  du = da*silu(g)."""
    sg = sigmoid(g)
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    return dg, du


def layer_forward(x, W, A, B, scale, eps=1e-5, rnd=True):
    """One layer.  W, A, B: dicts keyed by projection name (float64 values).

    Returns (x_next, cache)."""
    R = bf16_round if rnd else (lambda t: np.asarray(t, np.float64))
    x = np.asarray(x, np.float64)
    h, rstd = rmsnorm_forward(x, eps)
    h = R(h)
    out, T = {}, {}
    for p in QKVGU:
        y, T[p] = lora_forward(h, W[p], A[p], B[p], scale, rnd)
        out[p] = R(y)
    a = R(silu(out["gate"]) * out["up"])
    o, T["o"] = lora_forward(out["q"], W["o"], A["o"], B["o"], scale, rnd)
    d, T["down"] = lora_forward(a, W["down"], A["down"], B["down"], scale, rnd)
    x_next = R(x + o + d)
    cache = {"x": x, "h": h, "rstd": rstd, "a": a, "T": T, **out}
    return x_next, cache


def layer_backward(cache, dx_next, W, A, B, scale, dk_seed, dv_seed):
    """Backward of one layer.  dx_next: gradient of the loss wrt x_next.

    dk_seed / dv_seed: loss gradients wrt this layer's k and v.
    Returns (dx, dA: dict, dB: dict)."""
    dA, dB = {}, {}
    dq, dA["o"], dB["o"] = lora_backward(cache["q"], W["o"], A["o"], B["o"], cache["T"]["o"],
                                         dx_next, scale)
    da, dA["down"], dB["down"] = lora_backward(cache["a"], W["down"], A["down"], B["down"],
                                               cache["T"]["down"], dx_next, scale)
    dg, du = silu_mul_backward(cache["gate"], cache["up"], da)
    dY = {"q": dq, "k": dk_seed, "v": dv_seed, "gate": dg, "up": du}
    dh = np.zeros_like(cache["h"])
    for p in QKVGU:
        dX, dA[p], dB[p] = lora_backward(cache["h"], W[p], A[p], B[p], cache["T"][p], dY[p], scale)
        dh = dh + dX
    dx = dx_next + rmsnorm_backward(cache["x"], cache["rstd"], dh)
    return dx, dA, dB


def loss_terms(x_last, ks, vs, kv_coef=1e-3):
    L = 0.5 * np.mean(np.asarray(x_last, np.float64) ** 2)
    for k, v in zip(ks, vs):
        L += kv_coef * (np.mean(np.asarray(k, np.float64) ** 2) + np.mean(np.asarray(v, np.float64) ** 2))
    return L


def stack_forward_backward(x0, layers, scale, eps=1e-5, kv_coef=1e-3, rnd=True,
                           token_count=None):
    """Forward sweep over all layers, the loss, then the reverse backward sweep.

    layers: list of (W, A, B) dict triples.  ``token_count`` is the M that normalises the
    means (defaults to the rows of x0; a token slice of a larger batch passes the full M).
    Returns dict(loss, x_last, xs, caches, dA, dB, dx0)."""
    x = np.asarray(x0, np.float64)
    M = x.shape[0] if token_count is None else token_count
    caches, xs = [], [x]
    for (W, A, B) in layers:
        x, c = layer_forward(x, W, A, B, scale, eps, rnd)
        caches.append(c)
        xs.append(x)
    D = x.shape[1]
    loss = 0.5 * np.sum(x * x) / (M * D)
    for c in caches:
        dkv = c["k"].shape[1]
        loss += kv_coef * (np.sum(c["k"] ** 2) + np.sum(c["v"] ** 2)) / (M * dkv)
    dx = x / (M * D)
    dAs, dBs = [None] * len(layers), [None] * len(layers)
    for li in range(len(layers) - 1, -1, -1):
        W, A, B = layers[li]
        c = caches[li]
        dkv = c["k"].shape[1]
        coef = 2.0 * kv_coef / (M * dkv)
        dx, dAs[li], dBs[li] = layer_backward(c, dx, W, A, B, scale, coef * c["k"], coef * c["v"])
    return {"loss": loss, "x_last": xs[-1], "xs": xs, "caches": caches,
            "dA": dAs, "dB": dBs, "dx0": dx}


def frozen_stack_forward(x0, Ws, eps=1e-5, rnd=True):
    """The reference model of preference training: the same frozen base with the adapter
    disabled (the rug.gal radar item "soup-fine-tune-8b-4gb-laptop-gpu-layer-streaming",
    section "In detail": the DPO reference model reuses the base stream without LoRA).
    Ws: list of per-layer weight dicts.  Each layer is the synthetic layer with no LoRA terms:
    h = rmsnorm(x); p = h W_p^T; a = silu(gate) up; x' = x + q W_o^T + a W_d^T."""
    R = bf16_round if rnd else (lambda t: np.asarray(t, np.float64))
    x = np.asarray(x0, np.float64)
    for W in Ws:
        h, _ = rmsnorm_forward(x, eps)
        h = R(h)
        out = {p: R(h @ np.asarray(W[p], np.float64).T) for p in QKVGU}
        a = R(silu(out["gate"]) * out["up"])
        x = R(x + out["q"] @ np.asarray(W["o"], np.float64).T + a @ np.asarray(W["down"], np.float64).T)
    return x
