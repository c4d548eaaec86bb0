"""Writes stack_drift.json: how far two correct implementations of the 32-layer stack drift
apart end to end, which sizes the end-to-end tolerance of the full-stack GPU tests.

    python tests/golden/stack_drift.py        # about 15 minutes on 8 cores, 40 GB of RAM

The stated bars (forward max|y - y_ref| / max|y_ref| <= 2e-2, gradients relative Frobenius
<= 1e-2) hold for one layer on its own inputs.  Over 32 layers every stored bf16 tensor
(h, q, k, v, gate, up, a, the T's, x_l) is rounded in every layer, and an implementation that
accumulates its matrix products in fp32 instead of fp64 rounds a few of them the other way;
the stack amplifies those one-ulp differences layer after layer.  This script measures that
drift with no GPU involved: the oracle (oracle.stack, float64) against a twin that takes the
oracle's steps in the same order with the same bf16 rounding points but with its matrix
products in float32 (numpy's sgemm: fp32 accumulation, like the tensor cores).  It also
measures what the kernels' bf16 gradient operands alone change (the dX path is a bf16 GEMM:
dloss/dx' entering the o/down backward, dY_cat and the dT's are bf16 GEMM inputs there).

The weights are the oracle's own NF4 quantisation of the seeded workload weights; the inputs
are the seeded batch 1 x 512 tokens.  Nothing here touches the CUDA library.
"""
from __future__ import annotations

import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

from oracle import stack as ostack  # noqa: E402
from oracle.lora import bf16_round  # noqa: E402

QKVGU = ("q", "k", "v", "gate", "up")


def _mm(a, b, f32):
    if f32:
        return (np.asarray(a, np.float32) @ np.asarray(b, np.float32)).astype(np.float64)
    return np.asarray(a, np.float64) @ np.asarray(b, np.float64)


def _linear_fwd(X, W, A, B, s, f32):
    T = bf16_round(_mm(X, A.T, f32))
    return _mm(X, W.T, f32) + s * _mm(T, B.T, f32), T


def _layer_fwd(x, W, A, B, s, f32, eps=1e-5):
    h, rstd = ostack.rmsnorm_forward(x, eps)
    h = bf16_round(h)
    out, T = {}, {}
    for p in QKVGU:
        y, T[p] = _linear_fwd(h, W[p], A[p], B[p], s, f32)
        out[p] = bf16_round(y)
    a = bf16_round(ostack.silu(out["gate"]) * out["up"])
    o, T["o"] = _linear_fwd(out["q"], W["o"], A["o"], B["o"], s, f32)
    d, T["down"] = _linear_fwd(a, W["down"], A["down"], B["down"], s, f32)
    return bf16_round(x + o + d), {"x": x, "h": h, "rstd": rstd, "a": a, "T": T, **out}


def _linear_bwd(X, W, A, B, T, dY, s, f32, bf16_grads):
    R = bf16_round if bf16_grads else (lambda t: t)
    dY = R(dY)
    dT = R(s * _mm(dY, B, f32))
    return _mm(dY, W, f32) + _mm(dT, A, f32), _mm(dT.T, X, f32), s * _mm(dY.T, T, f32)


def twin_step(x0, layers, s, f32, bf16_grads, kv_coef=1e-3):
    """The oracle's forward sweep, loss seeds and reverse sweep, step by step, with the
    matrix products in float32 (f32) and/or the backward GEMM operands in bf16."""
    x, caches, xs = x0, [], [x0]
    for (W, A, B) in layers:
        x, c = _layer_fwd(x, W, A, B, s, f32)
        caches.append(c)
        xs.append(x)
    M, D = x.shape
    dx = x / (M * D)
    dA, dB = [None] * len(caches), [None] * len(caches)
    for li in range(len(caches) - 1, -1, -1):
        W, A, B = layers[li]
        c = caches[li]
        coef = 2.0 * kv_coef / (M * c["k"].shape[1])
        gA, gB = {}, {}
        dq, gA["o"], gB["o"] = _linear_bwd(c["q"], W["o"], A["o"], B["o"], c["T"]["o"], dx, s, f32, bf16_grads)
        da, gA["down"], gB["down"] = _linear_bwd(c["a"], W["down"], A["down"], B["down"], c["T"]["down"], dx, s,
                                                 f32, bf16_grads)
        dg, du = ostack.silu_mul_backward(c["gate"], c["up"], da)
        dY = {"q": dq, "k": coef * c["k"], "v": coef * c["v"], "gate": dg, "up": du}
        dh = 0.0
        for p in QKVGU:
            dXp, gA[p], gB[p] = _linear_bwd(c["h"], W[p], A[p], B[p], c["T"][p], dY[p], s, f32, bf16_grads)
            dh = dh + dXp
        dx = dx + ostack.rmsnorm_backward(c["x"], c["rstd"], dh)
        dA[li], dB[li] = gA, gB
    return {"xs": xs, "dx0": dx, "dA": dA, "dB": dB}


def twin_frozen(x0, Ws, f32, eps=1e-5):
    """oracle.stack.frozen_stack_forward with the matrix products in float32."""
    x = x0
    for W in Ws:
        h, _ = ostack.rmsnorm_forward(x, eps)
        h = bf16_round(h)
        out = {p: bf16_round(_mm(h, W[p].T, f32)) for p in QKVGU}
        a = bf16_round(ostack.silu(out["gate"]) * out["up"])
        x = bf16_round(x + _mm(out["q"], W["o"].T, f32) + _mm(a, W["down"].T, f32))
    return x


def _max_rel(a, b):
    return float(np.max(np.abs(a - b)) / np.max(np.abs(b)))


def _fro_rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def drift(got, ref, L):
    worst = max(max(_fro_rel(got["dA"][l][p], ref["dA"][l][p]), _fro_rel(got["dB"][l][p], ref["dB"][l][p]))
                for l in range(L) for p in ref["dA"][l])
    return {"x_L_max_rel": _max_rel(got["xs"][L], ref["xs"][L]),
            "x_l_max_rel": [_max_rel(got["xs"][l], ref["xs"][l]) for l in range(1, L + 1)],
            "dx0_fro_rel": _fro_rel(got["dx0"], ref["dx0"]), "worst_grad_fro_rel": worst}


def main():
    import synth
    from _oracle_layers import OracleLayers
    from oracle.nf4 import bf16_value
    L, M, s = 32, 512, 16.0 / 64
    t0 = time.time()
    layers = OracleLayers(L, workers=4)
    x0 = bf16_value(synth.stack_input(M, 4096)).astype(np.float64)
    ref = ostack.stack_forward_backward(x0, layers, s)                    # the oracle itself
    ref.pop("caches")
    twin = twin_step(x0, layers, s, f32=True, bf16_grads=True)           # fp32 products, bf16 grad operands
    ref_bf = twin_step(x0, layers, s, f32=False, bf16_grads=True)        # fp64, bf16 grad operands only
    fz_ref = ostack.frozen_stack_forward(x0, (layers.weights(l) for l in range(L)))
    fz_twin = twin_frozen(x0, (layers.weights(l) for l in range(L)), f32=True)
    rec = {
        "what": "end-to-end drift of the 32-layer stack at batch 1 x 512 tokens: the fp64 oracle against a twin with "
                "fp32-accumulated matrix products and the same bf16 rounding points",
        "command": "python tests/golden/stack_drift.py",
        "layers": L, "tokens": M,
        "fp32_twin_vs_oracle": drift(twin, ref, L),
        "fp32_twin_frozen_vs_oracle_frozen": {"x_L_max_rel": _max_rel(fz_twin, fz_ref)},
        "bf16_grad_operands_only_vs_oracle": {k: v for k, v in drift(ref_bf, ref, L).items() if k != "x_l_max_rel"},
        "seconds": time.time() - t0,
    }
    with open(os.path.join(HERE, "stack_drift.json"), "w") as f:
        json.dump(rec, f, indent=1)
    print(json.dumps({k: v for k, v in rec["fp32_twin_vs_oracle"].items() if k != "x_l_max_rel"}))


if __name__ == "__main__":
    main()
