"""Oracle side of the full-size stack tests: the NF4-dequantised weights of the 32
Llama-3.1-8B-shaped layers, computed by the oracle (``oracle.nf4``) from the seeded weights
in ``synth``, and per-layer access in the form ``oracle.stack`` takes.

Quantising one full layer in the oracle takes about 20 s and 3.4 GB, so the layers are
quantised by a pool of spawned worker processes (spawn, never fork: the test process has a
CUDA context).  The weights are kept as bf16 bit patterns (436 MB per layer) and handed out
as fp32 values, which are exact for bf16; the oracle computes in float64 from them.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np


def _dequantised_layer(args):
    layer, D, dkv, F = args
    import synth
    from oracle import nf4 as onf4
    W = synth.layer_weights(layer, D, dkv, F)
    return layer, {p: onf4.dequantize_bf16_bits(onf4.quantize(w)) for p, w in W.items()}


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


class OracleLayers:
    """Sequence of (W, A, B) dict triples, one per layer, in the form ``oracle.stack`` takes."""

    def __init__(self, n_layers, D=4096, dkv=1024, F=14336, r=64, workers=None):
        self.n = n_layers
        self.dims = (D, dkv, F, r)
        cpus = os.cpu_count() or 2
        workers = workers or max(1, min(n_layers, cpus // 2, 8))
        self.bits = [None] * n_layers
        with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
            for layer, b in ex.map(_dequantised_layer, [(l, D, dkv, F) for l in range(n_layers)]):
                self.bits[layer] = b

    def weights(self, layer):
        return {p: _f32(b) for p, b in self.bits[layer].items()}

    def lora(self, layer):
        import synth
        from oracle.nf4 import bf16_value
        D, dkv, F, r = self.dims
        A, B = synth.layer_lora(layer, r, D, dkv, F)
        return ({p: bf16_value(a).astype(np.float64) for p, a in A.items()},
                {p: bf16_value(b).astype(np.float64) for p, b in B.items()})

    def __len__(self):
        return self.n

    def __getitem__(self, layer):
        if not 0 <= layer < self.n:
            raise IndexError(layer)
        A, B = self.lora(layer)
        return self.weights(layer), A, B

    def __iter__(self):
        for layer in range(self.n):
            yield self[layer]
