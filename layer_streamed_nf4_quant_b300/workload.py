"""Synthetic Llama-3.1-8B-shaped workloads: pinned host stores of packed layer images, LoRA
blobs and inputs.  Weights and factors come from the seeded generators in ``synth``; the
packing is the library's host quantiser."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import synth

from . import PROJ, StackDesc


def _torch():
    import torch
    return torch


def build_store(desc: StackDesc, n_layers: int | None = None, pinned: bool = True, workers: int | None = None,
                seed_base: int = 100):
    """Packs layers 0..n_layers-1 (weights seeded seed_base + l) into one host uint8 tensor,
    layer l at byte offset l * desc.image_bytes."""
    torch = _torch()
    L = desc.n_layers if n_layers is None else n_layers
    nbytes = L * desc.image_bytes
    store = torch.empty(nbytes, dtype=torch.uint8, pin_memory=pinned)
    host = store.numpy()
    cpus = os.cpu_count() or 4
    workers = workers or max(1, min(L, cpus // 4, 16))
    pack_threads = max(1, cpus // workers)

    def one(layer: int):
        W = synth.layer_weights(layer, desc.d_model, desc.d_kv, desc.d_ff, seed_base=seed_base)
        dst = host[layer * desc.image_bytes:(layer + 1) * desc.image_bytes]
        desc.pack_layer(layer, W, dst=dst, n_threads=pack_threads)
        return layer

    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(one, range(L)))
    return store


def lora_blob(desc: StackDesc, layer: int, device="cuda", seed_base: int = 200):
    """One layer's LoRA blob (bf16, canonical layout) on the device."""
    torch = _torch()
    A, B = synth.layer_lora(layer, desc.rank, desc.d_model, desc.d_kv, desc.d_ff, seed_base=seed_base)
    parts = [A[p].reshape(-1) for p in PROJ] + [B[p].reshape(-1) for p in PROJ]
    bits = np.concatenate(parts)
    assert bits.size == desc.lora_elems
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor(bits, device="cuda"):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
