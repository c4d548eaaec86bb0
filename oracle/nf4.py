"""NF4 quantisation of the frozen base, written out step by step in float64.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may use this module.

What the pages fix, and the readings taken where they are silent:

* "Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained",
  section "Why NF4 matters so much": the frozen base is stored in NF4, the four-bit
  format of QLoRA, at about a quarter of its bf16 size.  The page names the format and
  links the QLoRA paper; it does not define the codebook.
* The workload description fixes the packing: blocks of 64 consecutive weights along the
  input dimension, one uint8 absmax code per block, and an fp32 scale and offset for every
  256 consecutive absmax values ("double quantisation").

Readings (each also listed in the design notes):

1. Codebook.  QLoRA's asymmetric normal-quantile construction: 8 positive levels at the
   standard-normal quantiles of 8 evenly spaced probabilities from ``delta`` down to (but
   excluding) 1/2, 7 negative levels likewise, plus an exact zero; all divided by the
   largest and rounded once to fp32.  ``delta = 1 - (1/30 + 1/32)/2`` places the outermost
   level between the outermost quantiles of a 15- and a 16-level grid.
2. Double quantisation: plain affine uint8 codes per 256-block group,
   ``scale = fp32_up((hi - lo)/255)``, ``q = ceil((a - lo)/scale)`` clamped to [0, 255],
   ``a' = fp32(fp32(q*scale) + lo)``; ``q`` is raised while ``a' < a`` and, if that would
   pass 255, the group's scale is raised by one fp32 ulp and the group redone.  This makes
   ``a' >= a`` for every block, so every normalised weight lies in [-1, 1].
3. Codes: ``n = w / a'`` in float64 (``n = 0`` when ``a' = 0``); the code is the number of
   fp64 midpoints ``(c_i + c_{i+1})/2`` strictly below ``n`` (a tie goes to the lower code).
4. Nibble order: element ``2j`` in the high nibble of byte ``j``.
5. Dequantised value: ``bf16_rne(fp32(c[code] * a'))``.
6. Packed layout of one matrix [N x K]: codes (N*K/2 bytes) | absmax codes (N*K/64 bytes)
   | scale fp32[G] | offset fp32[G], each section padded to 16 bytes, G = ceil(N*K/64/256).
"""
from __future__ import annotations

import numpy as np
from scipy.special import ndtri

BLOCK = 64          # weights per absmax block
GROUP = 256         # absmax blocks per (scale, offset) group


# ----------------------------------------------------------------------------- codebook

def outer_probability() -> float:
    """Probability of the outermost NF4 level (reading 1)."""
    return 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)


def codebook_f64() -> np.ndarray:
    """The 16 NF4 levels in float64, ascending, before the single fp32 rounding."""
    delta = outer_probability()
    positive = ndtri(np.linspace(delta, 0.5, 9)[:-1])      # 8 levels, Q(delta) .. > 0
    negative = -ndtri(np.linspace(delta, 0.5, 8)[:-1])     # 7 levels, -Q(delta) .. < 0
    levels = np.concatenate([negative, [0.0], positive])
    levels = levels / ndtri(delta)
    return np.sort(levels)


def codebook() -> np.ndarray:
    """The NF4 codebook as the fp32 table the method uses."""
    return codebook_f64().astype(np.float32)


def midpoints_f64() -> np.ndarray:
    c = codebook().astype(np.float64)
    return (c[:-1] + c[1:]) / 2.0          # exact in fp64: c_i are fp32


def codes_of(n) -> np.ndarray:
    """Code of normalised values n (float64): the number of midpoints strictly below n,
    i.e. the nearest level with ties going to the lower level."""
    return np.searchsorted(midpoints_f64(), np.asarray(n, np.float64), side="left").astype(np.uint8)


# ------------------------------------------------------------------------ fp32 helpers

def f32(x) -> np.ndarray:
    """Round float64 values to fp32 (round to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def f32_round_up(x64) -> np.ndarray:
    """Smallest fp32 value >= x (x >= 0, float64)."""
    x64 = np.asarray(x64, dtype=np.float64)
    r = x64.astype(np.float32)
    low = r.astype(np.float64) < x64
    r = np.where(low, np.nextafter(r, np.float32(np.inf)), r).astype(np.float32)
    return r


def bf16_bits(x32) -> np.ndarray:
    """fp32 -> bf16 by round-to-nearest-even on the bit pattern (finite inputs)."""
    x32 = np.ascontiguousarray(np.asarray(x32, dtype=np.float32))
    u = x32.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    bits = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------------- quantiser

def dequantised_absmax(q, scale, lo) -> np.ndarray:
    """a' = fp32(fp32(q * scale) + lo), each operation rounded once to fp32.

    ``q * scale`` is exact in float64 (an 8-bit integer times a 24-bit significand), so
    rounding it to fp32 is the correctly rounded fp32 product; the fp64 sum rounded to fp32
    is the correctly rounded fp32 sum (double rounding is innocuous for 53 >= 2*24+2).
    """
    t = f32(np.asarray(q, np.float64) * np.asarray(scale, np.float32).astype(np.float64))
    return f32(t.astype(np.float64) + np.asarray(lo, np.float32).astype(np.float64))


def _group_codes(a64, lo, scale):
    """Initial uint8 codes of a set of blocks for given per-block (lo, scale)."""
    s64 = scale.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.ceil((a64 - lo.astype(np.float64)) / s64)
    q = np.where(s64 > 0, q, 0.0)
    return np.clip(q, 0, 255)


def quantize(W) -> dict:
    """Quantise an fp32 matrix [N x K] (K a multiple of 64) to NF4 with double quantisation.

    Returns codes (uint8, one per weight, 0..15), absmax_q (uint8 per block), scale and
    offset (fp32 per group), and the dequantised absmax a' (fp32 per block).
    """
    W = np.ascontiguousarray(np.asarray(W, dtype=np.float32))
    if W.ndim != 2 or W.shape[1] % BLOCK != 0:
        raise ValueError("W must be [N x K] with K a multiple of 64")
    if not np.isfinite(W).all():
        raise ValueError("W must be finite")
    N, K = W.shape
    w = W.reshape(-1)
    nb = w.size // BLOCK
    G = -(-nb // GROUP)
    absmax = np.abs(w.reshape(nb, BLOCK)).max(axis=1)            # fp32, exact
    a64 = absmax.astype(np.float64)
    pad = G * GROUP - nb
    lo = np.concatenate([a64, np.full(pad, np.inf)]).reshape(G, GROUP).min(axis=1)
    hi = np.concatenate([a64, np.full(pad, -np.inf)]).reshape(G, GROUP).max(axis=1)
    lo = lo.astype(np.float32)                                      # exact: fp32 values
    hi = hi.astype(np.float32)
    scale = f32_round_up((hi.astype(np.float64) - lo.astype(np.float64)) / 255.0)
    gid = np.arange(nb) // GROUP

    redo = np.ones(G, dtype=bool)
    q = np.zeros(nb, dtype=np.float64)
    aq = np.zeros(nb, dtype=np.float32)
    while redo.any():
        sel = redo[gid]
        qs = _group_codes(a64[sel], lo[gid[sel]], scale[gid[sel]])
        ap = dequantised_absmax(qs, scale[gid[sel]], lo[gid[sel]])
        # raise codes while the dequantised absmax is below the true absmax
        while True:
            short = (ap.astype(np.float64) < a64[sel]) & (qs < 255)
            if not short.any():
                break
            qs = qs + short
            ap = dequantised_absmax(qs, scale[gid[sel]], lo[gid[sel]])
        q[sel] = qs
        aq[sel] = ap
        bad = np.zeros(G, dtype=bool)
        still = aq[sel].astype(np.float64) < a64[sel]
        bad[np.unique(gid[sel][still])] = True
        scale = np.where(bad, np.nextafter(scale, np.float32(np.inf)), scale).astype(np.float32)
        redo = bad

    # codes: nearest level of n = w / a', ties to the lower level
    a_elem = np.repeat(aq.astype(np.float64), BLOCK)
    with np.errstate(divide="ignore", invalid="ignore"):
        n = w.astype(np.float64) / a_elem
    n = np.where(a_elem == 0.0, 0.0, n)
    codes = codes_of(n)
    return {
        "N": N, "K": K,
        "codes": codes,
        "absmax_q": q.astype(np.uint8),
        "scale": scale.astype(np.float32),
        "offset": lo.astype(np.float32),
        "absmax_deq": aq,
        "absmax": absmax,
    }


# ---------------------------------------------------------------------- packed layout

def _align16(x: int) -> int:
    return (x + 15) // 16 * 16


def packed_layout(N: int, K: int) -> dict:
    """Byte offsets of the four sections of one packed matrix (reading 6)."""
    nb = N * K // BLOCK
    G = -(-nb // GROUP)
    codes = 0
    absmax = _align16(N * K // 2)
    scale = absmax + _align16(nb)
    offset = scale + _align16(4 * G)
    total = offset + _align16(4 * G)
    return {"codes": codes, "absmax": absmax, "scale": scale, "offset": offset,
            "total": total, "blocks": nb, "groups": G}


def pack(state) -> bytes:
    N, K = state["N"], state["K"]
    lay = packed_layout(N, K)
    buf = np.zeros(lay["total"], dtype=np.uint8)
    c = state["codes"].astype(np.uint8)
    buf[: N * K // 2] = (c[0::2] << 4) | c[1::2]
    buf[lay["absmax"]: lay["absmax"] + lay["blocks"]] = state["absmax_q"]
    G = lay["groups"]
    buf[lay["scale"]: lay["scale"] + 4 * G] = np.frombuffer(
        state["scale"].astype("<f4").tobytes(), dtype=np.uint8)
    buf[lay["offset"]: lay["offset"] + 4 * G] = np.frombuffer(
        state["offset"].astype("<f4").tobytes(), dtype=np.uint8)
    return buf.tobytes()


def unpack(buf, N: int, K: int) -> dict:
    lay = packed_layout(N, K)
    b = np.frombuffer(bytes(buf), dtype=np.uint8)
    if b.size < lay["total"]:
        raise ValueError("buffer too small")
    by = b[: N * K // 2]
    codes = np.empty(N * K, dtype=np.uint8)
    codes[0::2] = by >> 4
    codes[1::2] = by & 0xF
    G = lay["groups"]
    absmax_q = b[lay["absmax"]: lay["absmax"] + lay["blocks"]].copy()
    scale = np.frombuffer(b[lay["scale"]: lay["scale"] + 4 * G].tobytes(), dtype="<f4").astype(np.float32)
    offset = np.frombuffer(b[lay["offset"]: lay["offset"] + 4 * G].tobytes(), dtype="<f4").astype(np.float32)
    gid = np.arange(lay["blocks"]) // GROUP
    aq = dequantised_absmax(absmax_q.astype(np.float64), scale[gid], offset[gid])
    return {"N": N, "K": K, "codes": codes, "absmax_q": absmax_q, "scale": scale,
            "offset": offset, "absmax_deq": aq}


# ------------------------------------------------------------------------ dequantiser

def dequantize_f32(state) -> np.ndarray:
    """fp32(c[code] * a') per weight, [N x K] (the product rounded once to fp32)."""
    c = codebook().astype(np.float64)
    a_elem = np.repeat(state["absmax_deq"].astype(np.float64), BLOCK)
    return f32(c[state["codes"]] * a_elem).reshape(state["N"], state["K"])


def dequantize_bf16_bits(state) -> np.ndarray:
    """The dequantised weights as bf16 bit patterns [N x K] (reading 5)."""
    return bf16_bits(dequantize_f32(state))


def dequantize(state) -> np.ndarray:
    """The dequantised weights as float64 values of the bf16 results [N x K]."""
    return bf16_value(dequantize_bf16_bits(state)).astype(np.float64)
