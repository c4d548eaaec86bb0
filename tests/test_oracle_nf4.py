"""Pins of the NF4 oracle against what the definition and the pages fix (CPU only)."""
import os

import numpy as np
import pytest
from scipy.special import ndtr

from oracle import nf4
from synth import layer_shapes, single_linear_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# ----------------------------------------------------------------------------- codebook

def test_codebook_structure():
    c = nf4.codebook()
    assert c.dtype == np.float32 and c.shape == (16,)
    assert np.all(np.diff(c) > 0), "strictly ascending"
    assert c[0] == -1.0 and c[15] == 1.0
    assert np.count_nonzero(c == 0.0) == 1 and c[7] == 0.0, "exactly one exact zero"
    assert np.count_nonzero(c < 0) == 7 and np.count_nonzero(c > 0) == 8
    assert not np.signbit(c[7])


def _bisect_quantile(p):
    """Inverse of the normal CDF by bisection on ndtr (independent of ndtri)."""
    lo, hi = -10.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if ndtr(mid) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_codebook_levels_are_normal_quantiles():
    """Mapping each level back through the forward normal CDF recovers the evenly spaced
    probability grid of the construction (8 positive, 7 negative levels)."""
    delta = nf4.outer_probability()
    assert abs(delta - (1 - (1 / 30 + 1 / 32) / 2)) < 1e-15
    z = _bisect_quantile(delta)
    c64 = nf4.codebook_f64()
    pos = c64[8:][::-1]                 # descending positive levels
    neg = -c64[:7]                      # magnitudes of the negative levels, descending
    p_pos = ndtr(pos * z)
    p_neg = ndtr(neg * z)
    np.testing.assert_allclose(p_pos, delta - np.arange(8) * (delta - 0.5) / 8, rtol=0, atol=1e-12)
    np.testing.assert_allclose(p_neg, delta - np.arange(7) * (delta - 0.5) / 7, rtol=0, atol=1e-12)
    # the fp32 table is the single rounding of those levels
    c32 = nf4.codebook()
    ulp = np.spacing(np.abs(c32))
    assert np.all(np.abs(c32.astype(np.float64) - c64) <= 0.5 * ulp)


def test_midpoint_rule_equals_brute_force_argmin():
    rng = np.random.default_rng(5)
    c = nf4.codebook().astype(np.float64)
    n = np.concatenate([rng.uniform(-1, 1, 20000), c, [-1.0, 1.0, 0.0]])
    dist = np.abs(n[:, None] - c[None, :])
    brute = np.argmin(dist, axis=1)     # argmin returns the first (lower) index on ties
    np.testing.assert_array_equal(nf4.codes_of(n), brute)


def test_ties_go_to_lower_code():
    m = nf4.midpoints_f64()
    np.testing.assert_array_equal(nf4.codes_of(m), np.arange(15))
    np.testing.assert_array_equal(nf4.codes_of(np.nextafter(m, 2.0)), np.arange(1, 16))


# ----------------------------------------------------------------------- hand examples

def test_hand_example_exact_levels():
    g = _golden("nf4_hand_examples.txt")
    c = nf4.codebook()
    W = (np.float32(0.5) * np.tile(c, 4)).astype(np.float32).reshape(1, 64)
    st = nf4.quantize(W)
    np.testing.assert_array_equal(st["codes"], np.array(g["A_codes"], dtype=np.uint8))
    np.testing.assert_array_equal(st["absmax_q"], np.array(g["A_absmax_q"], dtype=np.uint8))
    assert st["scale"][0] == np.float32(g["A_scale"][0])
    assert st["offset"][0] == np.float32(g["A_offset"][0])
    np.testing.assert_array_equal(nf4.dequantize_f32(st), W)


def test_hand_example_group_arithmetic():
    g = _golden("nf4_hand_examples.txt")
    W = np.zeros((3, 64), np.float32)
    W[1, 0] = 255.0
    W[2, 0] = 100.5
    W[2, 1] = -50.25
    st = nf4.quantize(W)
    np.testing.assert_array_equal(st["absmax_q"], np.array(g["B_absmax_q"], dtype=np.uint8))
    assert st["scale"][0] == np.float32(g["B_scale"][0])
    assert st["offset"][0] == np.float32(g["B_offset"][0])
    codes = st["codes"].reshape(3, 64)
    assert codes[1, 0] == int(g["B_row1_col0_code"][0])
    assert codes[2, 0] == int(g["B_row2_col0_code"][0])
    assert codes[2, 1] == int(g["B_row2_col1_code"][0])
    zero = int(g["B_zero_code"][0])
    assert np.all(codes[0] == zero) and np.all(codes[1, 1:] == zero) and np.all(codes[2, 2:] == zero)


# ----------------------------------------------------------------------------- zeros

def test_exact_zero():
    W = np.zeros((4, 128), np.float32)
    st = nf4.quantize(W)
    assert np.all(st["codes"] == 7)
    deq = nf4.dequantize_bf16_bits(st)
    assert np.all(deq == 0), "all-zero input decodes to +0"
    rng = np.random.default_rng(1)
    W = rng.standard_normal((8, 128)).astype(np.float32)
    W[:, ::3] = 0.0
    W[2, 5] = -0.0
    st = nf4.quantize(W)
    deq = nf4.dequantize_bf16_bits(st).reshape(8, 128)
    zmask = W == 0.0
    assert np.all(st["codes"].reshape(8, 128)[zmask] == 7)
    assert np.all(deq[zmask] == 0)


# ------------------------------------------------------------------ error bound, a' >= a

def _check_bounds(W):
    st = nf4.quantize(W)
    c = nf4.codebook().astype(np.float64)
    w = W.reshape(-1).astype(np.float64)
    a = np.repeat(st["absmax_deq"].astype(np.float64), 64)
    assert np.all(st["absmax_deq"].astype(np.float64) >= st["absmax"].astype(np.float64))
    codes = st["codes"].astype(np.int64)
    approx = nf4.dequantize_f32(st).reshape(-1).astype(np.float64)
    # half-gap bound on the interval that contains n, plus the fp32 rounding of c*a'
    with np.errstate(divide="ignore", invalid="ignore"):
        n = np.where(a > 0, w / a, 0.0)
    idx = np.clip(np.searchsorted(c, n, side="right") - 1, 0, 14)
    gap = c[idx + 1] - c[idx]
    bound = a * gap / 2 + np.spacing(np.abs(approx).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(w - approx) <= bound * (1 + 1e-12))
    # the bf16 value adds at most half a bf16 ulp
    bf = nf4.bf16_value(nf4.dequantize_bf16_bits(st)).reshape(-1).astype(np.float64)
    bf_ulp = np.abs(bf) * 2.0 ** -7 + 1e-45
    assert np.all(np.abs(bf - approx) <= 0.5 * bf_ulp * 1.0000001 + 2.0 ** -133)
    assert np.all((codes >= 0) & (codes <= 15))
    return st


def test_roundtrip_error_bound_workload_weights():
    W = single_linear_inputs()["W"]
    st = _check_bounds(W)
    assert st["scale"].shape == (1024 * 512 // 64 // 256,)


def test_roundtrip_adversarial_blocks():
    rng = np.random.default_rng(7)
    rows = []
    rows.append(np.zeros(64))                                  # all zero
    rows.append(np.full(64, 0.37))                             # constant
    spike = np.zeros(64); spike[13] = 1e3; rows.append(spike)  # one spike
    rows.append(np.where(np.arange(64) % 2 == 0, 3.4e38, -3.4e38))   # +-max
    rows.append(rng.standard_normal(64) * 1e-40)               # subnormal fp32
    rows.append(np.full(64, -1e-45))                           # smallest subnormal
    c = nf4.codebook().astype(np.float64)
    mids = (c[:-1] + c[1:]) / 2
    rows.append(np.concatenate([mids, mids, mids, mids, [1.0, -1.0, 0.5, 0.25]]))  # midpoints
    for _ in range(50):                                        # widely varying absmax
        rows.append(rng.standard_normal(64) * 10.0 ** rng.uniform(-30, 30))
    W = np.array(rows, dtype=np.float32)
    _check_bounds(W)


def test_many_groups_absmax_never_below():
    """Random absmax spreads inside 256-block groups exercise the round-up of the scale and
    the raising of codes; a' >= a must hold everywhere."""
    rng = np.random.default_rng(11)
    blocks = rng.standard_normal((256 * 40, 64)).astype(np.float32)
    blocks *= (10.0 ** rng.uniform(-3, 3, (256 * 40, 1))).astype(np.float32)
    st = nf4.quantize(blocks.reshape(-1, 256))
    assert np.all(st["absmax_deq"].astype(np.float64) >= st["absmax"].astype(np.float64))


def test_partial_last_group():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((5, 64 * 7)).astype(np.float32)    # 35 blocks, one partial group
    st = _check_bounds(W)
    assert st["scale"].shape == (1,)
    lay = nf4.packed_layout(5, 64 * 7)
    assert lay["groups"] == 1 and lay["blocks"] == 35


def test_rejects_nonfinite():
    W = np.zeros((1, 64), np.float32)
    W[0, 3] = np.nan
    with pytest.raises(ValueError):
        nf4.quantize(W)
    with pytest.raises(ValueError):
        nf4.quantize(np.zeros((1, 65), np.float32))


# -------------------------------------------------------------------- fp32 emulation

def test_fp32_emulation_matches_float32_ops():
    rng = np.random.default_rng(2)
    q = rng.integers(0, 256, 100000).astype(np.float32)
    scale = (rng.random(100000) * 1e-2).astype(np.float32)
    lo = (rng.random(100000) * 1e-1).astype(np.float32)
    ref = (q * scale) + lo                      # numpy float32 ops: each rounded to fp32
    assert ref.dtype == np.float32
    np.testing.assert_array_equal(nf4.dequantised_absmax(q, scale, lo), ref)
    c = nf4.codebook()
    codes = rng.integers(0, 16, 100000)
    a = (rng.random(100000) * 3).astype(np.float32)
    st = {"N": 1, "K": 100032, "codes": np.concatenate([codes, np.zeros(32, int)]),
          "absmax_deq": np.concatenate([a[::64][: 100032 // 64]])}
    got = nf4.dequantize_f32(st).reshape(-1)
    a_elem = np.repeat(st["absmax_deq"], 64)
    np.testing.assert_array_equal(got, c[st["codes"]] * a_elem)


def test_bf16_rounding_rne():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -0.0,
                  3.3895313892515355e38], np.float32)
    got = nf4.bf16_value(nf4.bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -0.0,
                                                 3.3895313892515355e38], np.float32))


# -------------------------------------------------------------------- packed layout

def test_pack_unpack_roundtrip():
    W = single_linear_inputs()["W"]
    st = nf4.quantize(W)
    buf = nf4.pack(st)
    assert len(buf) == nf4.packed_layout(1024, 512)["total"] == 270592
    back = nf4.unpack(buf, 1024, 512)
    for k in ("codes", "absmax_q", "scale", "offset", "absmax_deq"):
        np.testing.assert_array_equal(back[k], st[k])
    b = np.frombuffer(buf, np.uint8)
    assert b[0] >> 4 == st["codes"][0] and b[0] & 15 == st["codes"][1]


def test_layer_store_size_matches_pages():
    g = _golden("layer_sizes.txt")
    per_layer = sum(nf4.packed_layout(n, k)["total"] for n, k in layer_shapes().values())
    assert per_layer == 112_566_272
    assert round(32 * per_layer / 1e9, 2) == float(g["store_gb_32_layers"][0])
    assert round(per_layer / 1e6) == int(g["slot_mb"][0])
    assert abs(per_layer / 2 ** 20 - float(g["layer_mib_about"][0])) / 105 < 0.05
    params = sum(n * k for n, k in layer_shapes().values())
    assert abs(per_layer / (2 * params) - float(g["fraction_of_bf16_about"][0])) < 0.02


def test_quantize_ties_go_to_lower_code():
    """Weights that normalise exactly onto a midpoint take the lower code.  A block with
    absmax 1 has a' = 1, so w / a' = w; the midpoints that are fp32 values are such weights."""
    m = nf4.midpoints_f64()
    exact = [x for x in m if float(np.float32(x)) == x]
    assert exact, "some midpoint is an fp32 value"
    row = np.zeros(64, np.float32)
    row[0] = 1.0                                 # absmax 1 -> a' = 1 (single block group)
    row[1:1 + len(exact)] = np.array(exact, np.float32)
    st = nf4.quantize(row.reshape(1, 64))
    assert st["absmax_deq"][0] == 1.0
    lower = np.searchsorted(m, np.array(exact), side="left")
    np.testing.assert_array_equal(st["codes"][1:1 + len(exact)], lower)


def test_scale_is_rounded_up_and_minimal():
    """scale >= (hi - lo)/255 exactly, and the next smaller fp32 value is either below that
    quotient or would leave some block of the group with a' < absmax."""
    from fractions import Fraction
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((64, 256 * 64)) * 10.0 ** rng.uniform(-4, 4, (64, 1))).astype(np.float32)
    st = nf4.quantize(W)
    a = st["absmax"].reshape(-1, 256)
    for g in range(a.shape[0]):
        lo, hi, s = a[g].min(), a[g].max(), st["scale"][g]
        target = (Fraction(float(hi)) - Fraction(float(lo))) / 255
        assert st["offset"][g] == lo
        assert Fraction(float(s)) >= target
        prev = np.nextafter(s, np.float32(0))
        if Fraction(float(prev)) >= target:
            ap = nf4.dequantised_absmax(np.full(256, 255.0), np.full(256, prev, np.float32),
                                        np.full(256, lo, np.float32))
            assert np.any(ap.astype(np.float64) < a[g].astype(np.float64))
