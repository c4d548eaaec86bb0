"""The oracle's layer forward against the hand-derived tiny layer in golden/tiny_layer.txt.

The file works out, step by step, one synthetic decoder layer (one token, d_model 2, d_kv 1,
d_ff 2, rank 1, s = 1/2, eps = 0) with values chosen so that each bf16 rounding point changes
a stored tensor and so that applying o to h instead of q, or rounding o and down before the
residual sum, changes x'.  These checks pin oracle.stack.layer_forward against something
other than itself: the finite-difference tests only check that its backward agrees with its
forward."""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import stack as ostack

HERE = os.path.join(os.path.dirname(__file__), "golden", "tiny_layer.txt")


def _golden():
    vals = {}
    for line in open(HERE):
        line = line.split("#", 1)[0].strip()
        if not line or "=" not in line:
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        rows = [[float(Fraction(t.strip())) for t in r.split(",")] for r in v.split(";")]
        vals[k] = np.array(rows, dtype=np.float64)
    return vals


def _layer(g):
    W, A, B = {}, {}, {}
    for p in ("q", "k", "v", "gate", "up", "o", "down"):
        W[p] = g["W_" + p]
        A[p] = g["A_" + p].reshape(1, -1)
        B[p] = g["B_" + p].reshape(-1, 1)
    return W, A, B


@pytest.fixture(scope="module")
def run():
    g = _golden()
    W, A, B = _layer(g)
    x_next, cache = ostack.layer_forward(g["x"].reshape(1, 2), W, A, B, 0.5, eps=0.0, rnd=True)
    return g, x_next, cache


def test_golden_inputs_have_the_stated_shapes(run):
    g, _, _ = run
    assert g["W_q"].shape == (2, 2) and g["W_k"].shape == (1, 2) and g["W_down"].shape == (2, 2)
    assert g["B_q"].shape == (2, 1) and g["A_down"].shape == (1, 2)


@pytest.mark.parametrize("name", ["h", "q", "k", "v", "gate", "up", "a"])
def test_stored_activations_match_the_hand_derivation(run, name):
    g, _, cache = run
    np.testing.assert_array_equal(cache[name].reshape(-1), g[name].reshape(-1))


@pytest.mark.parametrize("proj", ["q", "k", "v", "gate", "up", "o", "down"])
def test_lora_down_projections_match_the_hand_derivation(run, proj):
    g, _, cache = run
    np.testing.assert_array_equal(cache["T"][proj].reshape(-1), g["T_" + proj].reshape(-1))


def test_layer_output_matches_the_hand_derivation(run):
    g, x_next, _ = run
    np.testing.assert_array_equal(x_next.reshape(-1), g["x_next"].reshape(-1))


def test_unrounded_path_differs_where_the_derivation_rounds(run):
    """The same layer with the roundings switched off lands on the unrounded values the file
    lists beside each rounding (so each listed bf16 value really is a rounding point)."""
    g, _, _ = run
    W, A, B = _layer(g)
    x_next, cache = ostack.layer_forward(g["x"].reshape(1, 2), W, A, B, 0.5, eps=0.0, rnd=False)
    assert cache["h"][0, 0] == pytest.approx(0.632455532033676, abs=1e-15)   # x0 * (5/2)^-1/2
    for name in ("h", "q", "gate", "up", "a"):
        assert cache[name][0, 0] != g[name][0, 0], name
    for proj in ("q", "down"):
        assert cache["T"][proj][0, 0] != g["T_" + proj][0, 0], proj
    assert x_next[0, 0] != g["x_next"][0, 0]
