"""Pins of the AdamW oracle by closed forms (CPU only)."""
import numpy as np

from oracle import optim


def test_first_step_is_signed_lr():
    """At t = 1 the bias-corrected moments are g and g^2, so without decay each parameter
    moves by -lr * g / (|g| + eps)."""
    rng = np.random.default_rng(0)
    p = rng.standard_normal(1000)
    g = rng.standard_normal(1000)
    p1, m1, v1 = optim.adamw_step(p, g, np.zeros(1000), np.zeros(1000), 1, lr=1e-3, eps=1e-8)
    np.testing.assert_allclose(p1, p - 1e-3 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-12)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-12)


def test_constant_gradient_moments_are_unbiased():
    """With a constant gradient the bias-corrected moments equal g and g^2 at every step."""
    g = np.array([0.5, -2.0, 3e-3])
    p = np.zeros(3)
    m = np.zeros(3)
    v = np.zeros(3)
    for t in range(1, 30):
        p_prev = p.copy()
        p, m, v = optim.adamw_step(p, g, m, v, t, lr=0.01, eps=0.0)
        np.testing.assert_allclose(m / (1 - 0.9 ** t), g, rtol=1e-12)
        np.testing.assert_allclose(p - p_prev, -0.01 * np.sign(g), rtol=1e-10)


def test_decoupled_weight_decay():
    """With a zero gradient only the decay acts: p <- p (1 - lr wd)."""
    p = np.array([1.0, -4.0])
    p1, _, _ = optim.adamw_step(p, np.zeros(2), np.zeros(2), np.zeros(2), 3, lr=0.1, wd=0.5, eps=1e-8)
    np.testing.assert_allclose(p1, p * (1 - 0.05), rtol=1e-15)
