"""Pins of the LoRA-linear and layer-stack oracle (CPU only).

The backward is pinned by central finite differences of the float64 forward (unrounded
path); the forward by the LoRA merge identity, the B = 0 special case and closed forms of
RMSNorm, SiLU and the loss."""
import numpy as np
import pytest

from oracle import lora, stack
from oracle.stack import PROJ


def _rand(rng, *shape, s=1.0):
    return rng.standard_normal(shape) * s


# ------------------------------------------------------------------------ LoRA linear

def test_merge_identity():
    """Unrounded LoRA forward equals the plain linear with the merged weight W + s*B*A."""
    rng = np.random.default_rng(0)
    M, K, N, r, s = 7, 64, 48, 4, 2.0
    X, W, A, B = _rand(rng, M, K), _rand(rng, N, K), _rand(rng, r, K), _rand(rng, N, r)
    Y, _ = lora.lora_forward(X, W, A, B, s, rnd=False)
    merged = np.einsum("mk,nk->mn", X, W + s * np.einsum("nr,rk->nk", B, A))
    np.testing.assert_allclose(Y, merged, rtol=1e-12, atol=1e-12)


def test_B_zero_is_frozen_linear_and_A_zero_gives_zero_dB():
    rng = np.random.default_rng(1)
    M, K, N, r = 5, 64, 32, 8
    X, W, A = _rand(rng, M, K), _rand(rng, N, K), _rand(rng, r, K)
    Y, _ = lora.lora_forward(X, W, A, np.zeros((N, r)), 2.0)
    assert np.array_equal(Y, X @ W.T)
    dY = _rand(rng, M, N)
    _, dA, dB = lora.lora_backward(X, W, np.zeros((r, K)), _rand(rng, N, r),
                                   np.zeros((M, r)), dY, 2.0)
    assert np.all(dB == 0)


def _fd_dir(f, x, v, eps=1e-6):
    return (f(x + eps * v) - f(x - eps * v)) / (2 * eps)


def test_lora_backward_finite_differences():
    rng = np.random.default_rng(2)
    M, K, N, r, s = 4, 64, 64, 2, 0.25
    X, W, A, B = _rand(rng, M, K), _rand(rng, N, K), _rand(rng, r, K), _rand(rng, N, r)
    G = _rand(rng, M, N)

    def L(X_, A_, B_):
        Y, _ = lora.lora_forward(X_, W, A_, B_, s, rnd=False)
        return np.sum(G * Y)

    _, T = lora.lora_forward(X, W, A, B, s, rnd=False)
    dX, dA, dB = lora.lora_backward(X, W, A, B, T, G, s)
    for _ in range(3):
        vX, vA, vB = _rand(rng, M, K), _rand(rng, r, K), _rand(rng, N, r)
        for got, fd in ((np.sum(dX * vX), _fd_dir(lambda t: L(t, A, B), X, vX)),
                        (np.sum(dA * vA), _fd_dir(lambda t: L(X, t, B), A, vA)),
                        (np.sum(dB * vB), _fd_dir(lambda t: L(X, A, t), B, vB))):
            assert abs(got - fd) <= 1e-6 * max(1.0, abs(fd))


# ------------------------------------------------------------------ closed forms

def test_rmsnorm_closed_form():
    rng = np.random.default_rng(3)
    x = _rand(rng, 6, 32) * np.arange(1, 7)[:, None]
    eps = 1e-5
    h, rstd = stack.rmsnorm_forward(x, eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(h * h, axis=1), ms / (ms + eps), rtol=1e-13)
    h2, _ = stack.rmsnorm_forward(3.0 * x, 0.0)
    h1, _ = stack.rmsnorm_forward(x, 0.0)
    np.testing.assert_allclose(h1, h2, rtol=1e-13)


def test_silu_identities():
    g = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(stack.silu(-g), stack.silu(g) - g, atol=1e-12)
    assert stack.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(stack.silu(np.array([40.0])), [40.0], rtol=1e-15)
    u = np.cos(g)
    da = np.ones_like(g)
    dg, du = stack.silu_mul_backward(g, u, da)
    eps = 1e-6
    fd = (stack.silu(g + eps) * u - stack.silu(g - eps) * u) / (2 * eps)
    np.testing.assert_allclose(dg, fd, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(du, stack.silu(g), rtol=0, atol=0)


def test_loss_seed_gradient_closed_form():
    """With no layers, loss = 0.5 mean(x0^2) and its gradient is x0 / (M*D)."""
    rng = np.random.default_rng(4)
    x0 = _rand(rng, 5, 16)
    out = stack.stack_forward_backward(x0, [], 0.25, rnd=False)
    assert out["loss"] == pytest.approx(0.5 * np.mean(x0 ** 2), rel=1e-14)
    np.testing.assert_allclose(out["dx0"], x0 / x0.size, rtol=1e-14)


# ------------------------------------------------------------ stack finite differences

def _tiny_layers(rng, n_layers, d, dkv, dff, r):
    shapes = {"q": (d, d), "k": (dkv, d), "v": (dkv, d), "o": (d, d),
              "gate": (dff, d), "up": (dff, d), "down": (d, dff)}
    layers = []
    for _ in range(n_layers):
        W = {p: _rand(rng, n, k, s=0.3 / np.sqrt(k)) for p, (n, k) in shapes.items()}
        A = {p: _rand(rng, r, k, s=1 / np.sqrt(k)) for p, (n, k) in shapes.items()}
        B = {p: _rand(rng, n, r, s=0.2) for p, (n, k) in shapes.items()}
        layers.append((W, A, B))
    return layers


@pytest.mark.parametrize("n_layers", [1, 2])
def test_stack_backward_finite_differences(n_layers):
    rng = np.random.default_rng(10 + n_layers)
    d, dkv, dff, r, M, s = 16, 8, 24, 2, 3, 0.25
    layers = _tiny_layers(rng, n_layers, d, dkv, dff, r)
    x0 = _rand(rng, M, d)
    out = stack.stack_forward_backward(x0, layers, s, rnd=False)

    def loss_with(li=None, kind=None, p=None, v=None, eps=0.0, dx=None):
        ls = []
        for j, (W, A, B) in enumerate(layers):
            A2, B2 = dict(A), dict(B)
            if j == li:
                if kind == "A":
                    A2[p] = A[p] + eps * v
                else:
                    B2[p] = B[p] + eps * v
            ls.append((W, A2, B2))
        x = x0 if dx is None else x0 + dx
        return stack.stack_forward_backward(x, ls, s, rnd=False)["loss"]

    eps = 1e-6
    for li in range(n_layers):
        for p in PROJ:
            for kind in ("A", "B"):
                g = out["dA" if kind == "A" else "dB"][li][p]
                v = _rand(rng, *g.shape)
                fd = (loss_with(li, kind, p, v, eps) - loss_with(li, kind, p, v, -eps)) / (2 * eps)
                got = np.sum(g * v)
                assert abs(got - fd) <= 1e-6 * max(abs(fd), 1e-3), (li, p, kind, got, fd)
    v = _rand(rng, M, d)
    fd = (loss_with(dx=eps * v) - loss_with(dx=-eps * v)) / (2 * eps)
    assert abs(np.sum(out["dx0"] * v) - fd) <= 1e-6 * max(abs(fd), 1e-3)


def test_rounded_path_close_to_unrounded():
    """bf16 rounding of the stored tensors only perturbs the result at bf16 precision."""
    rng = np.random.default_rng(20)
    layers = _tiny_layers(rng, 2, 64, 32, 96, 4)
    x0 = _rand(rng, 8, 64)
    a = stack.stack_forward_backward(x0, layers, 0.25, rnd=False)
    b = stack.stack_forward_backward(x0, layers, 0.25, rnd=True)
    assert abs(a["loss"] - b["loss"]) / a["loss"] < 2e-2
    for li in range(2):
        for p in PROJ:
            num = np.linalg.norm(a["dA"][li][p] - b["dA"][li][p])
            assert num / np.linalg.norm(a["dA"][li][p]) < 5e-2


def test_frozen_forward_closed_forms():
    """Zero weights make every layer the identity; with weights it equals the policy forward
    whose adapter outputs are zero (B = 0), and differs once B is non-zero."""
    rng = np.random.default_rng(30)
    d, dkv, dff, r = 32, 16, 48, 4
    layers = _tiny_layers(rng, 2, d, dkv, dff, r)
    x0 = _rand(rng, 5, d)
    zeros = [{p: np.zeros_like(W[p]) for p in W} for (W, _, _) in layers]
    np.testing.assert_array_equal(stack.frozen_stack_forward(x0, zeros, rnd=False), x0)
    ref = stack.frozen_stack_forward(x0, [W for (W, _, _) in layers], rnd=False)
    no_adapter = [(W, A, {p: np.zeros_like(B[p]) for p in B}) for (W, A, B) in layers]
    x = x0
    for (W, A, B) in no_adapter:
        x, _ = stack.layer_forward(x, W, A, B, 0.25, rnd=False)
    np.testing.assert_allclose(ref, x, rtol=1e-13, atol=1e-13)
    x = x0
    for (W, A, B) in layers:
        x, _ = stack.layer_forward(x, W, A, B, 0.25, rnd=False)
    assert np.max(np.abs(ref - x)) > 1e-6
