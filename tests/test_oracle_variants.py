"""The oracle of TTT-Linear with a layer norm and a residual inside f, pinned (CPU only).

oracle/variants.py reads the normalised inner model as f(k; W) = k + LN(k W) and
trains it with the chunk rule. Its hand-written gradient is checked against
central finite differences of the loss and against torch autograd through
torch's own layer_norm; the token-by-token form against the chunk-by-chunk dual
form; eta = 0 (no update) and gamma = 0 (f no longer depends on W) against their
closed forms. A dropped mean in the normalisation's chain rule, a missing
residual or a gradient taken at the running weights each fail one of these.

The momentum variant (momentum gradient descent with chunk-start gradients) is
checked token by token against its closed-form dual, against the C oracle's
TTT-Linear at beta = 0, against torch autograd for every gradient, and at a zero
rate.

The bias variant (f(k) = k W + beta) is checked against the C oracle's plain
TTT-Linear on keys and queries extended by a constant 1 (an independent
implementation of the same chunk rule), its gradient against central finite
differences of 1/2 ||k W + beta - v||^2, and at eta = 0 against q W0 + beta0.
The per-token learning rate is checked against the C oracle at a constant rate,
against the C oracle with keys and values scaled by sqrt(eta_t) (the gradient of
token t picks up eta_t exactly once), and at eta_t = 0.
"""
import numpy as np
import pytest
import torch

from oracle.variants import LN_EPS, layer_norm, ln_residual_dual, ln_residual_error, ln_residual_primal


def rand_case(B, H, T, d, seed):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((B, H, T, d)) * 0.8 for _ in range(3))
    eta = g.uniform(0.05, 0.4, H)
    W0 = g.standard_normal((H, d, d)) * 0.4
    gamma = 1.0 + 0.3 * g.standard_normal((H, d))
    beta = 0.2 * g.standard_normal((H, d))
    return Q, K, V, eta, W0, gamma, beta


def loss(k, v, W, gamma, beta):
    return 0.5 * np.sum((k + layer_norm(k @ W, gamma, beta)[0] - v) ** 2)


@pytest.mark.parametrize("d", [2, 3, 8])
def test_gradient_equals_finite_differences(d):
    g = np.random.default_rng(d)
    k, v = g.standard_normal(d), g.standard_normal(d)
    W = g.standard_normal((d, d)) * 0.5
    gamma, beta = 1.0 + 0.3 * g.standard_normal(d), 0.2 * g.standard_normal(d)
    grad = np.outer(k, ln_residual_error(k[None], v[None], W, gamma, beta)[0])
    h = 1e-6
    fd = np.zeros_like(W)
    for i in range(d):
        for j in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += h
            Wm[i, j] -= h
            fd[i, j] = (loss(k, v, Wp, gamma, beta) - loss(k, v, Wm, gamma, beta)) / (2 * h)
    assert np.allclose(grad, fd, atol=1e-7, rtol=1e-6)


def test_gradient_equals_torch_autograd():
    g = np.random.default_rng(1)
    n, d = 5, 6
    k, v = g.standard_normal((n, d)), g.standard_normal((n, d))
    W = g.standard_normal((d, d)) * 0.5
    gamma, beta = 1.0 + 0.3 * g.standard_normal(d), 0.2 * g.standard_normal(d)
    Wt = torch.tensor(W, requires_grad=True)
    kt, vt = torch.tensor(k), torch.tensor(v)
    for t in range(n):  # one token's loss at a time: its gradient is k_t^T e_t
        out = kt[t] + torch.nn.functional.layer_norm(kt[t] @ Wt, (d,), torch.tensor(gamma), torch.tensor(beta),
                                                     eps=LN_EPS)
        (gW,) = torch.autograd.grad(0.5 * ((out - vt[t]) ** 2).sum(), Wt)
        e = ln_residual_error(k[t][None], v[t][None], W, gamma, beta)[0]
        assert np.allclose(np.outer(k[t], e), gW.numpy(), atol=1e-12, rtol=1e-10)


def test_layer_norm_equals_torch():
    g = np.random.default_rng(2)
    y = g.standard_normal((7, 5)) * 3 + 1
    gamma, beta = g.standard_normal(5), g.standard_normal(5)
    want = torch.nn.functional.layer_norm(torch.tensor(y), (5,), torch.tensor(gamma), torch.tensor(beta), eps=LN_EPS)
    assert np.allclose(layer_norm(y, gamma, beta)[0], want.numpy(), atol=1e-12)


@pytest.mark.parametrize("T,b", [(9, 1), (9, 4), (12, 12), (10, 3)])
def test_primal_equals_dual(T, b):
    args = rand_case(2, 2, T, 4, seed=T + b)
    Zp, Wp = ln_residual_primal(*args, b)
    Zd, Wd = ln_residual_dual(*args, b)
    assert np.allclose(Zp, Zd, atol=1e-12) and np.allclose(Wp, Wd, atol=1e-12)


def test_primal_equals_torch_loop():
    """Per-token loop in torch fp64 with torch's layer_norm and autograd for every gradient."""
    Q, K, V, eta, W0, gamma, beta = rand_case(1, 1, 8, 3, seed=4)
    b = 3
    Z, Wo = ln_residual_primal(Q, K, V, eta, W0, gamma, beta, b)
    gm, bt = torch.tensor(gamma[0]), torch.tensor(beta[0])
    f = lambda x, W: x + torch.nn.functional.layer_norm(x @ W, (3,), gm, bt, eps=LN_EPS)
    W = torch.tensor(W0[0])
    for t in range(8):
        if t % b == 0:
            Wa = W.clone().requires_grad_(True)
        k, v, q = (torch.tensor(a[0, 0, t]) for a in (K, V, Q))
        (gW,) = torch.autograd.grad(0.5 * ((f(k, Wa) - v) ** 2).sum(), Wa)
        W = W - eta[0] * gW
        assert np.allclose(f(q, W).detach().numpy(), Z[0, 0, t], atol=1e-12)
    assert np.allclose(W.detach().numpy(), Wo[0, 0], atol=1e-12)


def test_eta_zero_is_the_normalised_forward():
    Q, K, V, _, W0, gamma, beta = rand_case(2, 2, 7, 4, seed=5)
    Z, Wo = ln_residual_primal(Q, K, V, np.zeros(2), W0, gamma, beta, 3)
    for h in range(2):
        assert np.allclose(Z[:, h], Q[:, h] + layer_norm(Q[:, h] @ W0[h], gamma[h], beta[h])[0], atol=1e-13)
        assert np.array_equal(Wo[:, h], np.broadcast_to(W0[h], Wo[:, h].shape))


def test_gamma_zero_leaves_w_untouched():
    """With gamma = 0, f(k) = k + beta does not depend on W: no gradient, and z = q + beta."""
    Q, K, V, eta, W0, _, beta = rand_case(1, 2, 6, 4, seed=6)
    Z, Wo = ln_residual_primal(Q, K, V, eta, W0, np.zeros((2, 4)), beta, 2)
    assert np.array_equal(Wo[0], W0)
    assert np.allclose(Z, Q + beta[None, :, None, :], atol=1e-15)


def test_planted_mistakes_are_caught():
    """Variants of the error with one plausible slip each must disagree with torch autograd."""
    g = np.random.default_rng(8)
    d = 5
    k, v = g.standard_normal(d), g.standard_normal(d)
    W = g.standard_normal((d, d)) * 0.5
    gamma, beta = 1.0 + 0.3 * g.standard_normal(d), 0.2 * g.standard_normal(d)
    Wt = torch.tensor(W, requires_grad=True)
    out = torch.tensor(k) + torch.nn.functional.layer_norm(torch.tensor(k) @ Wt, (d,), torch.tensor(gamma),
                                                           torch.tensor(beta), eps=LN_EPS)
    (gW,) = torch.autograd.grad(0.5 * ((out - torch.tensor(v)) ** 2).sum(), Wt)
    o, x, s = layer_norm(k @ W, gamma, beta)
    r = k + o - v
    slips = {
        "no mean of g": (gamma * r - x * (gamma * r * x).mean()) / s,
        "no x term": (gamma * r - (gamma * r).mean()) / s,
        "no residual": (gamma * (o - v) - (gamma * (o - v)).mean() - x * (gamma * (o - v) * x).mean()) / s,
        "no gamma": (r - r.mean() - x * (r * x).mean()) / s,
    }
    for name, e in slips.items():
        assert not np.allclose(np.outer(k, e), gW.numpy(), atol=1e-6), name


# ---------------------------------------------------------------------------- momentum
from oracle.variants import momentum_dual, momentum_primal  # noqa: E402

import oracle  # noqa: E402


def momentum_case(B, H, T, d, seed):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((B, H, T, d)) * 0.8 for _ in range(3))
    alpha = g.uniform(0.05, 0.3, H)
    beta = g.uniform(0.1, 0.95, H)
    W0 = g.standard_normal((H, d, d)) * 0.3
    return Q, K, V, alpha, beta, W0


@pytest.mark.parametrize("T,b", [(11, 1), (11, 3), (12, 4), (9, 9), (10, 16)])
def test_momentum_primal_equals_closed_form_dual(T, b):
    args = momentum_case(2, 2, T, 3, seed=T + b)
    for got, want in zip(momentum_primal(*args, b), momentum_dual(*args, b)):
        assert np.allclose(got, want, atol=1e-12)


@pytest.mark.parametrize("b", [1, 4, 7])
def test_momentum_without_momentum_is_ttt_linear(b):
    """beta = 0: the C oracle's TTT-Linear with eta = alpha, by both forms."""
    Q, K, V, alpha, _, W0 = momentum_case(2, 3, 13, 4, seed=b)
    Zr, Wr = oracle.linear_primal(Q, K, V, alpha, W0, b)
    for Z, W, M in (momentum_primal(Q, K, V, alpha, np.zeros(3), W0, b),
                    momentum_dual(Q, K, V, alpha, np.zeros(3), W0, b)):
        assert np.allclose(Z, Zr, atol=1e-12) and np.allclose(W, Wr, atol=1e-12)


def test_momentum_gradient_equals_torch_autograd():
    """b = 3: every gradient comes from autograd of 1/2 ||k W_a - v||^2 at the chunk-start W_a."""
    Q, K, V, alpha, beta, W0 = momentum_case(1, 1, 8, 3, seed=3)
    b = 3
    Z, Wo, Mo = momentum_primal(Q, K, V, alpha, beta, W0, b)
    W, M = torch.tensor(W0[0]), torch.zeros(3, 3, dtype=torch.float64)
    for t in range(8):
        if t % b == 0:
            Wa = W.clone().requires_grad_(True)
        k, v, q = (torch.tensor(x[0, 0, t]) for x in (K, V, Q))
        (g,) = torch.autograd.grad(0.5 * ((k @ Wa - v) ** 2).sum(), Wa)
        M = beta[0] * M + (1 - beta[0]) * g
        W = W - alpha[0] * M
        assert np.allclose((q @ W).numpy(), Z[0, 0, t], atol=1e-12)
    assert np.allclose(W.numpy(), Wo[0, 0], atol=1e-12) and np.allclose(M.numpy(), Mo[0, 0], atol=1e-12)


def test_momentum_with_zero_rate_reads_out_w0():
    Q, K, V, _, beta, W0 = momentum_case(1, 2, 7, 3, seed=4)
    Z, W, M = momentum_primal(Q, K, V, np.zeros(2), beta, W0, 3)
    assert np.array_equal(W[0], W0) and np.allclose(Z[0], np.einsum("htd,hde->hte", Q[0], W0), atol=1e-14)


# ---------------------------------------------------------------------------- bias
def _bias_case(B, H, T, d, seed):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((B, H, T, d)) * 0.7 for _ in range(3))
    return Q, K, V, g.uniform(0.05, 0.4, H), g.standard_normal((H, d, d)) * 0.3, g.standard_normal((H, d)) * 0.3


@pytest.mark.parametrize("T,b", [(13, 1), (17, 4), (20, 20)])
def test_bias_equals_c_oracle_on_a_constant_extra_input(T, b):
    import oracle
    from oracle.variants import bias_primal
    B, H, d = 2, 2, 5
    Q, K, V, eta, W0, beta0 = _bias_case(B, H, T, d, 70 + T + b)
    Z, W, be = bias_primal(Q, K, V, eta, W0, beta0, b)
    one, zero = np.ones((B, H, T, 1)), np.zeros((B, H, T, 1))
    W0x = np.zeros((H, d + 1, d + 1))
    W0x[:, :d, :d], W0x[:, d, :d] = W0, beta0
    Zx, Wx = oracle.linear_primal(np.concatenate([Q, one], 3), np.concatenate([K, one], 3),
                                  np.concatenate([V, zero], 3), eta, W0x, b)
    assert np.allclose(Zx[..., :d], Z, atol=1e-12)
    assert np.allclose(Wx[:, :, :d, :d], W, atol=1e-12) and np.allclose(Wx[:, :, d, :d], be, atol=1e-12)


def test_bias_gradient_equals_finite_differences():
    """One token, b = 1: the step taken equals -eta times the central-difference gradient of
    1/2 ||k W + beta - v||^2 with respect to W and beta."""
    from oracle.variants import bias_primal
    g = np.random.default_rng(3)
    d, eta = 4, 0.3
    q, k, v = (g.standard_normal(d) for _ in range(3))
    W, be = g.standard_normal((d, d)) * 0.4, g.standard_normal(d) * 0.4
    _, W1, b1 = bias_primal(q[None, None, None], k[None, None, None], v[None, None, None], np.array([eta]),
                            W[None], be[None], 1)
    f = lambda W_, b_: 0.5 * np.sum((k @ W_ + b_ - v) ** 2)
    h = 1e-6
    gW = np.zeros_like(W)
    for i in range(d):
        for j in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += h
            Wm[i, j] -= h
            gW[i, j] = (f(Wp, be) - f(Wm, be)) / (2 * h)
    gb = np.array([(f(W, be + h * np.eye(d)[j]) - f(W, be - h * np.eye(d)[j])) / (2 * h) for j in range(d)])
    assert np.allclose(W1[0, 0], W - eta * gW, atol=1e-8)
    assert np.allclose(b1[0, 0], be - eta * gb, atol=1e-8)


def test_bias_eta_zero_reads_out_the_initial_model():
    from oracle.variants import bias_primal
    Q, K, V, _, W0, beta0 = _bias_case(1, 2, 9, 4, 5)
    Z, W, be = bias_primal(Q, K, V, np.zeros(2), W0, beta0, 3)
    assert np.allclose(Z, np.einsum("nhti,hij->nhtj", Q, W0) + beta0[None, :, None, :], atol=1e-14)
    assert np.array_equal(W[0], W0) and np.array_equal(be[0], beta0)


# ---------------------------------------------------------------------------- per-token rate
@pytest.mark.parametrize("T,b", [(11, 1), (19, 4), (16, 16)])
def test_token_eta_equals_c_oracle_at_a_constant_rate(T, b):
    import oracle
    from oracle.variants import token_eta_primal
    B, H, d = 2, 3, 4
    Q, K, V, eta, W0, _ = _bias_case(B, H, T, d, 90 + T)
    et = np.broadcast_to(eta[None, :, None], (B, H, T)).copy()
    Z, W = token_eta_primal(Q, K, V, et, W0, b)
    Zr, Wr = oracle.linear_primal(Q, K, V, eta, W0, b)
    assert np.allclose(Z, Zr, atol=1e-12) and np.allclose(W, Wr, atol=1e-12)


def test_token_eta_equals_c_oracle_on_scaled_keys_and_values():
    import oracle
    from oracle.variants import token_eta_primal
    B, H, T, d, b = 2, 2, 23, 5, 4
    Q, K, V, _, W0, _ = _bias_case(B, H, T, d, 11)
    et = np.random.default_rng(12).uniform(0.0, 0.5, (B, H, T))
    Z, W = token_eta_primal(Q, K, V, et, W0, b)
    r = np.sqrt(et)[..., None]
    Zs, Ws = oracle.linear_primal(Q, r * K, r * V, np.ones(H), W0, b)
    assert np.allclose(Z, Zs, atol=1e-12) and np.allclose(W, Ws, atol=1e-12)


def test_token_eta_zero_reads_out_w0():
    from oracle.variants import token_eta_primal
    Q, K, V, _, W0, _ = _bias_case(1, 2, 7, 3, 13)
    Z, W = token_eta_primal(Q, K, V, np.zeros((1, 2, 7)), W0, 2)
    assert np.allclose(Z, np.einsum("nhti,hij->nhtj", Q, W0), atol=1e-14) and np.array_equal(W[0], W0)
