"""ORACLE: inner-model variants of TTT-Linear in fp64 (test infrastructure).

Only the tests may import this module; the CUDA library never loads it and
shares no code with it.

Layer norm and a residual inside f. The ablation ladder of "5 · TestingTime
训练与长上下文" (section 3.1) adds, step by step to linear attention, a
learnable W0, a layer norm and a residual inside the inner model f, mini-batch
updates and a learnable learning rate. The page gives no formula for the
normalised f. This module takes the plainest reading:

    f(k; W) = k + LN(k W),   LN(y) = gamma * (y - mean(y)) / sqrt(var(y) + eps) + beta,

with mean and (biased) variance over the d features of one token, per-head
gamma and beta (outer-loop parameters, fixed within the sequence) and
eps = 1e-6. The inner loss is 1/2 ||f(k; W) - v||^2 and the update is the same
chunk rule as plain TTT-Linear (section 1.1 of the same page: every gradient
of a chunk is taken at the chunk-start weights); the output is
z_t = f(q_t; W_t) with the weights after token t's own gradient.

The gradient with respect to W of one token's loss is k^T e, where, writing
y = k W, s = sqrt(var(y) + eps), x = (y - mean(y)) / s and r = f(k; W) - v,
    g = gamma * r,    e = (g - mean(g) - x * mean(g * x)) / s
(the chain rule through the normalisation: the two means remove the components
of g along the constant vector and along x, to which a normalised vector is
insensitive).

Two forms are given, for the same reason as for plain TTT-Linear:
  - ln_residual_primal: token by token (gradient at the chunk-start W, update,
    then read out);
  - ln_residual_dual: chunk by chunk, E from the chunk-start W, then
    X = Q Wa - eta tril(Q K^T) E and Z = Q + LN(X), W = Wa - eta K^T E.
Pins (tests/test_oracle_variants.py): the gradient against central finite
differences of the loss and against torch autograd through torch's own
layer_norm; primal equals dual; eta = 0 and gamma = 0 in closed form.
"""
from __future__ import annotations

import numpy as np

LN_EPS = 1e-6


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def layer_norm(y, gamma, beta, eps: float = LN_EPS):
    """LN over the last axis; returns (LN(y), x, s) with x the normalised y and s the scale."""
    mu = y.mean(axis=-1, keepdims=True)
    s = np.sqrt(((y - mu) ** 2).mean(axis=-1, keepdims=True) + eps)
    x = (y - mu) / s
    return gamma * x + beta, x, s


def ln_residual_error(k, v, W, gamma, beta, eps: float = LN_EPS):
    """e with grad_W 1/2 ||k + LN(k W) - v||^2 = k^T e, for the rows of k and v at once."""
    o, x, s = layer_norm(k @ W, gamma, beta, eps)
    g = gamma * (k + o - v)
    return (g - g.mean(axis=-1, keepdims=True) - x * (g * x).mean(axis=-1, keepdims=True)) / s


def _check(Q, K, V, eta, W0, gamma, beta, b):
    Q, K, V, eta, W0, gamma, beta = map(_f64, (Q, K, V, eta, W0, gamma, beta))
    B, H, T, d = Q.shape
    assert K.shape == Q.shape and V.shape == Q.shape
    assert eta.shape == (H,) and W0.shape == (H, d, d) and gamma.shape == (H, d) and beta.shape == (H, d)
    if b < 1:
        raise ValueError("b must be positive")
    return Q, K, V, eta, W0, gamma, beta


def ln_residual_primal(Q, K, V, eta, W0, gamma, beta, b: int):
    """TTT-Linear with f(k) = k + LN(k W), token by token.

    Q, K, V [B,H,T,d]; eta [H]; W0 [H,d,d]; gamma, beta [H,d]. Returns Z [B,H,T,d]
    and the final W [B,H,d,d], fp64."""
    Q, K, V, eta, W0, gamma, beta = _check(Q, K, V, eta, W0, gamma, beta, b)
    B, H, T, d = Q.shape
    Z = np.zeros_like(Q)
    W_out = np.zeros((B, H, d, d))
    for n in range(B):
        for h in range(H):
            W = W0[h].copy()
            Wa = W
            for t in range(T):
                if t % b == 0:
                    Wa = W.copy()
                e = ln_residual_error(K[n, h, t][None], V[n, h, t][None], Wa, gamma[h], beta[h])[0]
                W = W - eta[h] * np.outer(K[n, h, t], e)
                Z[n, h, t] = Q[n, h, t] + layer_norm(Q[n, h, t] @ W, gamma[h], beta[h])[0]
            W_out[n, h] = W
    return Z, W_out


def ln_residual_dual(Q, K, V, eta, W0, gamma, beta, b: int):
    """The same layer chunk by chunk in dual form (see the module docstring)."""
    Q, K, V, eta, W0, gamma, beta = _check(Q, K, V, eta, W0, gamma, beta, b)
    B, H, T, d = Q.shape
    Z = np.zeros_like(Q)
    W_out = np.zeros((B, H, d, d))
    for n in range(B):
        for h in range(H):
            W = W0[h].copy()
            for c0 in range(0, T, b):
                Qc, Kc, Vc = Q[n, h, c0:c0 + b], K[n, h, c0:c0 + b], V[n, h, c0:c0 + b]
                E = ln_residual_error(Kc, Vc, W, gamma[h], beta[h])
                X = Qc @ W - eta[h] * np.tril(Qc @ Kc.T) @ E
                Z[n, h, c0:c0 + b] = Qc + layer_norm(X, gamma[h], beta[h])[0]
                W = W - eta[h] * Kc.T @ E
            W_out[n, h] = W
    return Z, W_out
