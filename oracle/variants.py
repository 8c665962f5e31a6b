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

Momentum. momentum_primal and momentum_dual hold the E²-TTT-style variant
(momentum gradient descent with chunk-start gradients); see momentum_primal.

Bias. "Test-Time Training (TTT) guide" (section 3) writes the linear inner
model with a bias, f(W, x) = W x + b. bias_primal trains (W, beta) together by
the same chunk rule on 1/2 ||k W + beta - v||^2 (row vectors): the gradient of
one token is (k^T e, e) with e = k W_a + beta_a - v at the chunk-start
weights, and the read-out is z_t = q_t W_t + beta_t.

Per-token learning rate. The ablation ladder of "5 · TestingTime 训练与长上下文"
(section 3.1) names a learnable learning rate. token_eta_primal reads it as a
rate eta_t per token (per batch row and head) that scales that token's gradient
in the chunk rule: W <- W - eta_t k_t^T (k_t W_a - v_t), read-out q_t W_t.
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


# ---------------------------------------------------------------------------- momentum
def momentum_primal(Q, K, V, alpha, beta, W0, b: int):
    """TTT-Linear with momentum gradient descent, token by token.

    "推理时的“临阵磨枪”：Test-Time Training如何教会AI“边做边学”" (zhichai),
    sections 2.3 and 5.1, describes E²-TTT: it keeps a momentum state M
    beside the fast weights W, takes every gradient at the chunk-start weights,
    and says the chunk's state then follows exactly from a recurrence; its
    displayed per-chunk update leaves the function f undefined. The reading here
    is momentum gradient descent at token level with those chunk-start gradients:
    for chunk c with start state W_a, and for each of its tokens t in order,
        g_t = k_t^T (k_t W_a - v_t),   M <- beta M + (1 - beta) g_t,   W <- W - alpha M,
    then z_t = q_t W. M starts at zero for every sequence. With beta = 0 this is
    the TTT-Linear chunk rule with eta = alpha. (The displayed per-chunk
    formula, read literally, would instead take one momentum step per chunk.)
    Parity with the page's own method is unpinned: the page gives neither f nor
    a read-out, nor any worked value. The pins hold this reading to the
    mathematics: beta = 0 against the C oracle's TTT-Linear, the gradient
    against torch autograd, and the primal against the closed-form dual.

    Q, K, V [B,H,T,d]; alpha, beta [H]. W0 [H,d,d]. Returns Z [B,H,T,d] and the
    final W and M [B,H,d,d], fp64."""
    Q, K, V, alpha, beta, W0 = map(_f64, (Q, K, V, alpha, beta, W0))
    B, H, T, d = Q.shape
    if b < 1:
        raise ValueError("b must be positive")
    Z = np.zeros_like(Q)
    W_out, M_out = np.zeros((B, H, d, d)), np.zeros((B, H, d, d))
    for n in range(B):
        for h in range(H):
            W, M = W0[h].copy(), np.zeros((d, d))
            Wa = W
            for t in range(T):
                if t % b == 0:
                    Wa = W.copy()
                g = np.outer(K[n, h, t], K[n, h, t] @ Wa - V[n, h, t])
                M = beta[h] * M + (1.0 - beta[h]) * g
                W = W - alpha[h] * M
                Z[n, h, t] = Q[n, h, t] @ W
            W_out[n, h], M_out[n, h] = W, M
    return Z, W_out, M_out


def momentum_dual(Q, K, V, alpha, beta, W0, b: int):
    """The same layer chunk by chunk, from the recurrence solved in closed form.

    Within a chunk with start (W_a, M_a) and errors E = K W_a - V, after its s-th
    token (s = 1, 2, ...)
        M_s = beta^s M_a + (1 - beta) sum_{i<=s} beta^(s-i) k_i^T e_i,
        W_s = W_a - alpha [c_s M_a + sum_{i<=s} (1 - beta^(s-i+1)) k_i^T e_i],
    with c_s = beta + beta^2 + ... + beta^s. So the read-out is a decay-masked
    dual form, Z = Q W_a - alpha c * (Q M_a) - alpha (tril(Q K^T) * D) E with
    D[s][i] = 1 - beta^(s-i+1), and the chunk's end state is the last row."""
    Q, K, V, alpha, beta, W0 = map(_f64, (Q, K, V, alpha, beta, W0))
    B, H, T, d = Q.shape
    if b < 1:
        raise ValueError("b must be positive")
    Z = np.zeros_like(Q)
    W_out, M_out = np.zeros((B, H, d, d)), np.zeros((B, H, d, d))
    for n in range(B):
        for h in range(H):
            a, be = alpha[h], beta[h]
            W, M = W0[h].copy(), np.zeros((d, d))
            for c0 in range(0, T, b):
                Qc, Kc, Vc = Q[n, h, c0:c0 + b], K[n, h, c0:c0 + b], V[n, h, c0:c0 + b]
                C = len(Kc)
                s = np.arange(1, C + 1)
                E = Kc @ W - Vc
                cs = np.cumsum(be ** s)                                     # c_s
                D = np.tril(1.0 - be ** np.maximum(s[:, None] - s[None, :] + 1, 1))  # 1 - beta^(s-i+1), i <= s
                Z[n, h, c0:c0 + C] = Qc @ W - a * cs[:, None] * (Qc @ M) - a * (np.tril(Qc @ Kc.T) * D) @ E
                G = Kc.T @ (E * (be ** (C - s))[:, None])                   # sum_i beta^(C-i) k_i^T e_i
                W_new = W - a * (cs[-1] * M + Kc.T @ (E * D[-1][:, None]))
                M = be ** C * M + (1.0 - be) * G
                W = W_new
            W_out[n, h], M_out[n, h] = W, M
    return Z, W_out, M_out


# ---------------------------------------------------------------------------- bias
def bias_primal(Q, K, V, eta, W0, beta0, b: int):
    """TTT-Linear with a bias, f(k) = k W + beta, token by token (see the module
    docstring). Q, K, V [B,H,T,d]; eta [H]; W0 [H,d,d]; beta0 [H,d] (shared by the
    batch rows, like W0). Returns Z [B,H,T,d], the final W [B,H,d,d] and beta [B,H,d]."""
    Q, K, V, eta, W0, beta0 = map(_f64, (Q, K, V, eta, W0, beta0))
    B, H, T, d = Q.shape
    if b < 1:
        raise ValueError("b must be positive")
    Z = np.zeros_like(Q)
    W_out, beta_out = np.zeros((B, H, d, d)), np.zeros((B, H, d))
    for n in range(B):
        for h in range(H):
            W, be = W0[h].copy(), beta0[h].copy()
            Wa, ba = W, be
            for t in range(T):
                if t % b == 0:
                    Wa, ba = W.copy(), be.copy()
                e = K[n, h, t] @ Wa + ba - V[n, h, t]
                W = W - eta[h] * np.outer(K[n, h, t], e)
                be = be - eta[h] * e
                Z[n, h, t] = Q[n, h, t] @ W + be
            W_out[n, h], beta_out[n, h] = W, be
    return Z, W_out, beta_out


# ---------------------------------------------------------------------------- per-token rate
def token_eta_primal(Q, K, V, eta_t, W0, b: int):
    """TTT-Linear with a learning rate per token, token by token (see the module
    docstring). Q, K, V [B,H,T,d]; eta_t [B,H,T]; W0 [H,d,d]. Returns Z [B,H,T,d]
    and the final W [B,H,d,d]."""
    Q, K, V, eta_t, W0 = map(_f64, (Q, K, V, eta_t, W0))
    B, H, T, d = Q.shape
    assert eta_t.shape == (B, H, T)
    if b < 1:
        raise ValueError("b must be positive")
    Z = np.zeros_like(Q)
    W_out = np.zeros((B, H, d, d))
    for n in range(B):
        for h in range(H):
            W = W0[h].copy()
            Wa = W
            for t in range(T):
                if t % b == 0:
                    Wa = W.copy()
                W = W - eta_t[n, h, t] * np.outer(K[n, h, t], K[n, h, t] @ Wa - V[n, h, t])
                Z[n, h, t] = Q[n, h, t] @ W
            W_out[n, h] = W
    return Z, W_out
