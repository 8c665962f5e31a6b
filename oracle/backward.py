"""ORACLE: backward of the chunked TTT-Linear scan in fp64 (test infrastructure).

Only the tests may import this module; the CUDA library never loads it and
shares no code with it.

What it computes. The scan's outputs, Z and the final state W_out, depend on
Q, K, V, the per-head learning rate eta and the initial state W0. The outer
loop trains the projections that make Q, K, V, and W0 itself, by backpropagating
through the inner loop ("5 · TestingTime 训练与长上下文", section 2.2: W0 and the
projections are outer-loop parameters). Given upstream gradients dZ and dW_out,
this returns the vector-Jacobian products dQ, dK, dV, deta and dW0.

The forward is the chunk rule of section 1.1 of the same page (gradients of the
whole chunk taken at the chunk-start weights), written per chunk c with
chunk-start state W as
    E  = K_c W - V_c
    S  = tril(Q_c K_c^T)        (diagonal kept: update-then-read)
    Z_c = Q_c W - eta S E
    W' = W - eta K_c^T E
and the backward reverses it chunk by chunk from G = dW_out. With G the gradient
of the next chunk's start state:
    dE  = -eta K_c G - eta S^T dZ_c            dW = G + Q_c^T dZ_c + K_c^T dE
    dS  = tril(-eta dZ_c E^T)                  dQ_c = dZ_c W^T + dS K_c
    dK_c = -eta E G^T + dS^T Q_c + dE W^T      dV_c = -dE
    deta += -sum(K_c^T E * G) - sum(S E * dZ_c)
and G <- dW for the chunk before. dW0 is the last G. This is the product rule
applied to the four lines above, each term written out; numpy's matrix product
is the only library step. Chunk-start states come from a forward pass kept in
memory, so this is for small cases only.

Pins (tests/test_oracle_backward.py): central finite differences of the
oracle's own primal forward on tiny inputs for every input; torch autograd
through a per-token primal loop; eta = 0 in closed form; a planted dropped term
is caught.

mlp_backward does the same for TTT-MLP ("Test-Time Training (TTT) guide",
section 3: two layers, hidden 4x, GELU), whose chunk step in dual form is
    U = K_c W1, A = s(U), G = A W2 - V_c, D = (G W2^T) * s'(U),
    Hq = Q_c W1 - eta tril(Q_c K_c^T) D, Aq = s(Hq),
    Z_c = Aq W2 - eta tril(Aq A^T) G,
    W1' = W1 - eta K_c^T D,   W2' = W2 - eta A^T G,
with s the tanh-GELU. D depends on U through s'(U), so the backward needs s''.
Each line is reversed in turn, last line first, with the product rule.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def linear_backward(Q, K, V, eta, W0, b: int, dZ, dW_out):
    """Vector-Jacobian product of the chunked TTT-Linear scan.

    Q, K, V, dZ [B,H,T,d]; eta [H]; W0 [H,d,d]; dW_out [B,H,d,d].
    Returns (dQ, dK, dV [B,H,T,d], deta [H], dW0 [H,d,d]) in fp64; deta and dW0
    are summed over the batch rows (W0 and eta are shared by them)."""
    Q, K, V, eta, W0, dZ, dW_out = map(_f64, (Q, K, V, eta, W0, dZ, dW_out))
    B, H, T, d = Q.shape
    if b < 1:
        raise ValueError("b must be positive")
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    deta = np.zeros(H)
    dW0 = np.zeros((H, d, d))
    bounds = [(c0, min(c0 + b, T)) for c0 in range(0, T, b)]
    for n in range(B):
        for h in range(H):
            e = eta[h]
            # forward: the chunk-start states
            starts = []
            W = W0[h].copy()
            for c0, c1 in bounds:
                starts.append(W.copy())
                E = K[n, h, c0:c1] @ W - V[n, h, c0:c1]
                W = W - e * K[n, h, c0:c1].T @ E
            # backward, last chunk first
            G = dW_out[n, h].copy()
            for (c0, c1), W in zip(reversed(bounds), reversed(starts)):
                Qc, Kc, Vc, dZc = Q[n, h, c0:c1], K[n, h, c0:c1], V[n, h, c0:c1], dZ[n, h, c0:c1]
                E = Kc @ W - Vc
                S = np.tril(Qc @ Kc.T)
                # W' = W - eta Kc^T E
                dE = -e * (Kc @ G)
                dKc = -e * (E @ G.T)
                deta[h] -= np.sum((Kc.T @ E) * G)
                dW = G.copy()
                # Z = Qc W - eta S E
                dQc = dZc @ W.T
                dW += Qc.T @ dZc
                dS = np.tril(-e * (dZc @ E.T))
                dE += -e * (S.T @ dZc)
                deta[h] -= np.sum((S @ E) * dZc)
                dQc += dS @ Kc
                dKc += dS.T @ Qc
                # E = Kc W - Vc
                dKc += dE @ W.T
                dW += Kc.T @ dE
                dQ[n, h, c0:c1] = dQc
                dK[n, h, c0:c1] = dKc
                dV[n, h, c0:c1] = -dE
                G = dW
            dW0[h] += G
    return dQ, dK, dV, deta, dW0


_GELU_C = np.sqrt(2.0 / np.pi)
_GELU_A = 0.044715


def _gelu_parts(u):
    """tanh-GELU s(u) = u (1 + th) / 2 with th = tanh(c (u + a u^3)), and its first
    and second derivatives, from the product and chain rules."""
    k = _GELU_C * (1.0 + 3.0 * _GELU_A * u * u)        # d/du of c (u + a u^3)
    th = np.tanh(_GELU_C * (u + _GELU_A * u ** 3))
    th1 = (1.0 - th * th) * k                         # d th / du
    th2 = -2.0 * th * th1 * k + (1.0 - th * th) * 6.0 * _GELU_A * _GELU_C * u
    s = 0.5 * u * (1.0 + th)
    s1 = 0.5 * (1.0 + th) + 0.5 * u * th1
    s2 = th1 + 0.5 * u * th2
    return s, s1, s2


def mlp_backward(Q, K, V, eta, W1, W2, b: int, dZ, dW1_out, dW2_out):
    """Vector-Jacobian product of the chunked TTT-MLP scan.

    Q, K, V, dZ [B,H,T,d]; eta [H]; W1 [H,d,m]; W2 [H,m,d]; dW1_out [B,H,d,m];
    dW2_out [B,H,m,d]. Returns (dQ, dK, dV [B,H,T,d], deta [H], dW1 [H,d,m],
    dW2 [H,m,d]) in fp64; deta, dW1 and dW2 are summed over the batch rows."""
    Q, K, V, eta, W1, W2, dZ, dW1_out, dW2_out = map(_f64, (Q, K, V, eta, W1, W2, dZ, dW1_out, dW2_out))
    B, H, T, d = Q.shape
    if b < 1:
        raise ValueError("b must be positive")
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    deta = np.zeros(H)
    dW1s, dW2s = np.zeros_like(W1), np.zeros_like(W2)
    bounds = [(c0, min(c0 + b, T)) for c0 in range(0, T, b)]
    for n in range(B):
        for h in range(H):
            e = eta[h]
            starts = []
            P1, P2 = W1[h].copy(), W2[h].copy()
            for c0, c1 in bounds:
                starts.append((P1.copy(), P2.copy()))
                Kc, Vc = K[n, h, c0:c1], V[n, h, c0:c1]
                U = Kc @ P1
                A, s1, _ = _gelu_parts(U)
                G = A @ P2 - Vc
                D = (G @ P2.T) * s1
                P1 = P1 - e * Kc.T @ D
                P2 = P2 - e * A.T @ G
            G1, G2 = dW1_out[n, h].copy(), dW2_out[n, h].copy()
            for (c0, c1), (P1, P2) in zip(reversed(bounds), reversed(starts)):
                Qc, Kc, Vc, dZc = Q[n, h, c0:c1], K[n, h, c0:c1], V[n, h, c0:c1], dZ[n, h, c0:c1]
                # forward of the chunk
                U = Kc @ P1
                A, s1, s2 = _gelu_parts(U)
                G = A @ P2 - Vc
                D1 = G @ P2.T
                D = D1 * s1
                S = np.tril(Qc @ Kc.T)
                Hq = Qc @ P1 - e * S @ D
                Aq, sq1, _ = _gelu_parts(Hq)
                R = np.tril(Aq @ A.T)
                # W1' = P1 - eta Kc^T D,  W2' = P2 - eta A^T G
                dP1, dP2 = G1.copy(), G2.copy()
                dK_ = -e * (D @ G1.T)
                dD = -e * (Kc @ G1)
                dA = -e * (G @ G2.T)
                dG = -e * (A @ G2)
                deta[h] -= np.sum((Kc.T @ D) * G1) + np.sum((A.T @ G) * G2)
                # Z = Aq P2 - eta R G
                dAq = dZc @ P2.T
                dP2 += Aq.T @ dZc
                dR = np.tril(-e * (dZc @ G.T))
                dG += -e * (R.T @ dZc)
                deta[h] -= np.sum((R @ G) * dZc)
                # R = tril(Aq A^T)
                dAq += dR @ A
                dA += dR.T @ Aq
                # Aq = s(Hq)
                dHq = dAq * sq1
                # Hq = Qc P1 - eta S D
                dQ_ = dHq @ P1.T
                dP1 += Qc.T @ dHq
                dS = np.tril(-e * (dHq @ D.T))
                dD += -e * (S.T @ dHq)
                deta[h] -= np.sum((S @ D) * dHq)
                # S = tril(Qc Kc^T)
                dQ_ += dS @ Kc
                dK_ += dS.T @ Qc
                # D = D1 * s'(U),  D1 = G P2^T
                dD1 = dD * s1
                dU = dD * D1 * s2
                dG += dD1 @ P2
                dP2 += dD1.T @ G
                # G = A P2 - Vc
                dV[n, h, c0:c1] = -dG
                dA += dG @ P2.T
                dP2 += A.T @ dG
                # A = s(U),  U = Kc P1
                dU += dA * s1
                dK_ += dU @ P1.T
                dP1 += Kc.T @ dU
                dQ[n, h, c0:c1] = dQ_
                dK[n, h, c0:c1] = dK_
                G1, G2 = dP1, dP2
            dW1s[h] += G1
            dW2s[h] += G2
    return dQ, dK, dV, deta, dW1s, dW2s
