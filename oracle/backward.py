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
