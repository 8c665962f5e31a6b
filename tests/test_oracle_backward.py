"""The oracle's backward of the TTT-Linear scan, pinned (CPU only).

linear_backward returns the vector-Jacobian product of (Z, W_out) with respect
to (Q, K, V, eta, W0). It is checked against:
  - central finite differences of the oracle's own per-token primal forward
    (the C code), for every input entry, with chunks of 1, 2, 3 and T tokens
    and with batch rows sharing eta and W0;
  - torch autograd through a per-token primal loop written with torch ops;
  - eta = 0, where the scan is Z = Q W0, W_out = W0 and the products are known
    in closed form.
Every term of the backward feeds some entry of some gradient at random inputs,
so a dropped term, a wrong sign or a transposed factor fails the finite
differences by far more than their tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import linear_backward


def rand_case(B, H, T, d, seed):
    g = np.random.default_rng(seed)
    Q = g.standard_normal((B, H, T, d)) * 0.7
    K = g.standard_normal((B, H, T, d)) * 0.7
    V = g.standard_normal((B, H, T, d))
    eta = g.uniform(0.05, 0.4, H)
    W0 = g.standard_normal((H, d, d)) * 0.3
    dZ = g.standard_normal((B, H, T, d))
    dW = g.standard_normal((B, H, d, d))
    return Q, K, V, eta, W0, dZ, dW


def loss(Q, K, V, eta, W0, b, dZ, dW):
    Z, Wo = oracle.linear_primal(Q, K, V, eta, W0, b)
    return float(np.sum(Z * dZ) + np.sum(Wo * dW))


def fd(f, x, h=1e-6):
    """Central differences of the scalar f at every entry of x."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


def rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


@pytest.mark.parametrize("B,H,T,d,b", [(1, 1, 7, 3, 1), (1, 1, 7, 3, 2), (1, 1, 7, 3, 3), (1, 1, 7, 3, 7),
                                       (2, 2, 6, 2, 4)])
def test_backward_equals_finite_differences(B, H, T, d, b):
    Q, K, V, eta, W0, dZ, dW = rand_case(B, H, T, d, seed=10 * T + b + B)
    dQ, dK, dV, deta, dW0 = linear_backward(Q, K, V, eta, W0, b, dZ, dW)
    fQ = fd(lambda x: loss(x, K, V, eta, W0, b, dZ, dW), Q)
    fK = fd(lambda x: loss(Q, x, V, eta, W0, b, dZ, dW), K)
    fV = fd(lambda x: loss(Q, K, x, eta, W0, b, dZ, dW), V)
    fe = fd(lambda x: loss(Q, K, V, x, W0, b, dZ, dW), eta)
    fW = fd(lambda x: loss(Q, K, V, eta, x, b, dZ, dW), W0)
    for name, got, want in (("dQ", dQ, fQ), ("dK", dK, fK), ("dV", dV, fV), ("deta", deta, fe), ("dW0", dW0, fW)):
        assert rel(got, want) < 1e-6, (name, rel(got, want))


def primal_torch(Q, K, V, eta, W0, b):
    """Per-token primal loop in torch fp64: each token's gradient at the chunk-start
    weights, then its read-out with the updated weights."""
    B, H, T, d = Q.shape
    Zs, Ws = [], []
    for n in range(B):
        zr, wr = [], []
        for h in range(H):
            W = W0[h]
            zs = []
            for t in range(T):
                if t % b == 0:
                    Wa = W
                e = K[n, h, t] @ Wa - V[n, h, t]
                W = W - eta[h] * torch.outer(K[n, h, t], e)
                zs.append(Q[n, h, t] @ W)
            zr.append(torch.stack(zs))
            wr.append(W)
        Zs.append(torch.stack(zr))
        Ws.append(torch.stack(wr))
    return torch.stack(Zs), torch.stack(Ws)


@pytest.mark.parametrize("T,b", [(9, 1), (9, 4), (12, 12)])
def test_backward_equals_autograd(T, b):
    Q, K, V, eta, W0, dZ, dW = rand_case(2, 2, T, 4, seed=T + b)
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V, eta, W0)]
    Z, Wo = primal_torch(*ts, b)
    L = (Z * torch.tensor(dZ)).sum() + (Wo * torch.tensor(dW)).sum()
    grads = torch.autograd.grad(L, ts)
    mine = linear_backward(Q, K, V, eta, W0, b, dZ, dW)
    for name, got, want in zip(("dQ", "dK", "dV", "deta", "dW0"), mine, grads):
        assert rel(got, want.numpy()) < 1e-12, (name, rel(got, want.numpy()))


def test_backward_eta_zero_closed_form():
    Q, K, V, _, W0, dZ, dW = rand_case(2, 3, 10, 4, seed=5)
    eta = np.zeros(3)
    dQ, dK, dV, _, dW0 = linear_backward(Q, K, V, eta, W0, 4, dZ, dW)
    # Z = Q W0 and W_out = W0: dQ = dZ W0^T; K and V do not enter; dW0 = sum_n (Q^T dZ + dW_out)
    assert np.allclose(dQ, np.einsum("nhtj,hij->nhti", dZ, W0), atol=1e-13)
    assert np.array_equal(dK, np.zeros_like(dK)) and np.array_equal(dV, np.zeros_like(dV))
    want = np.einsum("nhti,nhtj->hij", Q, dZ) + dW.sum(0)
    assert np.allclose(dW0, want, atol=1e-12)
