"""The oracle's backward of the TTT-Linear and TTT-MLP scans, pinned (CPU only).

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
differences by far more than their tolerance. mlp_backward is pinned the same
way: finite differences of the C TTT-MLP forward on every input, and torch
autograd (torch's own tanh-GELU and its derivatives) through a per-token loop.
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


# ---------------------------------------------------------------------------- TTT-MLP
from oracle.backward import mlp_backward  # noqa: E402


def rand_mlp(B, H, T, d, m, seed):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((B, H, T, d)) * 0.7 for _ in range(3))
    eta = g.uniform(0.05, 0.4, H)
    W1 = g.standard_normal((H, d, m)) * 0.4
    W2 = g.standard_normal((H, m, d)) * 0.4
    dZ = g.standard_normal((B, H, T, d))
    dW1 = g.standard_normal((B, H, d, m))
    dW2 = g.standard_normal((B, H, m, d))
    return Q, K, V, eta, W1, W2, dZ, dW1, dW2


def mlp_loss(Q, K, V, eta, W1, W2, b, dZ, dW1, dW2):
    Z, A1, A2 = oracle.mlp_primal(Q, K, V, eta, W1, W2, b)
    return float(np.sum(Z * dZ) + np.sum(A1 * dW1) + np.sum(A2 * dW2))


@pytest.mark.parametrize("B,H,T,d,m,b", [(1, 1, 6, 2, 5, 1), (1, 1, 6, 2, 5, 3), (1, 1, 6, 2, 5, 6),
                                         (2, 1, 5, 2, 3, 2)])
def test_mlp_backward_equals_finite_differences(B, H, T, d, m, b):
    args = rand_mlp(B, H, T, d, m, seed=T + b + m)
    Q, K, V, eta, W1, W2, dZ, dW1, dW2 = args
    got = mlp_backward(Q, K, V, eta, W1, W2, b, dZ, dW1, dW2)
    inputs = [Q, K, V, eta, W1, W2]
    for idx, (name, g) in enumerate(zip(("dQ", "dK", "dV", "deta", "dW1", "dW2"), got)):
        def f(x, idx=idx):
            xs = list(inputs)
            xs[idx] = x
            return mlp_loss(*xs, b, dZ, dW1, dW2)
        want = fd(f, inputs[idx])
        assert rel(g, want) < 1e-6, (name, rel(g, want))


def mlp_primal_torch(Q, K, V, eta, W1, W2, b):
    """Per-token TTT-MLP in torch fp64 with torch's own tanh-GELU: gradients at the
    chunk-start weights, read-out with the updated weights."""
    gelu = lambda x: torch.nn.functional.gelu(x, approximate="tanh")
    B, H, T, d = Q.shape
    Zs, W1s, W2s = [], [], []
    for n in range(B):
        zr, w1r, w2r = [], [], []
        for h in range(H):
            P1, P2 = W1[h], W2[h]
            zs = []
            for t in range(T):
                if t % b == 0:
                    A1, A2 = P1, P2
                u = K[n, h, t] @ A1
                a = gelu(u)
                gr = a @ A2 - V[n, h, t]
                # s'(u) by autograd, kept differentiable so that the outer gradient sees s''
                sprime = torch.autograd.functional.jacobian(gelu, u, create_graph=True).diagonal()
                dl = (gr @ A2.T) * sprime
                P1 = P1 - eta[h] * torch.outer(K[n, h, t], dl)
                P2 = P2 - eta[h] * torch.outer(a, gr)
                zs.append(gelu(Q[n, h, t] @ P1) @ P2)
            zr.append(torch.stack(zs))
            w1r.append(P1)
            w2r.append(P2)
        Zs.append(torch.stack(zr))
        W1s.append(torch.stack(w1r))
        W2s.append(torch.stack(w2r))
    return torch.stack(Zs), torch.stack(W1s), torch.stack(W2s)


def test_mlp_backward_equals_autograd():
    args = rand_mlp(1, 2, 5, 3, 4, seed=21)
    Q, K, V, eta, W1, W2, dZ, dW1, dW2 = args
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V, eta, W1, W2)]
    Z, A1, A2 = mlp_primal_torch(*ts, 2)
    L = (Z * torch.tensor(dZ)).sum() + (A1 * torch.tensor(dW1)).sum() + (A2 * torch.tensor(dW2)).sum()
    grads = torch.autograd.grad(L, ts)
    mine = mlp_backward(Q, K, V, eta, W1, W2, 2, dZ, dW1, dW2)
    for name, got, want in zip(("dQ", "dK", "dV", "deta", "dW1", "dW2"), mine, grads):
        assert rel(got, want.detach().numpy()) < 1e-10, (name, rel(got, want.detach().numpy()))
