"""The fp64 oracle pinned to what the pages and the mathematics fix (CPU only).

Each pin checks the oracle against something other than itself:
  - exact rational arithmetic of the delta rule (b = 1) and of causal linear
    attention (W0 = 0, one chunk);
  - finite differences and torch autograd (with torch's own tanh-GELU) for the
    gradient of 1/2 ||f(k) - v||^2 taken at the chunk-start weights;
  - the single closed form of one chunk, the eta = 0 forward, chaining,
    batch-row independence, and hand-worked examples in tests/golden/;
  - the segment affine maps against the per-token scan at every segment end,
    and a one-token map by hand in exact rationals.
A plausible slip (a dropped 1/2, a wrong sign, read-before-write, a gradient at
the running instead of the chunk-start weights, a transposed W) fails at least
one of them: test_planted_mistakes_are_caught plants each in a copy of the
per-token rule and checks that the pins would see it.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def rand_linear(B, H, T, d, w_std=0.3, eta_lo=0.05, eta_hi=0.5, seed=0):
    g = np.random.default_rng(seed)
    Q = g.standard_normal((B, H, T, d))
    K = g.standard_normal((B, H, T, d))
    K /= np.linalg.norm(K, axis=-1, keepdims=True)
    Q /= np.linalg.norm(Q, axis=-1, keepdims=True)
    V = g.standard_normal((B, H, T, d))
    eta = g.uniform(eta_lo, eta_hi, H)
    W0 = w_std * g.standard_normal((H, d, d))
    return Q, K, V, eta, W0


def rand_mlp(B, H, T, d, m, w_std=0.3, seed=0):
    Q, K, V, eta, _ = rand_linear(B, H, T, d, seed=seed)
    g = np.random.default_rng(seed + 1)
    W1 = w_std * g.standard_normal((H, d, m))
    W2 = w_std * g.standard_normal((H, m, d))
    return Q, K, V, eta, W1, W2


# ---------------------------------------------------------------- P1: delta rule
def _delta_rule_exact(q, k, v, beta, S0):
    """DeltaNet write rule in the pages' column-vector form, exact rationals:
    S_t = S_{t-1} (I - beta k_t k_t^T) + beta v_t k_t^T, read o_t = S_t q_t
    ('5 · TestingTime 训练与长上下文' sec. 2.1). S = W^T in row-vector terms."""
    d = len(k[0])
    S = [[Fraction(S0[r][c]) for c in range(d)] for r in range(d)]
    outs = []
    for t in range(len(k)):
        kt = [Fraction(x) for x in k[t]]
        vt = [Fraction(x) for x in v[t]]
        Sk = [sum(S[r][c] * kt[c] for c in range(d)) for r in range(d)]
        S = [[S[r][c] - beta * Sk[r] * kt[c] + beta * vt[r] * kt[c] for c in range(d)]
             for r in range(d)]
        outs.append([sum(S[r][c] * Fraction(q[t][c]) for c in range(d)) for r in range(d)])
    return outs, S


@pytest.mark.parametrize("T,d", [(6, 3), (5, 4)])
def test_b1_equals_delta_rule_exactly(T, d):
    g = np.random.default_rng(T * 10 + d)
    # dyadic inputs with few bits: every product and sum below is exact in fp64
    k = g.integers(-2, 3, (T, d)) / 2.0
    v = g.integers(-3, 4, (T, d)).astype(float)
    q = g.integers(-2, 3, (T, d)) / 2.0
    W0 = g.integers(-2, 3, (d, d)) / 4.0
    eta = 0.25
    Z, W = oracle.linear_primal(q[None, None], k[None, None], v[None, None], [eta], W0[None], b=1)
    outs, S = _delta_rule_exact(q.tolist(), k.tolist(), v.tolist(), Fraction(1, 4), W0.T.tolist())
    assert np.array_equal(Z[0, 0], np.array([[float(x) for x in o] for o in outs]))
    assert np.array_equal(W[0, 0].T, np.array([[float(x) for x in r] for r in S]))
    Zd, Wd = oracle.linear_dual(q[None, None], k[None, None], v[None, None], [eta], W0[None], b=1)
    assert np.array_equal(Zd, Z) and np.array_equal(Wd, W)


# ---------------------------------------------------- P2: causal linear attention
def test_w0_zero_one_chunk_is_causal_linear_attention_exactly():
    g = np.random.default_rng(7)
    T, d = 7, 3
    q = g.integers(-3, 4, (T, d)).tolist()
    k = g.integers(-3, 4, (T, d)).tolist()
    v = g.integers(-3, 4, (T, d)).tolist()
    eta = Fraction(1, 8)
    # z_t = eta sum_{i<=t} (q_t . k_i) v_i  and  W_out = eta K^T V
    Zx = [[eta * sum(sum(Fraction(q[t][c]) * k[i][c] for c in range(d)) * v[i][j]
                     for i in range(t + 1)) for j in range(d)] for t in range(T)]
    Wx = [[eta * sum(Fraction(k[t][a]) * v[t][c] for t in range(T)) for c in range(d)]
          for a in range(d)]
    args = (np.array(q, float)[None, None], np.array(k, float)[None, None],
            np.array(v, float)[None, None], [0.125], np.zeros((1, d, d)))
    for fn in (oracle.linear_primal, oracle.linear_dual):
        Z, W = fn(*args, b=T)
        assert np.array_equal(Z[0, 0], np.array(Zx, dtype=float))
        assert np.array_equal(W[0, 0], np.array(Wx, dtype=float))
        # any b >= T is one chunk too
        Z2, W2 = fn(*args, b=T + 5)
        assert np.array_equal(Z2, Z) and np.array_equal(W2, W)


def test_causal_linear_attention_random():
    Q, K, V, eta, _ = rand_linear(2, 3, 33, 8)
    W0 = np.zeros((3, 8, 8))
    Z, W = oracle.linear_primal(Q, K, V, eta, W0, b=33)
    for n in range(2):
        for h in range(3):
            A = np.tril(Q[n, h] @ K[n, h].T)
            assert rel(Z[n, h], eta[h] * A @ V[n, h]) < 1e-13
            assert rel(W[n, h], eta[h] * K[n, h].T @ V[n, h]) < 1e-13


# -------------------------------------------------- P8: one chunk, closed form
def test_one_chunk_closed_form_with_w0():
    Q, K, V, eta, W0 = rand_linear(1, 2, 16, 8)
    Z, W = oracle.linear_primal(Q, K, V, eta, W0, b=16)
    for h in range(2):
        q, k, v, w = Q[0, h], K[0, h], V[0, h], W0[h]
        E = k @ w - v
        assert rel(Z[0, h], q @ w - eta[h] * np.tril(q @ k.T) @ E) < 1e-13
        assert rel(W[0, h], w - eta[h] * k.T @ E) < 1e-13


# ------------------------------------------- P7: segment affine maps (a6 form)
@pytest.mark.parametrize("T,b,L", [(96, 16, 32), (100, 16, 48), (64, 8, 64), (45, 5, 15), (30, 3, 30)])
def test_segment_maps_compose_to_the_scan(T, b, L):
    """Each chunk's step is W -> (I - eta K^T K) W + eta K^T V; a segment's map
    is their composition. Applied in turn from W0 they must give the per-token
    scan's state at every segment end (the scan itself is pinned above)."""
    Q, K, V, eta, W0 = rand_linear(2, 3, T, 8, seed=T + b + L)
    A, Bm = oracle.linear_segment_maps(K, V, eta, b, L)
    S = -(-T // L)
    assert A.shape == (2, 3, S, 8, 8)
    for n in range(2):
        for h in range(3):
            W = W0[h].copy()
            for s in range(S):
                W = A[n, h, s] @ W + Bm[n, h, s]
                end = min(T, (s + 1) * L)
                _, Wref = oracle.linear_primal(Q[n:n + 1, :, :end], K[n:n + 1, :, :end], V[n:n + 1, :, :end],
                                               eta, W0, b)
                assert rel(W, Wref[0, h]) < 1e-12


def test_segment_map_of_one_token_is_exact():
    """One token, b = 1: the map is (I - eta k^T k, eta k^T v), by hand in exact rationals."""
    k = [[0.5, -1.0, 0.25]]
    v = [[2.0, 0.0, -3.0]]
    eta = Fraction(1, 4)
    d = 3
    A, Bm = oracle.linear_segment_maps(np.array(k)[None, None], np.array(v)[None, None], [0.25], 1, 1)
    Ax = [[(1 if i == j else 0) - eta * Fraction(k[0][i]) * Fraction(k[0][j]) for j in range(d)] for i in range(d)]
    Bx = [[eta * Fraction(k[0][i]) * Fraction(v[0][j]) for j in range(d)] for i in range(d)]
    assert np.array_equal(A[0, 0, 0], np.array(Ax, dtype=float))
    assert np.array_equal(Bm[0, 0, 0], np.array(Bx, dtype=float))


def test_segment_maps_of_long_segments_contract():
    """With unit keys and 0 < eta < 2, every chunk map shrinks the span of its
    keys, so a long segment's linear part is far below the identity."""
    _, K, V, eta, _ = rand_linear(1, 2, 512, 8, seed=3)
    A, _ = oracle.linear_segment_maps(K, V, eta, 16, 512)
    for h in range(2):
        assert np.linalg.norm(A[0, h, 0], 2) < 0.5


# ------------------------------------------------------------ P3: primal == dual
@pytest.mark.parametrize("T,b", [(64, 16), (50, 16), (37, 5), (16, 16), (9, 64), (1, 16), (40, 1)])
def test_linear_primal_equals_dual(T, b):
    Q, K, V, eta, W0 = rand_linear(2, 3, T, 8, seed=T + b)
    Zp, Wp = oracle.linear_primal(Q, K, V, eta, W0, b)
    Zd, Wd = oracle.linear_dual(Q, K, V, eta, W0, b)
    assert rel(Zd, Zp) < 1e-12 and rel(Wd, Wp) < 1e-12


@pytest.mark.parametrize("T,b", [(32, 16), (21, 8), (7, 16), (12, 1)])
def test_mlp_primal_equals_dual(T, b):
    Q, K, V, eta, W1, W2 = rand_mlp(2, 2, T, 4, 16, seed=T + b)
    Zp, W1p, W2p = oracle.mlp_primal(Q, K, V, eta, W1, W2, b)
    Zd, W1d, W2d = oracle.mlp_dual(Q, K, V, eta, W1, W2, b)
    assert rel(Zd, Zp) < 1e-12 and rel(W1d, W1p) < 1e-12 and rel(W2d, W2p) < 1e-12


# ------------------------------------------------- P4: gradients, FD and autograd
def _fd_grad(f, W, h=1e-6):
    G = np.zeros_like(W)
    it = np.nditer(W, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        Wp = W.copy(); Wp[idx] += h
        Wm = W.copy(); Wm[idx] -= h
        G[idx] = (f(Wp) - f(Wm)) / (2 * h)
    return G


def _lin_loss(W, k, v):
    """sum over rows t of 1/2 || k_t W - v_t ||^2 (loss of '5 · TestingTime 训练与长上下文' sec. 2.3)."""
    r = k @ W - v
    return 0.5 * float(np.sum(r * r))


@pytest.mark.parametrize("T,b", [(1, 1), (5, 5), (6, 3), (7, 3)])
def test_linear_update_is_gradient_step_at_chunk_start(T, b):
    d = 4
    Q, K, V, eta, W0 = rand_linear(1, 1, T, d, seed=T * 7 + b)
    _, W = oracle.linear_primal(Q, K, V, eta, W0, b)
    Wref = W0[0].copy()
    for c0 in range(0, T, b):
        k, v = K[0, 0, c0:c0 + b], V[0, 0, c0:c0 + b]
        g = _fd_grad(lambda X: _lin_loss(X, k, v), Wref)
        Wref = Wref - eta[0] * g
    assert np.max(np.abs(W[0, 0] - Wref)) < 1e-8


def _gelu_t(x):
    return torch.nn.functional.gelu(x, approximate="tanh")


def test_gelu_matches_torch_and_its_derivative():
    x = np.linspace(-8, 8, 2001)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    y = _gelu_t(xt)
    y.sum().backward()
    assert np.max(np.abs(oracle.gelu(x) - y.detach().numpy())) < 1e-14
    assert np.max(np.abs(oracle.gelu_prime(x) - xt.grad.numpy())) < 1e-13
    # special values and the tanh form's closeness to the exact x * Phi(x)
    assert oracle.gelu([0.0])[0] == 0.0 and oracle.gelu_prime([0.0])[0] == 0.5
    exact = torch.nn.functional.gelu(torch.tensor(x), approximate="none").numpy()
    assert np.max(np.abs(oracle.gelu(x) - exact)) < 1e-3


def _mlp_loss_t(W1, W2, k, v):
    return 0.5 * ((_gelu_t(k @ W1) @ W2 - v) ** 2).sum()


@pytest.mark.parametrize("T,b", [(1, 1), (4, 4), (6, 3), (5, 2)])
def test_mlp_update_is_gradient_step_at_chunk_start(T, b):
    d, m = 3, 12
    Q, K, V, eta, W1, W2 = rand_mlp(1, 1, T, d, m, seed=T * 5 + b)
    _, W1o, W2o = oracle.mlp_primal(Q, K, V, eta, W1, W2, b)
    A = torch.tensor(W1[0], dtype=torch.float64)
    Bm = torch.tensor(W2[0], dtype=torch.float64)
    for c0 in range(0, T, b):
        k = torch.tensor(K[0, 0, c0:c0 + b])
        v = torch.tensor(V[0, 0, c0:c0 + b])
        A1 = A.clone().requires_grad_(True)
        B1 = Bm.clone().requires_grad_(True)
        gA, gB = torch.autograd.grad(_mlp_loss_t(A1, B1, k, v), (A1, B1))
        A, Bm = A - eta[0] * gA, Bm - eta[0] * gB
    assert np.max(np.abs(W1o[0, 0] - A.numpy())) < 1e-12
    assert np.max(np.abs(W2o[0, 0] - Bm.numpy())) < 1e-12
    # and the autograd gradient against central differences of the same loss
    k = torch.tensor(K[0, 0, :b]); v = torch.tensor(V[0, 0, :b])
    f1 = lambda X: float(_mlp_loss_t(torch.tensor(X), torch.tensor(W2[0]), k, v))
    A1 = torch.tensor(W1[0]).requires_grad_(True)
    g1, = torch.autograd.grad(_mlp_loss_t(A1, torch.tensor(W2[0]), k, v), (A1,))
    assert np.max(np.abs(_fd_grad(f1, W1[0]) - g1.numpy())) < 1e-7


def test_mlp_readout_uses_updated_weights():
    """z_t = sigma(q_t W1_t) W2_t with W1_t, W2_t after token t's own gradient (update, then read)."""
    d, m, T, b = 3, 12, 5, 5
    Q, K, V, eta, W1, W2 = rand_mlp(1, 1, T, d, m, seed=3)
    Z, _, _ = oracle.mlp_primal(Q, K, V, eta, W1, W2, b)
    A0 = torch.tensor(W1[0]).requires_grad_(True)
    B0 = torch.tensor(W2[0]).requires_grad_(True)
    gA = torch.zeros_like(A0); gB = torch.zeros_like(B0)
    for t in range(T):
        k = torch.tensor(K[0, 0, t:t + 1]); v = torch.tensor(V[0, 0, t:t + 1])
        a, bb = torch.autograd.grad(_mlp_loss_t(A0, B0, k, v), (A0, B0))
        gA, gB = gA + a, gB + bb
        At, Bt = A0.detach() - eta[0] * gA, B0.detach() - eta[0] * gB
        z = _gelu_t(torch.tensor(Q[0, 0, t]) @ At) @ Bt
        assert np.max(np.abs(Z[0, 0, t] - z.numpy())) < 1e-12


# ---------------------------------------------------------------- P5: eta = 0
def test_eta_zero_is_plain_forward():
    Q, K, V, _, W0 = rand_linear(2, 2, 20, 6)
    Z, W = oracle.linear_primal(Q, K, V, np.zeros(2), W0, 4)
    assert rel(Z, np.einsum("nhti,hij->nhtj", Q, W0)) < 1e-14
    assert np.array_equal(W, np.broadcast_to(W0, W.shape))
    Q, K, V, _, W1, W2 = rand_mlp(1, 2, 9, 4, 16)
    Z, W1o, W2o = oracle.mlp_primal(Q, K, V, np.zeros(2), W1, W2, 4)
    ref = torch.einsum("nhtp,hpj->nhtj", _gelu_t(torch.einsum("nhti,hip->nhtp", torch.tensor(Q),
                                                                   torch.tensor(W1))), torch.tensor(W2))
    assert rel(Z, ref.numpy()) < 1e-14
    assert np.array_equal(W1o[0], W1) and np.array_equal(W2o[0], W2)


# ------------------------------------------------ P6: chaining and decoding
@pytest.mark.parametrize("T1,T2,b", [(32, 21, 16), (12, 12, 4), (5, 3, 1)])
def test_chain_two_calls_equal_one(T1, T2, b):
    Q, K, V, eta, W0 = rand_linear(2, 2, T1 + T2, 6, seed=T1)
    Z, W = oracle.linear_primal(Q, K, V, eta, W0, b)
    Za, Wa = oracle.linear_primal(Q[:, :, :T1], K[:, :, :T1], V[:, :, :T1], eta, W0, b)
    # restart from each row's own final state: one call per batch row
    for n in range(2):
        Zb, Wb = oracle.linear_primal(Q[n:n + 1, :, T1:], K[n:n + 1, :, T1:], V[n:n + 1, :, T1:],
                                      eta, Wa[n], b)
        assert rel(np.concatenate([Za[n], Zb[0]], axis=1), Z[n]) < 1e-13
        assert rel(Wb[0], W[n]) < 1e-13


def test_mlp_chain_two_calls_equal_one():
    Q, K, V, eta, W1, W2 = rand_mlp(1, 2, 24, 4, 16)
    Z, W1o, W2o = oracle.mlp_primal(Q, K, V, eta, W1, W2, 8)
    Za, W1a, W2a = oracle.mlp_primal(Q[:, :, :16], K[:, :, :16], V[:, :, :16], eta, W1, W2, 8)
    Zb, W1b, W2b = oracle.mlp_primal(Q[:, :, 16:], K[:, :, 16:], V[:, :, 16:], eta, W1a[0], W2a[0], 8)
    assert rel(np.concatenate([Za, Zb], axis=2), Z) < 1e-13
    assert rel(W1b, W1o) < 1e-13 and rel(W2b, W2o) < 1e-13


@pytest.mark.parametrize("T1,N,b", [(16, 20, 16), (0, 9, 4), (8, 3, 1)])
def test_decode_steps_equal_forward(T1, N, b):
    Q, K, V, eta, W0 = rand_linear(2, 3, T1 + N, 5, seed=N)
    Z, W = oracle.linear_primal(Q, K, V, eta, W0, b)
    if T1:
        _, Wp = oracle.linear_primal(Q[:, :, :T1], K[:, :, :T1], V[:, :, :T1], eta, W0, b)
    else:
        Wp = np.broadcast_to(W0, (2, 3, 5, 5)).copy()
    Wa, Wr = Wp.copy(), Wp.copy()
    for s in range(N):
        t = T1 + s
        z, Wa, Wr = oracle.linear_decode_step(Q[:, :, t], K[:, :, t], V[:, :, t], eta, Wa, Wr, t, b)
        assert rel(z, Z[:, :, t]) < 1e-13
    assert rel(Wr, W) < 1e-13


# ------------------------------------------------ per-sequence reset
def test_batch_rows_are_independent():
    Q, K, V, eta, W0 = rand_linear(3, 2, 20, 4)
    Z, W = oracle.linear_primal(Q, K, V, eta, W0, 8)
    perm = [2, 0, 1, 2]
    Zp, Wp = oracle.linear_primal(Q[perm], K[perm], V[perm], eta, W0, 8)
    assert np.array_equal(Zp, Z[perm]) and np.array_equal(Wp, W[perm])


# ------------------------------------------------ hand-worked examples
@pytest.mark.parametrize("name", ["linear_scalar_d1.json", "linear_matrix_d2.json"])
def test_golden_hand_worked(name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    args = [np.array(g[x], dtype=float) for x in ("q", "k", "v", "eta", "W0")]
    for fn in (oracle.linear_primal, oracle.linear_dual):
        Z, W = fn(*args, b=g["b"])
        assert np.array_equal(Z, np.array(g["Z"], dtype=float))
        assert np.array_equal(W, np.array(g["W_out"], dtype=float))


# ------------------------------------------------ the pins would catch these
def _planted(q, k, v, eta, W0, b, mistake):
    """A per-token TTT-Linear loop with one deliberate slip (never the oracle itself)."""
    T, d = k.shape
    W = W0.copy()
    Z = np.zeros((T, d))
    for c0 in range(0, T, b):
        Wa = W.copy()
        for t in range(c0, min(c0 + b, T)):
            Wg = W if mistake == "running_grad" else Wa
            e = (Wg @ k[t] if mistake == "transposed" else k[t] @ Wg) - v[t]
            scale = 2.0 if mistake == "no_half" else 1.0
            sign = -1.0 if mistake == "wrong_sign" else 1.0
            if mistake == "read_first":
                Z[t] = q[t] @ W
            W = W - sign * scale * eta * np.outer(k[t], e)
            if mistake != "read_first":
                Z[t] = q[t] @ W
    return Z, W


@pytest.mark.parametrize("mistake", ["running_grad", "transposed", "no_half", "wrong_sign", "read_first"])
def test_planted_mistakes_are_caught(mistake):
    caught = []
    for name in ("linear_scalar_d1.json", "linear_matrix_d2.json"):
        g = json.load(open(os.path.join(GOLDEN, name)))
        q, k, v = (np.array(g[x], float)[0, 0] for x in ("q", "k", "v"))
        Z, W = _planted(q, k, v, g["eta"][0], np.array(g["W0"], float)[0], g["b"], mistake)
        caught.append(not (np.allclose(Z, np.array(g["Z"])[0, 0]) and
                           np.allclose(W, np.array(g["W_out"])[0, 0])))
    # the same slip also breaks the finite-difference pin with b = T
    Q, K, V, eta, W0 = rand_linear(1, 1, 6, 3, seed=1)
    _, W = _planted(Q[0, 0], K[0, 0], V[0, 0], eta[0], W0[0], 6, mistake)
    g = _fd_grad(lambda X: _lin_loss(X, K[0, 0], V[0, 0]), W0[0])
    Zc, _ = _planted(Q[0, 0], K[0, 0], V[0, 0], eta[0], W0[0], 6, mistake)
    E = K[0, 0] @ W0[0] - V[0, 0]
    closed = Q[0, 0] @ W0[0] - eta[0] * np.tril(Q[0, 0] @ K[0, 0].T) @ E
    caught.append(np.max(np.abs(W - (W0[0] - eta[0] * g))) > 1e-6 or rel(Zc, closed) > 1e-9)
    assert any(caught), mistake


# ---------------------------------------------------------------- planted slips, TTT-MLP
def _mlp_planted(Q, K, V, eta, W1, W2, b, mistake):
    """The TTT-MLP chunk rule token by token with one plausible slip planted (fp64, one unit)."""
    c, a = np.sqrt(2 / np.pi), 0.044715
    th = lambda u: np.tanh(c * (u + a * u ** 3))
    gelu = lambda u: 0.5 * u * (1 + th(u))
    dgelu = lambda u: 0.5 * (1 + th(u)) + 0.5 * u * (1 - th(u) ** 2) * c * (1 + 3 * a * u * u)
    if mistake == "erf_gelu":
        from math import erf
        gelu = np.vectorize(lambda u: 0.5 * u * (1 + erf(u / np.sqrt(2))))
    A, Bm = W1.copy(), W2.copy()
    Z = np.zeros_like(Q)
    for t in range(len(Q)):
        if t % b == 0:
            A0, B0 = A.copy(), Bm.copy()
        u = K[t] @ A0
        act = gelu(u)
        g = act @ B0 - V[t]
        s1 = gelu(u) if mistake == "sigma_for_derivative" else (1.0 if mistake == "no_derivative" else dgelu(u))
        delta = (g @ (Bm if mistake == "running_w2" else B0).T) * s1
        if mistake == "read_first":
            Z[t] = gelu(Q[t] @ A) @ Bm
        A = A - eta * np.outer(K[t], delta)
        Bm = Bm - eta * np.outer(act, g)
        if mistake != "read_first":
            Z[t] = gelu(Q[t] @ A) @ Bm
    return Z, A, Bm


@pytest.mark.parametrize("mistake", ["none", "sigma_for_derivative", "no_derivative", "erf_gelu", "running_w2",
                                     "read_first"])
def test_mlp_planted_mistakes_are_caught(mistake):
    """Each slip moves the result far outside the 1e-12 the autograd pins hold the oracle to; the
    slip-free restatement matches the oracle."""
    d, m, T, b = 3, 12, 6, 3
    Q, K, V, eta, W1, W2 = rand_mlp(1, 1, T, d, m, seed=11)
    Z, A, Bm = oracle.mlp_primal(Q, K, V, eta, W1, W2, b)
    Zp, Ap, Bp = _mlp_planted(Q[0, 0], K[0, 0], V[0, 0], eta[0], W1[0], W2[0], b, mistake)
    gap = max(np.max(np.abs(Zp - Z[0, 0])), np.max(np.abs(Ap - A[0, 0])), np.max(np.abs(Bp - Bm[0, 0])))
    if mistake == "none":
        assert gap < 1e-12
    else:
        assert gap > 1e-6, mistake
