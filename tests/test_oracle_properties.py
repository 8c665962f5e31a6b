"""Properties of the oracle over random shapes (CPU only, hypothesis).

The fixed-case pins in test_oracle_pins.py tie the oracle to the pages at chosen
sizes. These draw the sizes instead (batch rows, heads, width, sequence length,
chunk size, segment length, ragged tails included) and check the identities
that must hold at any size: the per-token primal form equals the per-chunk dual
form (TTT-Linear and TTT-MLP); two calls chained at a chunk boundary equal one
call; decode tokens continue a forward exactly; the segment maps, composed from
W0, give the scan's state at every segment end; and with one chunk the whole
scan is the closed form Q W0 - eta tril(Q K^T)(K W0 - V).
"""
import numpy as np
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle

SETTINGS = settings(max_examples=40, deadline=None, suppress_health_check=[HealthCheck.too_slow])


def draw_inputs(seed, B, H, T, d):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((B, H, T, d)) for _ in range(3))
    K /= np.linalg.norm(K, axis=-1, keepdims=True)
    Q /= np.linalg.norm(Q, axis=-1, keepdims=True)
    eta = g.uniform(0.01, 0.6, H)
    W0 = g.standard_normal((H, d, d)) * 0.2
    return Q, K, V, eta, W0


shapes = st.tuples(st.integers(1, 2), st.integers(1, 3), st.integers(0, 40), st.integers(1, 6), st.integers(1, 12),
                   st.integers(0, 2 ** 31 - 1))


@SETTINGS
@given(shapes)
def test_primal_equals_dual(s):
    B, H, T, d, b, seed = s
    args = draw_inputs(seed, B, H, T, d)
    Zp, Wp = oracle.linear_primal(*args, b)
    Zd, Wd = oracle.linear_dual(*args, b)
    assert np.allclose(Zp, Zd, atol=1e-11) and np.allclose(Wp, Wd, atol=1e-11)


@SETTINGS
@given(shapes, st.integers(0, 4))
def test_two_calls_chained_at_a_chunk_boundary_equal_one(s, chunks):
    B, H, T, d, b, seed = s
    T1 = min(chunks * b, T)
    T1 -= T1 % b
    Q, K, V, eta, W0 = draw_inputs(seed, B, H, T, d)
    Z, Wo = oracle.linear_primal(Q, K, V, eta, W0, b)
    Z1, W1 = oracle.linear_primal(Q[:, :, :T1], K[:, :, :T1], V[:, :, :T1], eta, W0, b)
    for n in range(B):  # the second call starts every head of row n from row n's state
        Z2, W2 = oracle.linear_primal(Q[n:n + 1, :, T1:], K[n:n + 1, :, T1:], V[n:n + 1, :, T1:], eta, W1[n], b)
        assert np.allclose(Z[n, :, :T1], Z1[n], atol=1e-12) and np.allclose(Z[n, :, T1:], Z2[0], atol=1e-11)
        assert np.allclose(Wo[n], W2[0], atol=1e-11)


@SETTINGS
@given(shapes, st.integers(1, 4))
def test_segment_maps_compose_to_the_scan(s, chunks_per_segment):
    B, H, T, d, b, seed = s
    L = chunks_per_segment * b
    Q, K, V, eta, W0 = draw_inputs(seed, B, H, T, d)
    A, Bm = oracle.linear_segment_maps(K, V, eta, b, L)
    for n in range(B):
        for h in range(H):
            W = W0[h]
            for sgm in range(A.shape[2]):
                W = A[n, h, sgm] @ W + Bm[n, h, sgm]
                t_end = min((sgm + 1) * L, T)
                _, Wt = oracle.linear_primal(Q[n:n + 1, h:h + 1, :t_end], K[n:n + 1, h:h + 1, :t_end],
                                             V[n:n + 1, h:h + 1, :t_end], eta[h:h + 1], W0[h:h + 1], b)
                assert np.allclose(W, Wt[0, 0], atol=1e-10)


@SETTINGS
@given(st.integers(1, 24), st.integers(1, 6), st.integers(0, 2 ** 31 - 1))
def test_one_chunk_is_the_closed_form(T, d, seed):
    Q, K, V, eta, W0 = draw_inputs(seed, 1, 1, T, d)
    Z, Wo = oracle.linear_primal(Q, K, V, eta, W0, T)
    q, k, v, w, e = Q[0, 0], K[0, 0], V[0, 0], W0[0], eta[0]
    E = k @ w - v
    assert np.allclose(Z[0, 0], q @ w - e * np.tril(q @ k.T) @ E, atol=1e-12)
    assert np.allclose(Wo[0, 0], w - e * k.T @ E, atol=1e-12)


@SETTINGS
@given(st.integers(1, 2), st.integers(1, 2), st.integers(0, 20), st.integers(1, 4), st.integers(1, 8),
       st.integers(0, 2 ** 31 - 1))
def test_mlp_primal_equals_dual(B, H, T, d, b, seed):
    g = np.random.default_rng(seed)
    Q, K, V = (g.standard_normal((B, H, T, d)) * 0.7 for _ in range(3))
    eta = g.uniform(0.01, 0.3, H)
    W1, W2 = g.standard_normal((H, d, 4 * d)) * 0.3, g.standard_normal((H, 4 * d, d)) * 0.3
    Zp, A1, A2 = oracle.mlp_primal(Q, K, V, eta, W1, W2, b)
    Zd, D1, D2 = oracle.mlp_dual(Q, K, V, eta, W1, W2, b)
    assert np.allclose(Zp, Zd, atol=1e-11) and np.allclose(A1, D1, atol=1e-11) and np.allclose(A2, D2, atol=1e-11)


@SETTINGS
@given(shapes, st.integers(0, 3), st.integers(1, 12))
def test_decode_continues_a_forward(s, chunks, N):
    """A forward over whole chunks, then N decode tokens from (W_anchor, W_run) = (W_out, W_out),
    equals one forward over all the tokens: every z and the final state."""
    B, H, _, d, b, seed = s
    T1 = chunks * b
    Q, K, V, eta, W0 = draw_inputs(seed, B, H, T1 + N, d)
    Z, W = oracle.linear_primal(Q, K, V, eta, W0, b)
    _, Wp = oracle.linear_primal(Q[:, :, :T1], K[:, :, :T1], V[:, :, :T1], eta, W0, b)
    Wa, Wr = Wp.copy(), Wp.copy()
    for t in range(T1, T1 + N):
        z, Wa, Wr = oracle.linear_decode_step(Q[:, :, t], K[:, :, t], V[:, :, t], eta, Wa, Wr, t, b)
        assert np.allclose(z, Z[:, :, t], atol=1e-12)
    assert np.allclose(Wr, W, atol=1e-12)
