"""The algebra the fast kernels rely on, checked in fp64 on the host (no GPU).

Each kernel restates the chunk rule ("5 · TestingTime 训练与长上下文", section 1.1:
the gradients of a chunk are taken at its start weights) in a form that suits
the hardware. These tests check each restatement against the rule applied
chunk by chunk, on random inputs:
  - segment affine maps on tcgen05: several chunks of one 64-token group fold
    into one affine map, X_end = X0 + M X0 + [0 | Q], M = -eta Kh^T K,
    Q = eta Kh^T V, with Kh = T^T K and T = (I + eta N)^-1 (N: the strictly
    block-lower chunk blocks of K K^T);
  - the read-out kernel walks a chunk in 16-token tiles: each tile's error uses
    the chunk-start state, its read-out the running state;
  - the combine: W_start(s+1) = A_s W_start(s) + B_s reproduces the scan;
  - the backward's segment-parallel form (transposed maps);
  - restatements for faster kernels: Kh by a finite (nilpotent) series in
    Horner form, a read-out that takes a 64-token group of chunks at once, and
    group maps composed in pairs (exact, and with the kernel's bf16 rounding);
  - two inner-model variants that reduce to plain TTT-Linear on changed inputs:
    a bias in f (a constant extra input) and a per-token learning rate
    (keys and values scaled by its square root);
  - the momentum kernel's transposed per-tile form ("推理时的“临阵磨枪”：Test-Time
    Training如何教会AI“边做边学”", sections 2.3 and 5.1, read as token-level
    momentum with chunk-start gradients).
"""
import numpy as np
import pytest


def chunk_rule(K, V, eta, W, b):
    """State after the chunk rule over all of K, V (chunks of b tokens)."""
    for c0 in range(0, len(K), b):
        Kc, Vc = K[c0:c0 + b], V[c0:c0 + b]
        W = W - eta * Kc.T @ (Kc @ W - Vc)
    return W


@pytest.mark.parametrize("b", [16, 32, 64])
def test_group_of_chunks_is_one_affine_map(b):
    """64 tokens = 64/b chunks: the kernel's map, built from K and V alone, equals
    the chunk-by-chunk update of X = [A | B] from [I | 0] with value rows [0 | V]."""
    g = np.random.default_rng(b)
    d, n = 8, 64
    K = g.standard_normal((n, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = g.standard_normal((n, d))
    eta = 0.3
    # chunk rule on the augmented state: the A half follows A <- A - eta K^T K A,
    # the B half B <- B - eta K^T (K B - V)
    X0 = np.hstack([np.eye(d), np.zeros((d, d))])
    Y = np.hstack([np.zeros((n, d)), V])
    X = X0.copy()
    for c0 in range(0, n, b):
        Kc, Yc = K[c0:c0 + b], Y[c0:c0 + b]
        X = X - eta * Kc.T @ (Kc @ X - Yc)
    # the kernel's form
    G = K @ K.T
    blk = np.arange(n) // b
    N = np.where(blk[:, None] > blk[None, :], G, 0.0)  # strictly block-lower chunk blocks
    T = np.linalg.inv(np.eye(n) + eta * N)
    Kh = T.T @ K
    M = -eta * Kh.T @ K
    Q = eta * Kh.T @ V
    X_kernel = X0 + M @ X0 + np.hstack([np.zeros((d, d)), Q])
    assert np.allclose(X_kernel, X, atol=1e-12, rtol=0)
    # the map also advances any other start state the same way
    W = g.standard_normal((d, d))
    assert np.allclose(W + M @ W + Q, chunk_rule(K, V, eta, W, b), atol=1e-12, rtol=0)


@pytest.mark.parametrize("bt", [16, 32])
def test_unit_lower_blocks_of_T_transposed(bt):
    """The helper warps build T^T in 16-token blocks by U_cr = -eta sum_{c <= m < r} U_cm G_mr
    (U_cc = I), where G_mr, the (m, r) block of K K^T, enters only if blocks m and r lie in
    different chunks: that is the inverse of (I + eta N)^T."""
    g = np.random.default_rng(7 + bt)
    d = 8
    K = g.standard_normal((64, d))
    eta = 0.2
    G = K @ K.T
    blocks = 4
    Gb = lambda m, r: G[16 * m:16 * m + 16, 16 * r:16 * r + 16] * ((16 * m) // bt < (16 * r) // bt)
    U = {}
    for c in range(blocks):
        U[c, c] = np.eye(16)
        for r in range(c + 1, blocks):
            U[c, r] = -eta * sum(U[c, m] @ Gb(m, r) for m in range(c, r))
    Tt = np.block([[U[c, r] if r >= c else np.zeros((16, 16)) for r in range(blocks)] for c in range(blocks)])
    blk = np.arange(64) // bt
    N = np.where(blk[:, None] > blk[None, :], G, 0.0)
    assert np.allclose(Tt, np.linalg.inv(np.eye(64) + eta * N).T, atol=1e-12)


@pytest.mark.parametrize("b", [32, 48, 64])
def test_chunk_walked_in_16_token_tiles(b):
    """Z of a chunk equals, tile by tile, Q_u W_run - eta tril(Q_u K_u^T) E_u, where
    E_u = K_u W_a - V_u uses the chunk-start state W_a and W_run has taken the
    gradients of the chunk's earlier tiles."""
    g = np.random.default_rng(b)
    d = 8
    Q, K, V = (g.standard_normal((b, d)) for _ in range(3))
    Wa = g.standard_normal((d, d)) * 0.3
    eta = 0.25
    E = K @ Wa - V
    Z_dual = Q @ Wa - eta * np.tril(Q @ K.T) @ E  # the chunk rule in dual form
    Wrun = Wa.copy()
    Z_tiles = np.zeros_like(Z_dual)
    for u0 in range(0, b, 16):
        Qu, Ku, Eu = Q[u0:u0 + 16], K[u0:u0 + 16], E[u0:u0 + 16]
        Z_tiles[u0:u0 + 16] = Qu @ Wrun - eta * np.tril(Qu @ Ku.T) @ Eu
        Wrun = Wrun - eta * Ku.T @ Eu
    assert np.allclose(Z_tiles, Z_dual, atol=1e-12)
    assert np.allclose(Wrun, Wa - eta * K.T @ E, atol=1e-12)


def test_segment_maps_combine_to_the_scan():
    """The combine kernel's recurrence over the segment maps gives every segment's
    start state of the chunk-by-chunk scan."""
    g = np.random.default_rng(3)
    d, b, L, S = 6, 4, 12, 5
    K = g.standard_normal((L * S, d)) * 0.5
    V = g.standard_normal((L * S, d))
    eta = 0.3
    W0 = g.standard_normal((d, d))
    W = W0
    for s in range(S - 1):
        Ks, Vs = K[s * L:(s + 1) * L], V[s * L:(s + 1) * L]
        A = chunk_rule(Ks, np.zeros_like(Vs), eta, np.eye(d), b)
        B = chunk_rule(Ks, Vs, eta, np.zeros((d, d)), b)
        W = A @ W + B
        assert np.allclose(W, chunk_rule(K[:(s + 1) * L], V[:(s + 1) * L], eta, W0, b), atol=1e-12)


def test_backward_runs_segment_parallel_on_the_transposed_maps():
    """The state gradient is affine too: with Z_c = P_c W_c + eta S_c V_c, P_c = Q_c - eta S_c K_c,
    G_c = A_c^T G_{c+1} + P_c^T dZ_c from G = dW_out at the end. A segment's backward map is
    therefore (A_s^T, H_s): the transpose of its forward map, and an additive term that depends
    on the inputs and dZ only. Composed from the last segment back, these maps give the chunk-level
    gradient at every segment start, and at the first one dW0 of the oracle's backward."""
    from oracle.backward import linear_backward
    g = np.random.default_rng(11)
    d, b, L, S = 5, 4, 12, 4
    T = L * S
    Q, K, V, dZ = (g.standard_normal((T, d)) * 0.6 for _ in range(4))
    W0, dW = g.standard_normal((d, d)) * 0.4, g.standard_normal((d, d))
    eta = 0.3

    def chunk_terms(c0):
        Qc, Kc, dZc = Q[c0:c0 + b], K[c0:c0 + b], dZ[c0:c0 + b]
        A = np.eye(d) - eta * Kc.T @ Kc
        P = Qc - eta * np.tril(Qc @ Kc.T) @ Kc
        return A, P.T @ dZc

    # chunk level, last chunk first
    G = dW.copy()
    G_at = {}
    for c0 in reversed(range(0, T, b)):
        A, H = chunk_terms(c0)
        G = A.T @ G + H
        G_at[c0] = G
    _, _, _, _, dW0 = linear_backward(Q[None, None], K[None, None], V[None, None], np.array([eta]), W0[None], b,
                                      dZ[None, None], dW[None, None])
    assert np.allclose(G_at[0], dW0[0], atol=1e-12)
    # segment level: (A_s^T, H_s) per segment, each from its own chunks only
    maps = []
    for s in range(S):
        As, Hs = np.eye(d), np.zeros((d, d))
        for c0 in reversed(range(s * L, (s + 1) * L, b)):  # G_start = A_s^T G_end + H_s
            A, H = chunk_terms(c0)
            As, Hs = As @ A, A.T @ Hs + H
        fwd = chunk_rule(K[s * L:(s + 1) * L], np.zeros((L, d)), eta, np.eye(d), b)  # the forward map's A_s
        assert np.allclose(As, fwd, atol=1e-12)  # the backward map's matrix is the forward one, transposed
        maps.append((As, Hs))
    G = dW.copy()
    for s in reversed(range(S)):
        As, Hs = maps[s]
        G = As.T @ G + Hs
        assert np.allclose(G, G_at[s * L], atol=1e-12)


@pytest.mark.parametrize("b", [1, 3, 8])
def test_bias_is_an_extra_constant_input(b):
    """TTT-Linear with a bias, f(k) = k W + beta, trained like W (the same chunk rule on the
    loss 1/2 ||k W + beta - v||^2, read-out q W_t + beta_t), equals plain TTT-Linear on keys
    and queries extended by a constant 1, with state [W; beta^T]. The state stays square by
    one more output column (target 0, start 0); the output columns learn independently, so
    that column never touches the others. So the library serves the bias variant for d <= 63
    with no new kernel."""
    import oracle
    g = np.random.default_rng(b)
    T, d = 11, 4
    Q, K, V = (g.standard_normal((T, d)) for _ in range(3))
    W0, beta0 = g.standard_normal((d, d)) * 0.3, g.standard_normal(d) * 0.3
    eta = 0.2
    # the bias variant, token by token: gradients at the chunk-start (W, beta), then read-out
    W, beta = W0.copy(), beta0.copy()
    Z = np.zeros((T, d))
    for t in range(T):
        if t % b == 0:
            Wa, ba = W.copy(), beta.copy()
        e = K[t] @ Wa + ba - V[t]
        W = W - eta * np.outer(K[t], e)
        beta = beta - eta * e
        Z[t] = Q[t] @ W + beta
    one, zero = np.ones((T, 1)), np.zeros((T, 1))
    W0x = np.zeros((d + 1, d + 1))
    W0x[:d, :d], W0x[d, :d] = W0, beta0
    Zx, Wx = oracle.linear_primal(np.hstack([Q, one])[None, None], np.hstack([K, one])[None, None],
                                  np.hstack([V, zero])[None, None], np.array([eta]), W0x[None], b)
    assert np.allclose(Zx[0, 0, :, :d], Z, atol=1e-12)
    assert np.allclose(Wx[0, 0, :, :d], np.vstack([W, beta]), atol=1e-12)


@pytest.mark.parametrize("b", [16, 32, 64])
def test_khat_by_a_nilpotent_series(b):
    """T = (I + eta N)^-1 needs no inversion: N is strictly block-lower with 64/b chunk blocks, so
    (eta N)^(64/b) = 0 and T is the finite series sum_p (-eta N)^p. Applied to K in Horner form,
    Kh = T^T K = K - eta N^T (K - eta N^T (K - eta N^T K)) for four chunks: 64/b - 1 dependent
    products of the same 64 x 64 by 64 x d shape, a form for tensor cores in place of the block
    recursion of the helper warps."""
    g = np.random.default_rng(40 + b)
    d, n, eta = 8, 64, 0.35
    K = g.standard_normal((n, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    blk = np.arange(n) // b
    N = np.where(blk[:, None] > blk[None, :], K @ K.T, 0.0)
    depth = n // b
    assert np.allclose(np.linalg.matrix_power(eta * N, depth), 0.0, atol=0)
    Kh = K.copy()
    for _ in range(depth - 1):
        Kh = K - eta * N.T @ Kh
    assert np.allclose(Kh, np.linalg.inv(np.eye(n) + eta * N).T @ K, atol=1e-12)


@pytest.mark.parametrize("b", [16, 32])
def test_readout_of_a_64_token_group(b):
    """A read-out can take a 64-token group of several chunks in one pass. With P = K W0 - V the
    errors at the chunk starts follow E_c = P_c - eta sum_{c' < c} (K_c K_c'^T) E_c' (a short
    recursion over the group's chunks, or E = T P); then Z = Q W0 - eta tril(Q K^T) E over the whole
    group (the earlier chunks' blocks are full, the chunk's own is lower-triangular, so the mask is
    plain causal) and W_end = W0 - eta K^T E. This equals the chunk rule chunk by chunk, with one
    state update per group instead of one per chunk."""
    g = np.random.default_rng(50 + b)
    d, n, eta = 8, 64, 0.3
    Q, K, V = (g.standard_normal((n, d)) for _ in range(3))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    W0 = g.standard_normal((d, d)) * 0.3
    # the chunk rule in dual form, chunk by chunk
    W, Zc = W0.copy(), np.zeros((n, d))
    for c0 in range(0, n, b):
        Qc, Kc, Vc = Q[c0:c0 + b], K[c0:c0 + b], V[c0:c0 + b]
        E = Kc @ W - Vc
        Zc[c0:c0 + b] = Qc @ W - eta * np.tril(Qc @ Kc.T) @ E
        W = W - eta * Kc.T @ E
    # the group form
    P = K @ W0 - V
    E = np.zeros_like(P)
    for c0 in range(0, n, b):
        E[c0:c0 + b] = P[c0:c0 + b] - eta * (K[c0:c0 + b] @ K[:c0].T) @ E[:c0]
    blk = np.arange(n) // b
    N = np.where(blk[:, None] > blk[None, :], K @ K.T, 0.0)
    assert np.allclose(E, np.linalg.solve(np.eye(n) + eta * N, P), atol=1e-12)
    assert np.allclose(Q @ W0 - eta * np.tril(Q @ K.T) @ E, Zc, atol=1e-12)
    assert np.allclose(W0 - eta * K.T @ E, W, atol=1e-12)


def test_per_token_learning_rate_is_a_scaling_of_keys_and_values():
    """A per-token inner learning rate eta_t >= 0 (gradient of token t scaled by eta_t) equals plain
    TTT-Linear with eta = 1 on keys and values scaled by sqrt(eta_t), queries unchanged: the error
    becomes sqrt(eta_t) e_t, so each outer product k^T e and each read-out weight (q . k_i) e_i picks
    up eta_t exactly once. So the library serves it for any d and b with no new kernel."""
    import oracle
    g = np.random.default_rng(9)
    T, d, b = 13, 4, 4
    Q, K, V = (g.standard_normal((T, d)) for _ in range(3))
    et = g.uniform(0.0, 0.5, T)
    W0 = g.standard_normal((d, d)) * 0.3
    W, Z = W0.copy(), np.zeros((T, d))
    for t in range(T):
        if t % b == 0:
            Wa = W.copy()
        W = W - et[t] * np.outer(K[t], K[t] @ Wa - V[t])
        Z[t] = Q[t] @ W
    r = np.sqrt(et)[:, None]
    Zs, Ws = oracle.linear_primal(Q[None, None], (r * K)[None, None], (r * V)[None, None], np.array([1.0]),
                                  W0[None], b)
    assert np.allclose(Zs[0, 0], Z, atol=1e-12)
    assert np.allclose(Ws[0, 0], W, atol=1e-12)


def test_group_maps_compose_in_any_association():
    """The chain X <- X + M_g X + [0 | Q_g] over a segment's groups is a product of affine maps, so
    composing them pairwise first, [I+M2 | Q2] o [I+M1 | Q1] = [(I+M2)(I+M1) | (I+M2) Q1 + Q2], and then
    chaining the pairs gives the same segment map as the group-by-group chain."""
    g = np.random.default_rng(21)
    d, n, b, eta, groups = 6, 16, 4, 0.3, 8
    K = g.standard_normal((groups * n, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = g.standard_normal((groups * n, d))
    maps = []
    for gi in range(groups):  # each group's map from the chunk rule alone
        Kg, Vg = K[gi * n:(gi + 1) * n], V[gi * n:(gi + 1) * n]
        A = chunk_rule(Kg, np.zeros_like(Vg), eta, np.eye(d), b)
        maps.append((A - np.eye(d), chunk_rule(Kg, Vg, eta, np.zeros((d, d)), b)))
    X = np.hstack([np.eye(d), np.zeros((d, d))])
    for M, Q in maps:  # the chain, group by group
        X = X + M @ X + np.hstack([np.zeros((d, d)), Q])

    def compose(second, first):
        (M2, Q2), (M1, Q1) = second, first
        return M1 + M2 + M2 @ M1, Q1 + Q2 + M2 @ Q1

    pairs = [compose(maps[i + 1], maps[i]) for i in range(0, groups, 2)]
    quads = [compose(pairs[i + 1], pairs[i]) for i in range(0, len(pairs), 2)]
    Y = np.hstack([np.eye(d), np.zeros((d, d))])
    for M, Q in quads:
        Y = Y + M @ Y + np.hstack([np.zeros((d, d)), Q])
    assert np.allclose(Y, X, atol=1e-12)
    assert np.allclose(X[:, :d], chunk_rule(K, np.zeros_like(V), eta, np.eye(d), b), atol=1e-12)
    assert np.allclose(X[:, d:], chunk_rule(K, V, eta, np.zeros((d, d)), b), atol=1e-12)


def test_pairwise_composition_keeps_the_rounding_error_of_the_chain():
    """The same segment map with bf16 operands and fp32 accumulation at the tcgen05 kernel's rounding
    points (Kh and the chain's X rounded to bf16; M and Q formed from bf16 operands): composing group
    maps in pairs once or twice before the chain leaves the error in B (which dominates a segment's start
    state) within 15 % of the chain's; A's relative error grows, but A itself is negligible."""
    import torch

    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()
    f32 = lambda x: x.astype(np.float32).astype(np.float64)
    g = np.random.default_rng(0)
    d, n, b, eta, L = 64, 64, 16, 0.1, 4864
    K = g.standard_normal((L, d))
    K = bf(K / np.linalg.norm(K, axis=1, keepdims=True))
    V = bf(g.standard_normal((L, d)))
    blk = np.arange(n) // b
    exact, rounded = [], []
    for g0 in range(0, L, n):
        Kg, Vg = K[g0:g0 + n], V[g0:g0 + n]
        N = np.where(blk[:, None] > blk[None, :], Kg @ Kg.T, 0.0)
        Kh = np.linalg.inv(np.eye(n) + eta * N).T @ Kg
        exact.append((-eta * Kh.T @ Kg, eta * Kh.T @ Vg))
        rounded.append((f32(-eta * bf(Kh).T @ bf(Kg)), f32(eta * bf(Kh).T @ bf(Vg))))

    def run(maps, levels, kernel):
        for _ in range(levels):
            nxt = []
            for i in range(0, len(maps), 2):
                if i + 1 == len(maps):
                    nxt.append(maps[i])
                    continue
                (M1, Q1), (M2, Q2) = maps[i], maps[i + 1]
                P, R = (bf(M2) @ bf(M1), bf(M2) @ bf(Q1)) if kernel else (M2 @ M1, M2 @ Q1)
                nxt.append((f32(M1 + M2 + P), f32(Q1 + Q2 + R)) if kernel else (M1 + M2 + P, Q1 + Q2 + R))
            maps = nxt
        X = np.hstack([np.eye(d), np.zeros((d, d))])
        for M, Q in maps:
            Qx = np.hstack([np.zeros((d, d)), bf(Q) if kernel else Q])
            X = f32(X + bf(M) @ bf(X) + Qx) if kernel else X + M @ X + Qx
        return X

    ref = run(exact, 0, False)
    err = lambda X, part: np.linalg.norm(X[:, part] - ref[:, part]) / np.linalg.norm(ref[:, part])
    A, B = slice(0, d), slice(d, 2 * d)
    chain = run(rounded, 0, True)
    assert err(chain, B) < 5e-3 and err(chain, A) < 1e-2
    for levels in (1, 2):
        X = run(rounded, levels, True)
        assert err(X, B) < 1.15 * err(chain, B)
        # A's part of a start state, |dA| |W| with |W| ~ |B|, stays below B's own error
        assert np.linalg.norm(X[:, A] - ref[:, A]) * np.linalg.norm(ref[:, B]) < np.linalg.norm(X[:, B] - ref[:, B])


@pytest.mark.parametrize("T,beta", [(16, 0.5), (37, 0.9), (100, 0.0), (5, 0.7)])
def test_momentum_in_transposed_16_token_tiles(T, beta):
    """The momentum kernel's per-tile form (W^T and M^T per output-column block, token-column
    scalings of E^T, a ragged last tile with its own n) equals token-level momentum with
    chunk-start gradients: g_t = k_t^T (k_t W_a - v_t), M = beta M + (1 - beta) g_t,
    W = W - alpha M, z_t = q_t W."""
    g = np.random.default_rng(T)
    d, alpha = 16, 0.1
    Q, K, V = g.standard_normal((T, d)) / 4, g.standard_normal((T, d)) / 4, g.standard_normal((T, d))
    W0 = 0.05 * g.standard_normal((d, d))
    # token by token
    W, M, Wa, Z = W0.copy(), np.zeros((d, d)), W0.copy(), np.zeros((T, d))
    for t in range(T):
        if t % 16 == 0:
            Wa = W.copy()
        M = beta * M + (1 - beta) * np.outer(K[t], K[t] @ Wa - V[t])
        W = W - alpha * M
        Z[t] = Q[t] @ W
    # the kernel's tiles: transposed states, beta powers as a table
    pw = beta ** np.arange(18)
    c = np.cumsum(pw[1:17])                                   # c[t] = beta + ... + beta^(t+1)
    t16 = np.arange(16)
    D = np.tril(1.0 - pw[np.clip(t16[:, None] - t16[None, :] + 1, 0, 17)])
    Wt, Mt, Zk = W0.T.copy(), np.zeros((d, d)), np.zeros((T, d))
    for c0 in range(0, T, 16):
        n = min(16, T - c0)
        Qc, Kc, Vc = (np.zeros((16, d)) for _ in range(3))
        Qc[:n], Kc[:n], Vc[:n] = Q[c0:c0 + n], K[c0:c0 + n], V[c0:c0 + n]
        Et = Wt @ Kc.T - Vc.T                                 # rows j, columns t
        S = np.tril(Qc @ Kc.T)
        Zt = Wt @ Qc.T - alpha * (Mt @ Qc.T) * c[None, :] - alpha * Et @ (S * D).T
        Zk[c0:c0 + n] = Zt.T[:n]
        dvec = np.where(t16 < n, 1.0 - pw[np.clip(n - t16, 0, 17)], 0.0)
        wvec = np.where(t16 < n, pw[np.clip(n - 1 - t16, 0, 17)], 0.0)
        Wt = Wt - alpha * c[n - 1] * Mt - alpha * (Et * dvec[None, :]) @ Kc
        Mt = pw[n] * Mt + (1 - beta) * (Et * wvec[None, :]) @ Kc
    assert np.allclose(Zk, Z, rtol=0, atol=1e-12)
    assert np.allclose(Wt.T, W, rtol=0, atol=1e-12) and np.allclose(Mt.T, M, rtol=0, atol=1e-12)
