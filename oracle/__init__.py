"""ORACLE: plain fp64 CPU reference of the chunked TTT scan (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library never loads it and shares no
code with it. The arithmetic lives in ``ttt_oracle.c`` (plain C, fp64, OpenMP
over (batch row, head) units); this file compiles it with gcc on first use and
marshals numpy arrays.

What it computes, and the passages it follows, is in the C file's header. In
short: TTT-Linear and TTT-MLP, per-token primal form (the reference) and a
separate per-chunk dual form (kept to pin primal == dual), the affine map of
each segment of chunks (the segment-parallel form), plus one decode token with
an (anchor, running) weight pair. ``oracle.backward.linear_backward`` (numpy,
fp64, small cases) is the backward of the TTT-Linear scan: dQ, dK, dV, deta and
dW0 for upstream dZ and dW_out, pinned in tests/test_oracle_backward.py.
``oracle.variants`` (numpy, fp64) holds TTT-Linear with a layer norm and a
residual inside the inner model, pinned in tests/test_oracle_variants.py.

Parity pins live in tests/test_oracle_pins.py (b = 1 delta rule; causal linear
attention; finite differences and autograd; eta = 0; chaining; b = T closed
form; hand-worked scalar examples in tests/golden/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ttt_oracle.c")
_LIB = os.path.join(_HERE, "libttt_oracle.so")


def build(force: bool = False) -> str:
    """Compile ttt_oracle.c into libttt_oracle.so beside it (gcc -O2, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lin = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, dp, dp, ci]
        mlp = [dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, i64, dp, dp, dp, ci]
        for name, args in (("oracle_linear_primal", lin), ("oracle_linear_dual", lin),
                           ("oracle_mlp_primal", mlp), ("oracle_mlp_dual", mlp),
                           ("oracle_linear_decode_step",
                            [dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, dp])):
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ci
        lib.oracle_linear_segment_maps.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64, dp, dp, ci]
        lib.oracle_linear_segment_maps.restype = ci
        lib.oracle_gelu_array.argtypes = [dp, i64, dp, dp]
        lib.oracle_gelu_array.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ci
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_load().oracle_max_threads())


def _linear(fn, Q, K, V, eta, W0, b, nthreads):
    Q, K, V, eta, W0 = map(_f64, (Q, K, V, eta, W0))
    B, H, T, d = Q.shape
    assert K.shape == Q.shape and V.shape == Q.shape
    assert eta.shape == (H,) and W0.shape == (H, d, d)
    Z = np.empty_like(Q)
    W = np.empty((B, H, d, d))
    rc = fn(_p(Q), _p(K), _p(V), _p(eta), _p(W0), B, H, T, d, int(b), _p(Z), _p(W), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")
    return Z, W


def linear_primal(Q, K, V, eta, W0, b, nthreads: int = 0):
    """TTT-Linear, per-token primal form. Q, K, V [B,H,T,d]; eta [H]; W0 [H,d,d].
    Returns (Z [B,H,T,d], W_out [B,H,d,d]) in fp64."""
    return _linear(_load().oracle_linear_primal, Q, K, V, eta, W0, b, nthreads)


def linear_dual(Q, K, V, eta, W0, b, nthreads: int = 0):
    """TTT-Linear, per-chunk dual form (same results as linear_primal up to rounding)."""
    return _linear(_load().oracle_linear_dual, Q, K, V, eta, W0, b, nthreads)


def linear_segment_maps(K, V, eta, b, L, nthreads: int = 0):
    """Affine map of every L-token segment of TTT-Linear (L a multiple of b):
    the segment takes its start state W to A_s W + B_s. K, V [B,H,T,d]; eta [H].
    Returns (A [B,H,S,d,d], B [B,H,S,d,d]) in fp64, S = ceil(T / L)."""
    K, V, eta = map(_f64, (K, V, eta))
    B, H, T, d = K.shape
    assert V.shape == K.shape and eta.shape == (H,)
    S = (T + L - 1) // L
    A = np.empty((B, H, S, d, d))
    Bm = np.empty((B, H, S, d, d))
    rc = _load().oracle_linear_segment_maps(_p(K), _p(V), _p(eta), B, H, T, d, int(b), int(L), _p(A), _p(Bm),
                                             int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")
    return A, Bm


def _mlp(fn, Q, K, V, eta, W1, W2, b, nthreads):
    Q, K, V, eta, W1, W2 = map(_f64, (Q, K, V, eta, W1, W2))
    B, H, T, d = Q.shape
    m = W1.shape[-1]
    assert W1.shape == (H, d, m) and W2.shape == (H, m, d) and eta.shape == (H,)
    Z = np.empty_like(Q)
    W1o = np.empty((B, H, d, m))
    W2o = np.empty((B, H, m, d))
    rc = fn(_p(Q), _p(K), _p(V), _p(eta), _p(W1), _p(W2), B, H, T, d, m, int(b), _p(Z), _p(W1o),
            _p(W2o), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")
    return Z, W1o, W2o


def mlp_primal(Q, K, V, eta, W1, W2, b, nthreads: int = 0):
    """TTT-MLP (tanh-GELU, hidden m = W1.shape[-1]), per-token primal form.
    Returns (Z, W1_out [B,H,d,m], W2_out [B,H,m,d])."""
    return _mlp(_load().oracle_mlp_primal, Q, K, V, eta, W1, W2, b, nthreads)


def mlp_dual(Q, K, V, eta, W1, W2, b, nthreads: int = 0):
    """TTT-MLP, per-chunk dual form (same results as mlp_primal up to rounding)."""
    return _mlp(_load().oracle_mlp_dual, Q, K, V, eta, W1, W2, b, nthreads)


def linear_decode_step(q, k, v, eta, W_anchor, W_run, pos, b):
    """One TTT-Linear token per (batch row, head); q, k, v [B,H,d].
    Returns (z [B,H,d], W_anchor', W_run') without modifying the arguments."""
    q, k, v, eta = map(_f64, (q, k, v, eta))
    Wa = np.array(W_anchor, dtype=np.float64, copy=True, order="C")
    Wr = np.array(W_run, dtype=np.float64, copy=True, order="C")
    B, H, d = q.shape
    z = np.empty_like(q)
    rc = _load().oracle_linear_decode_step(_p(q), _p(k), _p(v), _p(eta), _p(Wa), _p(Wr), B, H, d,
                                           int(pos), int(b), _p(z))
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")
    return z, Wa, Wr


def gelu(x):
    """tanh-GELU in fp64, elementwise."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_gelu_array(_p(x), x.size, _p(y), None)
    return y


def gelu_prime(x):
    """Derivative of tanh-GELU in fp64, elementwise."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_gelu_array(_p(x), x.size, None, _p(y))
    return y
