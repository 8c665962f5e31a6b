"""Seeded synthetic inputs for the chunked TTT scan.

The tests and the benchmark draw every input here and give the same arrays to
the CUDA library and to the fp64 oracle. This module holds none of the scan's
arithmetic: it draws numbers (counter-mode splitmix64 + Box-Muller, in
``synth.c``), L2-normalises rows and rounds to the input dtype. Each element of
a [B, H, T, d] tensor is addressed by its flat index, so one (batch row, head)
slice can be drawn on its own and match the full tensor bit for bit.

Workloads follow the pages' shapes: a 125M-parameter model has 12 heads of
width 64, long context means 128K tokens, and the TTT chunk holds b = 16 tokens
("5 · TestingTime 训练与长上下文", sections 1.1 and 3.1; "Test-Time Training
(TTT) guide", section 3). No dataset is read; these inputs stand in for the
pages' corpora.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libttt_synth.so")

STREAM_Q, STREAM_K, STREAM_V, STREAM_W0, STREAM_W1, STREAM_W2, STREAM_ETA = 1, 2, 3, 4, 5, 6, 7


def build(force: bool = False) -> str:
    """Compile synth.c into libttt_synth.so beside it (gcc, OpenMP)."""
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
        u64, i64, dp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_normal.argtypes = [u64, u64, u64, i64, dp]
        lib.synth_uniform.argtypes = [u64, u64, u64, i64, dp]
        lib.synth_normalize_rows.argtypes = [dp, i64, i64]
        lib.synth_round_bf16.argtypes = [dp, i64, dp, dp]
        lib.synth_round_f32.argtypes = [dp, i64, dp, dp]
        for f in (lib.synth_normal, lib.synth_uniform, lib.synth_normalize_rows,
                  lib.synth_round_bf16, lib.synth_round_f32):
            f.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def normal(seed: int, stream: int, count: int, first: int = 0) -> np.ndarray:
    """Standard normal draws number first .. first+count-1 of (seed, stream)."""
    out = np.empty(int(count), dtype=np.float64)
    _load().synth_normal(seed, stream, first, int(count), _ptr(out))
    return out


def uniform(seed: int, stream: int, count: int, first: int = 0) -> np.ndarray:
    """Uniform draws in (0, 1], number first .. first+count-1 of (seed, stream)."""
    out = np.empty(int(count), dtype=np.float64)
    _load().synth_uniform(seed, stream, first, int(count), _ptr(out))
    return out


def normalize_rows(x: np.ndarray) -> np.ndarray:
    """L2-normalise the last axis in place (fp64)."""
    assert x.dtype == np.float64
    d = x.shape[-1]
    _load().synth_normalize_rows(_ptr(x), x.size // d if d else 0, d)
    return x


def round_bf16(x: np.ndarray, want_exact: bool = True):
    """Round fp64 -> bf16 (RNE). Returns (uint16 bit patterns, exact fp64 values or None)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    bits = np.empty(x.shape, dtype=np.uint16)
    back = np.empty(x.shape, dtype=np.float64) if want_exact else None
    _load().synth_round_bf16(_ptr(x), x.size, _ptr(bits), _ptr(back) if back is not None else None)
    return bits, back


def round_f32(x: np.ndarray, want_exact: bool = True):
    """Round fp64 -> fp32 (RNE). Returns (float32 array, exact fp64 values or None)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    f = np.empty(x.shape, dtype=np.float32)
    back = np.empty(x.shape, dtype=np.float64) if want_exact else None
    _load().synth_round_f32(_ptr(x), x.size, _ptr(f), _ptr(back) if back is not None else None)
    return f, back


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype and value recipe."""
    name: str
    B: int
    H: int
    T: int
    d: int
    b: int
    dtype: str                    # "f32" or "bf16": the dtype of Q, K, V and Z
    seed: int
    eta: tuple                    # ("const", value) or ("uniform", lo, hi)
    w_std: float                  # std of the initial state (0 => zeros)
    q_mode: str = "normalized"    # "normalized" rows, or "scaled" by 1/sqrt(d)
    variant: str = "linear"       # "linear" or "mlp"
    hidden: int = 0               # TTT-MLP hidden width (4 d)
    note: str = field(default="", compare=False)

    @property
    def units(self) -> int:
        return self.B * self.H

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the scan (names give their sizes; seeds are fixed).
WORKLOADS = {
    "linear_tiny_f32": Workload("linear_tiny_f32", 1, 1, 64, 16, 16, "f32", 0, ("const", 0.5), 0.0,
                                q_mode="scaled",
                                note="B1 H1 T64 d16 b16, fp32, Q iid N(0,1)/sqrt(d), K rows unit, W0=0, eta=0.5"),
    "linear_small": Workload("linear_small", 2, 4, 2048, 64, 16, "bf16", 1, ("const", 0.1), 0.02,
                             note="B2 H4 T2048 d64 b16, bf16, Q/K rows unit, V N(0,1), W0 N(0,0.02^2), eta=0.1"),
    "linear_125m": Workload("linear_125m", 8, 12, 8192, 64, 16, "bf16", 2, ("uniform", 0.05, 0.5), 0.02,
                            note="B8 H12 T8192 d64 b16, bf16, eta_h ~ U[0.05,0.5]"),
    "linear_long": Workload("linear_long", 1, 32, 131072, 64, 16, "bf16", 3, ("const", 0.1), 0.02,
                            note="B1 H32 T131072 d64, b in {16,64,256}, bf16, eta=0.1"),
    "mlp_125m": Workload("mlp_125m", 4, 12, 8192, 64, 16, "bf16", 4, ("const", 0.05), 0.02,
                         variant="mlp", hidden=256,
                         note="B4 H12 T8192 d64 hidden 256 b16, bf16, W1/W2 N(0,0.02^2), eta=0.05"),
}


@dataclass
class Inputs:
    """Arrays for one workload (or one (batch row, head) slice of it).

    ``q, k, v`` are what the GPU reads: uint16 bf16 bit patterns or float32,
    shape [B, H, T, d]. ``q64, k64, v64`` are their exact fp64 values (None if
    not requested). ``eta`` [H] and the initial state are float32, with fp64
    copies: W0 [H, d, d] (TTT-Linear) or W1 [H, d, m], W2 [H, m, d] (TTT-MLP).
    """
    w: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    q64: np.ndarray | None
    k64: np.ndarray | None
    v64: np.ndarray | None
    eta: np.ndarray
    eta64: np.ndarray
    W0: np.ndarray | None = None
    W0_64: np.ndarray | None = None
    W1: np.ndarray | None = None
    W1_64: np.ndarray | None = None
    W2: np.ndarray | None = None
    W2_64: np.ndarray | None = None


_BLOCK_ROWS = 1 << 18


def _tensor(w: Workload, stream: int, normalize: bool, scale: float, first_row: int, rows: int,
            want_exact: bool):
    d = w.d
    if w.dtype == "bf16":
        out = np.empty((rows, d), dtype=np.uint16)
    else:
        out = np.empty((rows, d), dtype=np.float32)
    exact = np.empty((rows, d), dtype=np.float64) if want_exact else None
    for r0 in range(0, rows, _BLOCK_ROWS):
        r1 = min(rows, r0 + _BLOCK_ROWS)
        x = normal(w.seed, stream, (r1 - r0) * d, (first_row + r0) * d).reshape(r1 - r0, d)
        if normalize:
            normalize_rows(x)
        if scale != 1.0:
            x *= scale
        if w.dtype == "bf16":
            bits, back = round_bf16(x, want_exact)
            out[r0:r1] = bits
        else:
            f, back = round_f32(x, want_exact)
            out[r0:r1] = f
        if want_exact:
            exact[r0:r1] = back
    return out, exact


def _state(w: Workload, stream: int, shape):
    n = int(np.prod(shape))
    if w.w_std == 0.0:
        x = np.zeros(n)
    else:
        x = w.w_std * normal(w.seed, stream, n)
    f, back = round_f32(x)
    return f.reshape(shape), back.reshape(shape)


def make_eta(w: Workload):
    if w.eta[0] == "const":
        x = np.full(w.H, float(w.eta[1]))
    else:
        lo, hi = float(w.eta[1]), float(w.eta[2])
        x = lo + (hi - lo) * uniform(w.seed, STREAM_ETA, w.H)
    f, back = round_f32(x)
    return f, back


def make_inputs(w: Workload, units=None, want_exact: bool = True) -> Inputs:
    """Draw the inputs of workload ``w``.

    ``units`` = None draws the whole [B, H, T, d] tensors. A list of (n, h)
    pairs draws only those slices as one batch row of len(units) heads,
    [1, len(units), T, d], identical to the same slices of the full draw; eta
    and the initial state are then the heads' own ([len(units)] and
    [len(units), ...]).
    """
    qscale = 1.0
    qnorm = True
    if w.q_mode == "scaled":
        qnorm, qscale = False, 1.0 / np.sqrt(w.d)
    eta, eta64 = make_eta(w)
    if w.variant == "mlp":
        m = w.hidden
        W1, W1_64 = _state(w, STREAM_W1, (w.H, w.d, m))
        W2, W2_64 = _state(w, STREAM_W2, (w.H, m, w.d))
        W0 = W0_64 = None
    else:
        W0, W0_64 = _state(w, STREAM_W0, (w.H, w.d, w.d))
        W1 = W1_64 = W2 = W2_64 = None
    if units is None:
        rows = w.B * w.H * w.T
        q, q64 = _tensor(w, STREAM_Q, qnorm, qscale, 0, rows, want_exact)
        k, k64 = _tensor(w, STREAM_K, True, 1.0, 0, rows, want_exact)
        v, v64 = _tensor(w, STREAM_V, False, 1.0, 0, rows, want_exact)
        shp = (w.B, w.H, w.T, w.d)
        rs = (lambda a: None if a is None else a.reshape(shp))
        return Inputs(w, q.reshape(shp), k.reshape(shp), v.reshape(shp), rs(q64), rs(k64), rs(v64),
                      eta, eta64, W0, W0_64, W1, W1_64, W2, W2_64)
    parts = {key: [] for key in ("q", "k", "v", "q64", "k64", "v64")}
    hs = []
    for (n, h) in units:
        first_row = (n * w.H + h) * w.T
        for name, stream, norm, sc in (("q", STREAM_Q, qnorm, qscale), ("k", STREAM_K, True, 1.0),
                                       ("v", STREAM_V, False, 1.0)):
            a, a64 = _tensor(w, stream, norm, sc, first_row, w.T, want_exact)
            parts[name].append(a.reshape(1, w.T, w.d))
            parts[name + "64"].append(None if a64 is None else a64.reshape(1, w.T, w.d))
        hs.append(h)
    hs = np.array(hs)
    st = (lambda L: None if L[0] is None else np.concatenate(L).reshape(1, len(L), w.T, w.d))
    sel = (lambda a: None if a is None else np.ascontiguousarray(a[hs]))
    return Inputs(w, st(parts["q"]), st(parts["k"]), st(parts["v"]), st(parts["q64"]),
                  st(parts["k64"]), st(parts["v64"]), np.ascontiguousarray(eta[hs]),
                  np.ascontiguousarray(eta64[hs]), sel(W0), sel(W0_64), sel(W1), sel(W1_64),
                  sel(W2), sel(W2_64))
