"""Python binding of the B300 chunked TTT scan library (libttt_b300.so).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels. torch provides device memory and the current stream; the functions
take torch CUDA tensors, pass their data pointers to the C ABI of
include/ttt.h and raise on a non-OK status. There is no CPU fallback: if the
library is missing or no GPU is present the calls fail loudly.

Names match the C entry points: ttt_workspace_bytes(_ex), ttt_linear_plan, ttt_linear_fwd,
ttt_linear_bias_fwd, ttt_linear_token_eta_fwd, ttt_linear_ln_fwd, ttt_linear_momentum_fwd,
ttt_linear_variant_workspace_bytes (the variants' *_ex calls are reached through fast=True),
ttt_mlp_fwd, ttt_mlp_fwd_noalloc, ttt_mlp_noalloc_last_device_status, ttt_linear_decode_step, ttt_linear_bwd_workspace_bytes,
ttt_linear_bwd, ttt_mlp_bwd_workspace_bytes, ttt_mlp_bwd, ttt_last_device_status, ttt_status_str. The *_fwd_ex forms are reached
through the options argument.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libttt_b300.so")

TTT_OK, TTT_ERR_ARG, TTT_ERR_UNSUPPORTED, TTT_ERR_CUDA, TTT_ERR_TIMEOUT, TTT_ERR_DEVICE_CHECK = 0, -1, -2, -3, -4, -5
TTT_F32, TTT_BF16 = 0, 1
TTT_VARIANT_LINEAR, TTT_VARIANT_MLP = 0, 1
TTT_INNER_BIAS, TTT_INNER_TOKEN_ETA, TTT_INNER_LN, TTT_INNER_MOMENTUM = 1, 2, 3, 4
PATH_AUTO, PATH_SIMT, PATH_TENSOR, PATH_SEGMENTED = 0, 1, 2, 3

# Every entry point include/ttt.h declares.
EXPORTS = ("ttt_workspace_bytes", "ttt_workspace_bytes_ex", "ttt_linear_plan", "ttt_linear_fwd", "ttt_linear_fwd_ex", "ttt_mlp_fwd", "ttt_mlp_fwd_ex",
           "ttt_mlp_fwd_noalloc", "ttt_mlp_noalloc_last_device_status", "ttt_linear_decode_step", "ttt_linear_bwd_workspace_bytes", "ttt_linear_bwd",
           "ttt_last_device_status", "ttt_status_str", "ttt_linear_bias_fwd", "ttt_linear_token_eta_fwd",
           "ttt_linear_ln_fwd", "ttt_linear_momentum_fwd", "ttt_linear_decode",
           "ttt_linear_variant_workspace_bytes", "ttt_linear_bias_fwd_ex", "ttt_linear_token_eta_fwd_ex",
           "ttt_mlp_bwd_workspace_bytes", "ttt_mlp_bwd", "ttt_linear_momentum_fwd_ex",
           "ttt_linear_ln_fwd_ex")


class TTTError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({ttt_status_str(status)})")


class ttt_options(ctypes.Structure):
    _fields_ = [("wait_timeout_ns", ctypes.c_uint64), ("inject_stall", ctypes.c_int32),
                ("force_path", ctypes.c_int32), ("seg_len", ctypes.c_int32),
                ("phase_events", ctypes.c_void_p), ("pieces", ctypes.c_int32)]


class ttt_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("seg_len", ctypes.c_int32), ("seg_count", ctypes.c_int32),
                ("kernels", ctypes.c_int32), ("affine", ctypes.c_int32), ("pieces", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libttt_b300.so (raises if it has not been built) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.ttt_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.ttt_workspace_bytes.restype = sz
    lib.ttt_workspace_bytes_ex.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ttt_options)]
    lib.ttt_workspace_bytes_ex.restype = sz
    lib.ttt_linear_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ttt_options), ctypes.POINTER(ttt_plan)]
    lib.ttt_linear_plan.restype = i
    lin = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp, vp, vp, sz, vp]
    lib.ttt_linear_fwd.argtypes = lin
    lib.ttt_linear_fwd_ex.argtypes = lin + [ctypes.POINTER(ttt_options)]
    mlp = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
    lib.ttt_mlp_fwd.argtypes = mlp
    lib.ttt_mlp_fwd_ex.argtypes = mlp + [ctypes.POINTER(ttt_options)]
    lib.ttt_mlp_fwd_noalloc.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp]
    lib.ttt_mlp_noalloc_last_device_status.argtypes = [vp]
    lib.ttt_linear_decode_step.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp]
    lib.ttt_linear_decode.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.ttt_last_device_status.argtypes = [vp, vp]
    lib.ttt_linear_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.ttt_linear_bwd_workspace_bytes.restype = sz
    lib.ttt_linear_bwd.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ttt_linear_bias_fwd.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp]
    lib.ttt_linear_token_eta_fwd.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp, vp, vp]
    lib.ttt_linear_ln_fwd.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, i, i, i, i, i, vp, vp, vp]
    lib.ttt_linear_momentum_fwd.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp]
    lib.ttt_mlp_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.ttt_mlp_bwd_workspace_bytes.restype = sz
    lib.ttt_mlp_bwd.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                vp]
    lib.ttt_linear_variant_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.ttt_linear_variant_workspace_bytes.restype = sz
    lib.ttt_linear_bias_fwd_ex.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp, sz, vp]
    lib.ttt_linear_token_eta_fwd_ex.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp, vp, vp, sz, vp]
    lib.ttt_linear_momentum_fwd_ex.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp, sz, vp, vp]
    lib.ttt_linear_ln_fwd_ex.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, i, i, i, i, i, vp, vp, vp, sz, vp, vp]
    lib.ttt_status_str.argtypes = [i]
    lib.ttt_status_str.restype = ctypes.c_char_p
    for f in ("ttt_linear_fwd", "ttt_linear_fwd_ex", "ttt_mlp_fwd", "ttt_mlp_fwd_ex", "ttt_mlp_fwd_noalloc",
              "ttt_mlp_noalloc_last_device_status", "ttt_linear_bias_fwd", "ttt_linear_token_eta_fwd",
              "ttt_linear_ln_fwd", "ttt_linear_momentum_fwd", "ttt_linear_decode", "ttt_linear_bias_fwd_ex",
              "ttt_linear_token_eta_fwd_ex", "ttt_linear_momentum_fwd_ex", "ttt_linear_ln_fwd_ex", "ttt_mlp_bwd",
              "ttt_linear_decode_step", "ttt_linear_bwd", "ttt_last_device_status"):
        getattr(lib, f).restype = i
    _lib = lib
    return lib


def ttt_status_str(status: int) -> str:
    return load_library().ttt_status_str(int(status)).decode()


def ttt_workspace_bytes(B: int, H: int, T: int, d: int, b: int, variant: int = TTT_VARIANT_LINEAR,
                        options=None) -> int:
    lib = load_library()
    if options is None:
        return int(lib.ttt_workspace_bytes(B, H, T, d, b, variant))
    return int(lib.ttt_workspace_bytes_ex(B, H, T, d, b, variant, _opts(options)))


def ttt_linear_plan(B: int, H: int, T: int, d: int, b: int, dtype: int = TTT_BF16, options=None) -> dict:
    """How ttt_linear_fwd runs for these sizes: {path, seg_len, seg_count, kernels, affine, pieces}."""
    out = ttt_plan()
    st = load_library().ttt_linear_plan(B, H, T, d, b, dtype, _opts(options), ctypes.byref(out))
    if st != TTT_OK:
        raise TTTError("ttt_linear_plan", st)
    return {f: int(getattr(out, f)) for f, _ in ttt_plan._fields_}


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return TTT_BF16
    if t.dtype == torch.float32:
        return TTT_F32
    raise TypeError(f"Q/K/V must be bfloat16 or float32, got {t.dtype}")


def _is_device_tensor(t) -> bool:
    import torch
    return isinstance(t, torch.Tensor) and t.is_cuda


def _check(t, name, dtype=None, shape=None, device=None):
    """t is a contiguous CUDA tensor of this dtype and shape on this device (None: any)."""
    if not _is_device_tensor(t):
        raise TypeError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}; the call's tensors are on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _on_device(device):
    """Context that makes `device` current for a call (nothing to do if it already is, as inside
    a stream capture on that device)."""
    import contextlib

    import torch
    if device.index is None or torch.cuda.current_device() == device.index:
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _stream_ptr(stream, device=None):
    """The stream to enqueue on: `stream`, which must belong to `device`, or the device's current one."""
    import torch
    s = torch.cuda.current_stream(device) if stream is None else stream
    if device is not None and getattr(s, "device", device) != device:
        raise ValueError(f"stream is on {s.device}; the call's tensors are on {device}")
    return ctypes.c_void_p(s.cuda_stream)


def _opts(options):
    if options is None:
        return None
    if isinstance(options, ttt_options):
        return ctypes.byref(options)
    o = ttt_options()
    for k, v in dict(options).items():
        setattr(o, k, v)
    return ctypes.byref(o)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def ttt_linear_fwd(Q, K, V, eta, W0, b: int, Z=None, W_out=None, workspace=None, stream=None, options=None):
    """TTT-Linear over [B, H, T, d] sequences; returns (Z, W_out). Asynchronous on `stream`."""
    import torch
    lib = load_library()
    B, H, T, d = Q.shape
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check(t, n, Q.dtype, (B, H, T, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W0, "W0", torch.float32, (H, d, d), dev)
    if Z is None:
        Z = torch.empty_like(Q)
    if W_out is None:
        W_out = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    _check(Z, "Z", Q.dtype, (B, H, T, d), dev)
    _check(W_out, "W_out", torch.float32, (B, H, d, d), dev)
    with _on_device(dev):
        need = ttt_workspace_bytes(B, H, T, d, b, TTT_VARIANT_LINEAR, options)
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(workspace, "workspace", device=dev)
        args = (_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W0), B, H, T, d, int(b), _p(Z), _p(W_out),
                _p(workspace), _nbytes(workspace), _stream_ptr(stream, dev))
        if options is None:
            st = lib.ttt_linear_fwd(*args)
        else:
            st = lib.ttt_linear_fwd_ex(*args, _opts(options))
    if st != TTT_OK:
        raise TTTError("ttt_linear_fwd", st)
    return Z, W_out


def ttt_mlp_fwd(Q, K, V, eta, W1_0, W2_0, b: int, Z=None, W1_out=None, W2_out=None, workspace=None,
                stream=None, options=None):
    """TTT-MLP (hidden 4d, tanh-GELU) over [B, H, T, d]; returns (Z, W1_out, W2_out)."""
    import torch
    lib = load_library()
    B, H, T, d = Q.shape
    m = 4 * d
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check(t, n, Q.dtype, (B, H, T, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W1_0, "W1_0", torch.float32, (H, d, m), dev)
    _check(W2_0, "W2_0", torch.float32, (H, m, d), dev)
    if Z is None:
        Z = torch.empty_like(Q)
    if W1_out is None:
        W1_out = torch.empty((B, H, d, m), dtype=torch.float32, device=dev)
    if W2_out is None:
        W2_out = torch.empty((B, H, m, d), dtype=torch.float32, device=dev)
    _check(Z, "Z", Q.dtype, (B, H, T, d), dev)
    _check(W1_out, "W1_out", torch.float32, (B, H, d, m), dev)
    _check(W2_out, "W2_out", torch.float32, (B, H, m, d), dev)
    with _on_device(dev):
        need = ttt_workspace_bytes(B, H, T, d, b, TTT_VARIANT_MLP)
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(workspace, "workspace", device=dev)
        args = (_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W1_0), _p(W2_0), B, H, T, d, int(b), _p(Z),
                _p(W1_out), _p(W2_out), _p(workspace), _nbytes(workspace), _stream_ptr(stream, dev))
        if options is None:
            st = lib.ttt_mlp_fwd(*args)
        else:
            st = lib.ttt_mlp_fwd_ex(*args, _opts(options))
    if st != TTT_OK:
        raise TTTError("ttt_mlp_fwd", st)
    return Z, W1_out, W2_out


def ttt_mlp_fwd_noalloc(Q, K, V, eta, W1_0, W2_0, b: int, Z=None, W1_out=None, W2_out=None, stream=None):
    """TTT-MLP without a workspace, for callers that cannot allocate device memory: the library's fixed
    scratch array serves instead (any number of units on the tensor-core kernel; at d = 64 up to 64 units
    on the fp32 SIMT kernel). Calls that overlap on the GPU race on that array."""
    import torch
    lib = load_library()
    B, H, T, d = Q.shape
    m = 4 * d
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check(t, n, Q.dtype, (B, H, T, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W1_0, "W1_0", torch.float32, (H, d, m), dev)
    _check(W2_0, "W2_0", torch.float32, (H, m, d), dev)
    Z = torch.empty_like(Q) if Z is None else Z
    W1_out = torch.empty((B, H, d, m), dtype=torch.float32, device=dev) if W1_out is None else W1_out
    W2_out = torch.empty((B, H, m, d), dtype=torch.float32, device=dev) if W2_out is None else W2_out
    _check(Z, "Z", Q.dtype, (B, H, T, d), dev)
    _check(W1_out, "W1_out", torch.float32, (B, H, d, m), dev)
    _check(W2_out, "W2_out", torch.float32, (B, H, m, d), dev)
    with _on_device(dev):
        st = lib.ttt_mlp_fwd_noalloc(_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W1_0), _p(W2_0), B, H, T,
                                     d, int(b), _p(Z), _p(W1_out), _p(W2_out), _stream_ptr(stream, dev))
    if st != TTT_OK:
        raise TTTError("ttt_mlp_fwd_noalloc", st)
    return Z, W1_out, W2_out


def ttt_mlp_noalloc_last_device_status(stream=None, device=None) -> int:
    """Wait for the stream, then read and clear the status word of ttt_mlp_fwd_noalloc's fixed array
    on `device` (default: the current device)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with _on_device(dev):
        return int(load_library().ttt_mlp_noalloc_last_device_status(_stream_ptr(stream, dev)))


def _variant_prologue(Q, K, V, W0):
    import torch
    B, H, T, d = Q.shape
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check(t, n, Q.dtype, (B, H, T, d), dev)
    _check(W0, "W0", torch.float32, (H, d, d), dev)
    Z = torch.empty_like(Q)
    W_out = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    return B, H, T, d, dev, Z, W_out


def _variant_call(name, *args, dev):
    with _on_device(dev):
        st = getattr(load_library(), name)(*args)
    if st != TTT_OK:
        raise TTTError(name, st)


def ttt_linear_variant_workspace_bytes(variant: int, dtype: int, B: int, H: int, T: int, d: int, b: int) -> int:
    return int(load_library().ttt_linear_variant_workspace_bytes(variant, dtype, B, H, T, d, b))


def _variant_workspace(variant, Q, B, H, T, d, b, dev, workspace):
    import torch
    need = ttt_linear_variant_workspace_bytes(variant, _dtype_code(Q), B, H, T, d, b)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    return workspace


def ttt_linear_bias_fwd(Q, K, V, eta, W0, beta0, b: int, stream=None, fast=False, workspace=None):
    """TTT-Linear with f(k) = k W + beta; returns (Z, W_out, beta_out). fast=True calls
    ttt_linear_bias_fwd_ex (the tensor-core path on padded inputs where it applies)."""
    import torch
    B, H, T, d, dev, Z, W_out = _variant_prologue(Q, K, V, W0)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(beta0, "beta0", torch.float32, (H, d), dev)
    beta_out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    args = (_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W0), _p(beta0), B, H, T, d, int(b), _p(Z), _p(W_out),
            _p(beta_out))
    if fast:
        ws = _variant_workspace(TTT_INNER_BIAS, Q, B, H, T, d, b, dev, workspace)
        _variant_call("ttt_linear_bias_fwd_ex", *args, _p(ws), ws.numel(), _stream_ptr(stream, dev), dev=dev)
    else:
        _variant_call("ttt_linear_bias_fwd", *args, _stream_ptr(stream, dev), dev=dev)
    return Z, W_out, beta_out


def ttt_linear_token_eta_fwd(Q, K, V, eta_tok, W0, b: int, stream=None, fast=False, workspace=None):
    """TTT-Linear with a learning rate per token, eta_tok [B, H, T]; returns (Z, W_out).
    fast=True calls ttt_linear_token_eta_fwd_ex (the tensor-core path on scaled inputs where it
    applies)."""
    import torch
    B, H, T, d, dev, Z, W_out = _variant_prologue(Q, K, V, W0)
    _check(eta_tok, "eta_tok", torch.float32, (B, H, T), dev)
    args = (_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta_tok), _p(W0), B, H, T, d, int(b), _p(Z), _p(W_out))
    if fast:
        ws = _variant_workspace(TTT_INNER_TOKEN_ETA, Q, B, H, T, d, b, dev, workspace)
        _variant_call("ttt_linear_token_eta_fwd_ex", *args, _p(ws), ws.numel(), _stream_ptr(stream, dev), dev=dev)
    else:
        _variant_call("ttt_linear_token_eta_fwd", *args, _stream_ptr(stream, dev), dev=dev)
    return Z, W_out


def ttt_linear_ln_fwd(Q, K, V, eta, W0, gamma, beta, b: int, stream=None, fast=False, workspace=None,
                      options=None):
    """TTT-Linear with f(k) = k + LN(k W) (gamma, beta [H, d]); returns (Z, W_out). fast=True calls
    ttt_linear_ln_fwd_ex (the tensor-core kernel for bf16, d = 64, b = 16), with `options` passed
    through."""
    import torch
    B, H, T, d, dev, Z, W_out = _variant_prologue(Q, K, V, W0)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(gamma, "gamma", torch.float32, (H, d), dev)
    _check(beta, "beta", torch.float32, (H, d), dev)
    args = (_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W0), _p(gamma), _p(beta), B, H, T, d, int(b), _p(Z),
            _p(W_out))
    if fast:
        ws = _variant_workspace(TTT_INNER_LN, Q, B, H, T, d, b, dev, workspace)
        _variant_call("ttt_linear_ln_fwd_ex", *args, _p(ws), ws.numel(), _stream_ptr(stream, dev), _opts(options),
                      dev=dev)
    else:
        _variant_call("ttt_linear_ln_fwd", *args, _stream_ptr(stream, dev), dev=dev)
    return Z, W_out


def ttt_linear_momentum_fwd(Q, K, V, alpha, beta, W0, b: int, stream=None, fast=False, workspace=None,
                            options=None):
    """TTT-Linear with momentum gradient descent (alpha, beta [H]); returns (Z, W_out, M_out).
    fast=True calls ttt_linear_momentum_fwd_ex (the tensor-core kernel for bf16, d = 64, b = 16),
    with `options` (a dict or ttt_options) passed through."""
    import torch
    B, H, T, d, dev, Z, W_out = _variant_prologue(Q, K, V, W0)
    _check(alpha, "alpha", torch.float32, (H,), dev)
    _check(beta, "beta", torch.float32, (H,), dev)
    M_out = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    args = (_p(Q), _p(K), _p(V), _dtype_code(Q), _p(alpha), _p(beta), _p(W0), B, H, T, d, int(b), _p(Z), _p(W_out),
            _p(M_out))
    if fast:
        ws = _variant_workspace(TTT_INNER_MOMENTUM, Q, B, H, T, d, b, dev, workspace)
        _variant_call("ttt_linear_momentum_fwd_ex", *args, _p(ws), ws.numel(), _stream_ptr(stream, dev),
                      _opts(options), dev=dev)
    else:
        _variant_call("ttt_linear_momentum_fwd", *args, _stream_ptr(stream, dev), dev=dev)
    return Z, W_out, M_out


def ttt_linear_decode_step(q, k, v, eta, W_anchor, W_run, pos: int, b: int, z=None, stream=None):
    """One decode token per (batch row, head); q, k, v [B, H, d]. Updates W_anchor/W_run in place; returns z."""
    import torch
    lib = load_library()
    B, H, d = q.shape
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check(t, n, q.dtype, (B, H, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W_anchor, "W_anchor", torch.float32, (B, H, d, d), dev)
    _check(W_run, "W_run", torch.float32, (B, H, d, d), dev)
    if z is None:
        z = torch.empty_like(q)
    _check(z, "z", q.dtype, (B, H, d), dev)
    with _on_device(dev):
        st = lib.ttt_linear_decode_step(_p(q), _p(k), _p(v), _dtype_code(q), _p(eta), _p(W_anchor), _p(W_run),
                                        B, H, d, int(pos), int(b), _p(z), _stream_ptr(stream, dev))
    if st != TTT_OK:
        raise TTTError("ttt_linear_decode_step", st)
    return z


def ttt_linear_decode(q, k, v, eta, W_anchor, W_run, pos: int, b: int, z=None, stream=None):
    """N decode tokens per (batch row, head) in one launch; q, k, v [B, H, N, d]. Updates
    W_anchor/W_run in place; returns z [B, H, N, d]."""
    import torch
    lib = load_library()
    B, H, N, d = q.shape
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check(t, n, q.dtype, (B, H, N, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W_anchor, "W_anchor", torch.float32, (B, H, d, d), dev)
    _check(W_run, "W_run", torch.float32, (B, H, d, d), dev)
    if z is None:
        z = torch.empty_like(q)
    _check(z, "z", q.dtype, (B, H, N, d), dev)
    with _on_device(dev):
        st = lib.ttt_linear_decode(_p(q), _p(k), _p(v), _dtype_code(q), _p(eta), _p(W_anchor), _p(W_run), B, H, N, d,
                                   int(pos), int(b), _p(z), _stream_ptr(stream, dev))
    if st != TTT_OK:
        raise TTTError("ttt_linear_decode", st)
    return z


def ttt_linear_bwd_workspace_bytes(B: int, H: int, T: int, d: int, b: int) -> int:
    return int(load_library().ttt_linear_bwd_workspace_bytes(B, H, T, d, b))


def ttt_linear_bwd(Q, K, V, eta, W0, b: int, dZ, dW_out, workspace=None, stream=None):
    """Backward of ttt_linear_fwd: returns (dQ, dK, dV, deta, dW0) for upstream gradients
    dZ [B, H, T, d] (the dtype of Q: float32 or bfloat16) and dW_out [B, H, d, d] float32;
    dQ, dK, dV come in the dtype of Q. Asynchronous on `stream`."""
    import torch
    lib = load_library()
    B, H, T, d = Q.shape
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V), ("dZ", dZ)):
        _check(t, n, Q.dtype, (B, H, T, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W0, "W0", torch.float32, (H, d, d), dev)
    _check(dW_out, "dW_out", torch.float32, (B, H, d, d), dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    deta = torch.empty((H,), dtype=torch.float32, device=dev)
    dW0 = torch.empty((H, d, d), dtype=torch.float32, device=dev)
    need = ttt_linear_bwd_workspace_bytes(B, H, T, d, b)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", device=dev)
    with _on_device(dev):
        st = lib.ttt_linear_bwd(_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W0), B, H, T, d, int(b), _p(dZ),
                                _p(dW_out), _p(dQ), _p(dK), _p(dV), _p(deta), _p(dW0), _p(workspace),
                                _nbytes(workspace), _stream_ptr(stream, dev))
    if st != TTT_OK:
        raise TTTError("ttt_linear_bwd", st)
    return dQ, dK, dV, deta, dW0


def ttt_mlp_bwd_workspace_bytes(B: int, H: int, T: int, d: int, b: int) -> int:
    return int(load_library().ttt_mlp_bwd_workspace_bytes(B, H, T, d, b))


def ttt_mlp_bwd(Q, K, V, eta, W1_0, W2_0, b: int, dZ, dW1_out, dW2_out, workspace=None, stream=None):
    """Backward of ttt_mlp_fwd: returns (dQ, dK, dV, deta, dW1, dW2) for upstream gradients dZ
    [B, H, T, d] (the dtype of Q), dW1_out [B, H, d, 4d] and dW2_out [B, H, 4d, d] float32.
    Asynchronous on `stream`."""
    import torch
    lib = load_library()
    B, H, T, d = Q.shape
    m = 4 * d
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V), ("dZ", dZ)):
        _check(t, n, Q.dtype, (B, H, T, d), dev)
    _check(eta, "eta", torch.float32, (H,), dev)
    _check(W1_0, "W1_0", torch.float32, (H, d, m), dev)
    _check(W2_0, "W2_0", torch.float32, (H, m, d), dev)
    _check(dW1_out, "dW1_out", torch.float32, (B, H, d, m), dev)
    _check(dW2_out, "dW2_out", torch.float32, (B, H, m, d), dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    deta = torch.empty((H,), dtype=torch.float32, device=dev)
    dW1 = torch.empty((H, d, m), dtype=torch.float32, device=dev)
    dW2 = torch.empty((H, m, d), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(ttt_mlp_bwd_workspace_bytes(B, H, T, d, b), 256), dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", device=dev)
    with _on_device(dev):
        st = lib.ttt_mlp_bwd(_p(Q), _p(K), _p(V), _dtype_code(Q), _p(eta), _p(W1_0), _p(W2_0), B, H, T, d, int(b),
                             _p(dZ), _p(dW1_out), _p(dW2_out), _p(dQ), _p(dK), _p(dV), _p(deta), _p(dW1), _p(dW2),
                             _p(workspace), _nbytes(workspace), _stream_ptr(stream, dev))
    if st != TTT_OK:
        raise TTTError("ttt_mlp_bwd", st)
    return dQ, dK, dV, deta, dW1, dW2


def ttt_last_device_status(workspace, stream=None) -> int:
    """Wait for the stream, then read and clear the workspace's device status word."""
    _check(workspace, "workspace")
    with _on_device(workspace.device):
        return int(load_library().ttt_last_device_status(_p(workspace), _stream_ptr(stream, workspace.device)))
