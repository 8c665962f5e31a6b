"""The C ABI without a GPU: the library loads, exports every declared entry
point, sizes its workspace and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import test_sequence_layers_06_b300 as ttt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from test_sequence_layers_06_b300 import build
    build.build()
    return ttt.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ttt.h")).read()
    return sorted(set(re.findall(r"TTT_API\s+[\w\s\*]+?\b(ttt_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) == 26
    assert set(names) == set(ttt.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert ttt.ttt_status_str(0) == "ok"
    assert "argument" in ttt.ttt_status_str(-1)
    assert "time" in ttt.ttt_status_str(-4)


def test_workspace_bytes(lib):
    assert ttt.ttt_workspace_bytes(1, 32, 131072, 64, 16, 0) >= 256
    mlp = ttt.ttt_workspace_bytes(4, 12, 8192, 64, 16, 1)
    assert mlp >= 256 + 4 * 12 * 2 * 64 * 256 * 4
    assert ttt.ttt_workspace_bytes(0, 1, 1, 64, 16, 0) == 0
    assert ttt.ttt_workspace_bytes(1, 1, 1, 64, 0, 0) == 0
    assert ttt.ttt_workspace_bytes(1, 1, 1, 64, 16, 7) == 0


def test_workspace_bytes_for_the_segment_parallel_form(lib):
    """bf16 TTT-Linear with few units is cut into segments whose affine maps and
    start states live in the workspace: 3 d^2 floats per segment boundary."""
    base = ttt.ttt_workspace_bytes(1, 32, 131072, 64, 16, 0)
    assert base > 256 and (base - 256) % (3 * 32 * 64 * 64 * 4) == 0
    # a forced one-pass run needs only the status block; a forced segment length sets the count
    assert ttt.ttt_workspace_bytes(1, 32, 131072, 64, 16, 0, {"force_path": ttt.PATH_TENSOR}) == 256
    seg = ttt.ttt_workspace_bytes(2, 3, 1000, 64, 16, 0, {"force_path": ttt.PATH_SEGMENTED, "seg_len": 256})
    assert seg == 256 + 3 * (2 * 3) * 3 * 64 * 64 * 4  # ceil(1000 / 256) = 4 segments, 3 boundaries
    # plenty of units: one pass
    assert ttt.ttt_workspace_bytes(64, 64, 8192, 64, 16, 0) == 256


def test_linear_plan(lib):
    assert ttt.ttt_linear_plan(1, 32, 131072, 64, 16)["path"] == 3
    p = ttt.ttt_linear_plan(2, 3, 1000, 64, 16, options={"force_path": ttt.PATH_SEGMENTED, "seg_len": 256})
    assert p == {"path": 3, "seg_len": 256, "seg_count": 4, "kernels": 3, "affine": 2, "pieces": 1}
    # pieces: clamped to the segment count; three kernels per piece; -1 is refused
    p = ttt.ttt_linear_plan(2, 3, 1000, 64, 16, options={"force_path": ttt.PATH_SEGMENTED, "seg_len": 256,
                                                         "pieces": 3})
    assert p["pieces"] == 3 and p["kernels"] == 9
    assert ttt.ttt_linear_plan(2, 3, 1000, 64, 16, options={"force_path": ttt.PATH_SEGMENTED, "seg_len": 256,
                                                            "pieces": 9})["pieces"] == 4
    with pytest.raises(ttt.TTTError):
        ttt.ttt_linear_plan(2, 3, 1000, 64, 16, options={"pieces": -1})
    p = ttt.ttt_linear_plan(2, 3, 1000, 64, 16, options={"force_path": ttt.PATH_SEGMENTED, "seg_len": 48})
    assert p["affine"] == 1  # 48-token segments are not whole 64-token steps
    assert ttt.ttt_linear_plan(1, 1, 100, 64, 16)["path"] == 2       # too short to cut
    assert ttt.ttt_linear_plan(1, 1, 100, 32, 16)["path"] == 1       # width the tensor kernels do not take
    assert ttt.ttt_linear_plan(1, 1, 100, 64, 16, ttt.TTT_F32)["path"] == 1
    assert ttt.ttt_linear_plan(1, 1, 0, 64, 16)["kernels"] == 0
    with pytest.raises(ttt.TTTError):
        ttt.ttt_linear_plan(1, 1, 100, 64, 16, options={"force_path": ttt.PATH_SEGMENTED, "seg_len": 24})


MB = 1 << 20  # fake device addresses 1 MB apart: no two buffers of these small calls overlap


def _lin(lib, **kw):
    a = dict(Q=1 * MB, K=2 * MB, V=3 * MB, dt=1, eta=4 * MB, W0=5 * MB, B=1, H=1, T=16, d=64, b=16, Z=6 * MB,
             W=7 * MB, ws=8 * MB, wsb=1 << 20, s=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.ttt_linear_fwd(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]), vp(a["W0"]), a["B"],
                              a["H"], a["T"], a["d"], a["b"], vp(a["Z"]), vp(a["W"]), vp(a["ws"]), a["wsb"],
                              vp(a["s"]))


@pytest.mark.parametrize("kw", [dict(Q=0), dict(K=4100), dict(eta=0), dict(W0=8), dict(ws=0), dict(wsb=16),
                                dict(B=0), dict(H=-1), dict(T=-1), dict(b=0), dict(d=0), dict(dt=5),
                                dict(Z=0)])
def test_linear_rejects_bad_arguments(lib, kw):
    assert _lin(lib, **kw) == ttt.TTT_ERR_ARG


def test_linear_rejects_unsupported_width(lib):
    assert _lin(lib, d=65) == ttt.TTT_ERR_UNSUPPORTED


def test_forced_tensor_path_rejects_shapes_it_cannot_serve(lib):
    vp = ctypes.c_void_p
    o = ttt.ttt_options(0, 0, ttt.PATH_TENSOR)
    for kw in (dict(d=32), dict(b=8), dict(dt=0)):
        a = dict(dt=1, d=64, b=16)
        a.update(kw)
        st = lib.ttt_linear_fwd_ex(vp(4096), vp(4096), vp(4096), a["dt"], vp(4096), vp(4096), 1, 1, 16, a["d"],
                                   a["b"], vp(4096), vp(4096), vp(4096), 1 << 20, vp(0), ctypes.byref(o))
        assert st == ttt.TTT_ERR_UNSUPPORTED, kw


def test_segment_options_are_checked(lib):
    vp = ctypes.c_void_p

    def call(o, b=16, dt=1):
        return lib.ttt_linear_fwd_ex(vp(4096), vp(4096), vp(4096), dt, vp(4096), vp(4096), 1, 1, 1024, 64, b,
                                     vp(4096), vp(4096), vp(4096), 1 << 20, vp(0), ctypes.byref(o))
    assert call(ttt.ttt_options(0, 0, ttt.PATH_SEGMENTED, 40)) == ttt.TTT_ERR_ARG   # not a multiple of 16
    assert call(ttt.ttt_options(0, 0, ttt.PATH_SEGMENTED, 48), b=32) == ttt.TTT_ERR_ARG  # not a multiple of b
    assert call(ttt.ttt_options(0, 0, ttt.PATH_SEGMENTED, -16)) == ttt.TTT_ERR_ARG
    assert call(ttt.ttt_options(0, 0, 4, 0)) == ttt.TTT_ERR_ARG
    assert call(ttt.ttt_options(0, 0, ttt.PATH_SEGMENTED, 0), dt=0) == ttt.TTT_ERR_UNSUPPORTED
    assert call(ttt.ttt_options(0, 0, ttt.PATH_SEGMENTED, 0), b=8) == ttt.TTT_ERR_UNSUPPORTED


def test_segment_grid_must_fit_a_launch(lib):
    """One read-out CTA per (unit, segment) and 8 combine CTAs per unit: a forced segment length
    whose grids would need 2^31 or more CTAs is refused before anything is enqueued."""
    plan = ttt.ttt_plan()
    o = ttt.ttt_options(0, 0, ttt.PATH_SEGMENTED, 16)
    assert lib.ttt_linear_plan(65536, 1024, 1024, 64, 16, 1, ctypes.byref(o), ctypes.byref(plan)) == \
        ttt.TTT_ERR_UNSUPPORTED  # 2^26 units x 64 segments
    assert lib.ttt_linear_plan(65536, 512, 1024, 64, 16, 1, ctypes.byref(o), ctypes.byref(plan)) == \
        ttt.TTT_ERR_UNSUPPORTED  # exactly 2^31
    assert lib.ttt_linear_plan(65536, 511, 1024, 64, 16, 1, ctypes.byref(o), ctypes.byref(plan)) == ttt.TTT_OK
    assert (plan.path, plan.seg_len, plan.seg_count) == (3, 16, 64)  # 2^31 - 2^22 CTAs: still fits


def test_mlp_and_decode_reject_bad_arguments(lib):
    vp = ctypes.c_void_p
    st = lib.ttt_mlp_fwd(vp(4096), vp(4096), vp(4096), 1, vp(4096), vp(4096), vp(4096), 1, 1, 16, 64, 16,
                         vp(4096), vp(4096), vp(4096), vp(4096), 256, vp(0))
    assert st == ttt.TTT_ERR_ARG  # workspace too small for the snapshot
    st = lib.ttt_linear_decode_step(vp(4096), vp(4096), vp(4096), 1, vp(4096), vp(4096), vp(4096), 1, 1, 64, 0,
                                    16, vp(4096), vp(0))
    assert st == ttt.TTT_ERR_ARG  # W_anchor and W_run alias
    st = lib.ttt_linear_decode_step(vp(4096), vp(4096), vp(4096), 1, vp(4096), vp(4096), vp(8192), 1, 1, 64, -1,
                                    16, vp(4096), vp(0))
    assert st == ttt.TTT_ERR_ARG
    assert lib.ttt_last_device_status(vp(0), vp(0)) == ttt.TTT_ERR_ARG


def _bwd(lib, **kw):
    a = dict(Q=1 * MB, K=2 * MB, V=3 * MB, dt=0, eta=4 * MB, W0=5 * MB, B=2, H=3, T=40, d=16, b=8, dZ=6 * MB,
             dW=7 * MB, dQ=8 * MB, dK=9 * MB, dV=10 * MB, deta=11 * MB, dW0=12 * MB, ws=16 * MB, wsb=1 << 24, s=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.ttt_linear_bwd(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]), vp(a["W0"]), a["B"],
                              a["H"], a["T"], a["d"], a["b"], vp(a["dZ"]), vp(a["dW"]), vp(a["dQ"]), vp(a["dK"]),
                              vp(a["dV"]), vp(a["deta"]), vp(a["dW0"]), vp(a["ws"]), a["wsb"], vp(a["s"]))


def test_backward_workspace_bytes_with_segments(lib):
    """bf16-sized at d = 64, b = 16 with few units: the sequence is cut into segments that fill the
    SMs (148 without a GPU), which adds per-segment partials and six d x d matrices per segment
    boundary (forward maps and start states, H_s and A_s, end gradients)."""
    B, H, T = 1, 2, 8192
    S = 64                                   # min(8192 / 64, 148 // 2) = 74 -> 128-token segments -> 64
    base = 2 * (T // 16) * 64 * 64 * 4 + 2 * (64 * 64 + 1) * 4
    seg = -(-2 * S * (64 * 64 + 1) * 4 // 256) * 256 + 2 * (S - 1) * 64 * 64 * 4 * 6
    assert ttt.ttt_linear_bwd_workspace_bytes(B, H, T, 64, 16) == 256 + -(-base // 16) * 16 + seg
    # 84 units: one segment each, no extra
    base = 84 * (200 // 16 + 1) * 64 * 64 * 4 + 84 * (64 * 64 + 1) * 4
    assert ttt.ttt_linear_bwd_workspace_bytes(7, 12, 200, 64, 16) == 256 + -(-base // 16) * 16


def test_backward_workspace_bytes(lib):
    """A status block, every chunk-start state and a per-unit partial of dW0 and d eta."""
    assert ttt.ttt_linear_bwd_workspace_bytes(2, 3, 40, 16, 8) == 256 + 6 * 5 * 16 * 16 * 4 + 6 * (16 * 16 + 1) * 4 + 8
    assert ttt.ttt_linear_bwd_workspace_bytes(1, 1, 0, 16, 8) == 256 + 1 * (16 * 16 + 1) * 4 + 12
    assert ttt.ttt_linear_bwd_workspace_bytes(0, 1, 8, 16, 8) == 0
    # chunks longer than 64 tokens add one chunk's E and dE per unit (at most T tokens of them)
    states, part = 6 * 2 * 16 * 16 * 4, 6 * (16 * 16 + 1) * 4
    assert ttt.ttt_linear_bwd_workspace_bytes(2, 3, 130, 16, 100) == 256 + states + part + 6 * 2 * 100 * 16 * 4 + 8
    assert ttt.ttt_linear_bwd_workspace_bytes(2, 3, 70, 16, 128) == 256 + 6 * 16 * 16 * 4 + part + 6 * 2 * 70 * 16 * 4 + 8


@pytest.mark.parametrize("kw,want", [(dict(Q=0), ttt.TTT_ERR_ARG), (dict(dZ=0), ttt.TTT_ERR_ARG),
                                     (dict(deta=0), ttt.TTT_ERR_ARG), (dict(dW0=4100), ttt.TTT_ERR_ARG),
                                     (dict(wsb=4096), ttt.TTT_ERR_ARG), (dict(b=0), ttt.TTT_ERR_ARG),
                                     (dict(dt=5), ttt.TTT_ERR_ARG), (dict(dt=1, d=65), ttt.TTT_ERR_UNSUPPORTED),
                                     (dict(d=65), ttt.TTT_ERR_UNSUPPORTED), (dict(b=65, wsb=4096), ttt.TTT_ERR_ARG)])
def test_backward_rejects_bad_arguments(lib, kw, want):
    assert _bwd(lib, **kw) == want


def test_no_cpu_fallback_without_a_gpu(lib):
    """With valid arguments and no GPU the call fails loudly instead of computing on the host."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the CPU-only failure mode")
    assert _lin(lib) == ttt.TTT_ERR_CUDA


@pytest.mark.parametrize("kw", [dict(Z=1 * MB + 1024), dict(Z=3 * MB - 1024), dict(W=5 * MB), dict(ws=4 * MB),
                                dict(W=6 * MB + 1024), dict(ws=7 * MB)])
def test_linear_refuses_outputs_that_overlap(lib, kw):
    """Z, W_out and the workspace may overlap neither an input nor one another (Q holds 2 KB here)."""
    assert _lin(lib, **kw) == ttt.TTT_ERR_ARG


def test_inputs_may_alias_and_outputs_may_abut(lib):
    """Q = K = V is allowed, and so is Z starting right where Q ends; with no GPU such a call gets past
    every argument check and fails only at the first CUDA call."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; these fake addresses must not reach a kernel")
    assert _lin(lib, K=1 * MB, V=1 * MB) == ttt.TTT_ERR_CUDA
    assert _lin(lib, Z=1 * MB + 2048) == ttt.TTT_ERR_CUDA       # Q is 16 x 64 bf16 = 2048 bytes
    assert _lin(lib, Z=1 * MB + 2032) == ttt.TTT_ERR_ARG        # one 16-byte step into Q


@pytest.mark.parametrize("kw", [dict(dQ=1 * MB), dict(dK=6 * MB + 4096), dict(deta=4 * MB), dict(dW0=7 * MB + 1024),
                                dict(ws=12 * MB - 1024), dict(dV=9 * MB)])
def test_backward_refuses_outputs_that_overlap(lib, kw):
    """Each output moved onto an input (dQ on Q, dK inside dZ, deta on eta, dW0 inside dW_out) or onto
    another output (the 16 MB workspace over dW0, dV on dK)."""
    assert _bwd(lib, **kw) == ttt.TTT_ERR_ARG


def test_decode_refuses_states_that_overlap():
    vp = ctypes.c_void_p
    lib = ttt.load_library()

    def call(q, z, Wa, Wr):
        return lib.ttt_linear_decode_step(vp(q), vp(q), vp(q), 1, vp(4 * MB), vp(Wa), vp(Wr), 1, 2, 64, 0, 16, vp(z),
                                          vp(0))
    assert call(1 * MB, 2 * MB, 5 * MB, 5 * MB + 16 * 1024) == ttt.TTT_ERR_ARG  # W_run inside W_anchor (32 KB)
    assert call(1 * MB, 1 * MB + 128, 5 * MB, 6 * MB) == ttt.TTT_ERR_ARG       # z inside q (256 bytes)
    assert call(1 * MB, 2 * MB, 4 * MB, 6 * MB) == ttt.TTT_ERR_ARG             # W_anchor on eta


def test_variant_workspace_bytes(lib):
    """Status word, the inner forward's workspace, the changed inputs (padded to 64 features) and
    W0'; Q', Z' and W_out' only where rows are padded. Shapes without the tensor-core path need the
    status word alone; LN and momentum have no workspace call."""
    bf, f32 = ttt.TTT_BF16, ttt.TTT_F32
    seq = 6 * 40 * 64 * 2
    padded = 256 + 256 + 4 * seq + 3 * 64 * 64 * 4 + 6 * 64 * 64 * 4 + 256
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_BIAS, bf, 2, 3, 40, 16, 16) == padded
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, bf, 2, 3, 40, 32, 16) == padded
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, bf, 2, 3, 40, 64, 16) == \
        256 + 256 + 2 * seq + 3 * 64 * 64 * 4 + 256
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_BIAS, bf, 2, 3, 40, 64, 16) == 256   # no room for 1
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_BIAS, f32, 2, 3, 40, 16, 16) == 256
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, bf, 2, 3, 40, 64, 5) == 256
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_LN, bf, 2, 3, 40, 64, 16) == 256
    assert ttt.ttt_linear_variant_workspace_bytes(7, bf, 2, 3, 40, 64, 16) == 0
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_MOMENTUM, bf, 2, 3, 40, 64, 16) == 256
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_MOMENTUM, f32, 2, 3, 40, 16, 5) == 256
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_MOMENTUM, bf, 2, 3, 40, 64, 0) == 0
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_BIAS, bf, 0, 3, 40, 16, 16) == 0
    # the long-context shape: the inner forward's segment scratch is part of it
    inner = ttt.ttt_workspace_bytes(1, 32, 131072, 64, 16)
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, bf, 1, 32, 131072, 64, 16) == \
        256 + -(-inner // 256) * 256 + 2 * 32 * 131072 * 64 * 2 + 32 * 64 * 64 * 4 + 256


def _var_ex(lib, name, **kw):
    a = dict(Q=1 * MB, K=2 * MB, V=3 * MB, dt=1, eta=4 * MB, W0=5 * MB, beta0=6 * MB, gb=7 * MB, B=2, H=3, T=40,
             d=16, b=16,
             Z=8 * MB, W=9 * MB, beta=10 * MB, ws=16 * MB, wsb=1 << 24, s=0)
    a.update(kw)
    vp = ctypes.c_void_p
    if name == "bias":
        return lib.ttt_linear_bias_fwd_ex(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]), vp(a["W0"]),
                                          vp(a["beta0"]), a["B"], a["H"], a["T"], a["d"], a["b"], vp(a["Z"]),
                                          vp(a["W"]), vp(a["beta"]), vp(a["ws"]), a["wsb"], vp(a["s"]))
    if name == "ln":
        o = ttt.ttt_options()
        o.force_path = a.get("fp", 0)
        return lib.ttt_linear_ln_fwd_ex(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]), vp(a["W0"]),
                                        vp(a["beta0"]), vp(a["gb"]), a["B"], a["H"], a["T"], a["d"], a["b"], vp(a["Z"]),
                                        vp(a["W"]), vp(a["ws"]), a["wsb"], vp(a["s"]), ctypes.byref(o))
    if name == "momentum":
        o = ttt.ttt_options()
        o.force_path = a.get("fp", 0)
        return lib.ttt_linear_momentum_fwd_ex(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]),
                                              vp(a["beta0"]), vp(a["W0"]), a["B"], a["H"], a["T"], a["d"], a["b"],
                                              vp(a["Z"]), vp(a["W"]), vp(a["beta"]), vp(a["ws"]), a["wsb"], vp(a["s"]),
                                              ctypes.byref(o))
    return lib.ttt_linear_token_eta_fwd_ex(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]), vp(a["W0"]),
                                           a["B"], a["H"], a["T"], a["d"], a["b"], vp(a["Z"]), vp(a["W"]), vp(a["ws"]),
                                           a["wsb"], vp(a["s"]))


@pytest.mark.parametrize("kw,want", [(dict(fp=3), ttt.TTT_ERR_UNSUPPORTED), (dict(fp=2, d=32), ttt.TTT_ERR_UNSUPPORTED),
                                     (dict(fp=2, b=24), ttt.TTT_ERR_UNSUPPORTED), (dict(fp=2, dt=0), ttt.TTT_ERR_UNSUPPORTED),
                                     (dict(fp=2, T=0), ttt.TTT_ERR_UNSUPPORTED), (dict(fp=5), ttt.TTT_ERR_ARG),
                                     (dict(beta0=0), ttt.TTT_ERR_ARG), (dict(beta=9 * MB + 4096), ttt.TTT_ERR_ARG),
                                     (dict(beta=4 * MB), ttt.TTT_ERR_ARG)])
def test_momentum_fast_call_paths_and_arguments(lib, kw, want):
    """ttt_linear_momentum_fwd_ex: no segment-parallel form; the tensor kernel, when forced, only for
    bf16, d = 64, b a multiple of 16 and T > 0; a bad path, a null beta, M_out over W_out or over an input:
    refused before anything runs (M_out is the `beta` slot of the shared argument set)."""
    base = dict(d=64, W=9 * MB, beta=9 * MB + 64 * 64 * 4 * 6)
    base.update(kw)
    assert _var_ex(lib, "momentum", **base) == want


@pytest.mark.parametrize("kw,want", [(dict(fp=3), ttt.TTT_ERR_UNSUPPORTED), (dict(fp=2, d=32), ttt.TTT_ERR_UNSUPPORTED),
                                     (dict(fp=2, b=24), ttt.TTT_ERR_UNSUPPORTED), (dict(fp=2, dt=0), ttt.TTT_ERR_UNSUPPORTED),
                                     (dict(fp=2, T=0), ttt.TTT_ERR_UNSUPPORTED), (dict(fp=-1), ttt.TTT_ERR_ARG),
                                     (dict(gb=0), ttt.TTT_ERR_ARG), (dict(W=7 * MB + 256), ttt.TTT_ERR_ARG)])
def test_ln_fast_call_paths_and_arguments(lib, kw, want):
    """ttt_linear_ln_fwd_ex: no segment-parallel form; the tensor kernel, when forced, only for bf16,
    d = 64, b a multiple of 16 and T > 0; a bad path, a null beta, W_out over beta: refused before anything runs
    (gamma is the `beta0` slot of the shared argument set, beta the `gb` slot)."""
    base = dict(d=64, W=9 * MB)
    base.update(kw)
    assert _var_ex(lib, "ln", **base) == want


@pytest.mark.parametrize("name", ["bias", "token_eta", "momentum", "ln"])
@pytest.mark.parametrize("kw,want", [(dict(ws=0), ttt.TTT_ERR_ARG), (dict(ws=16 * MB + 8), ttt.TTT_ERR_ARG),
                                     (dict(wsb=4096), ttt.TTT_ERR_ARG), (dict(Q=0), ttt.TTT_ERR_ARG),
                                     (dict(ws=2 * MB), ttt.TTT_ERR_ARG), (dict(Z=16 * MB + 4096), ttt.TTT_ERR_ARG),
                                     (dict(d=65), ttt.TTT_ERR_UNSUPPORTED), (dict(dt=7), ttt.TTT_ERR_ARG),
                                     (dict(b=0), ttt.TTT_ERR_ARG)])
def test_variant_fast_calls_reject_bad_arguments(lib, name, kw, want):
    """No workspace, a misaligned or too small one, a null input, the workspace over an input or an
    output inside the workspace, d > 64, a bad dtype or chunk size: refused before anything runs."""
    if name in ("momentum", "ln") and kw == dict(wsb=4096):
        kw = dict(wsb=128)  # its workspace is the 256-byte status word alone
    assert _var_ex(lib, name, **kw) == want


def test_mlp_backward_workspace_bytes(lib):
    """A status block, then per unit: every chunk-start (W1, W2), four d x 4d gradient buffers,
    one chunk's matrices (8 of b x d, 11 of b x 4d, 3 of b x b, b capped at T); then per-unit
    partials of dW1, dW2, d eta."""
    d, m, T, b, units = 16, 64, 40, 16, 6
    per = 3 * 2 * d * m + 4 * d * m + 8 * b * d + 11 * b * m + 3 * b * b
    raw = 4 * (units * per + units * (2 * d * m + 1))
    assert ttt.ttt_mlp_bwd_workspace_bytes(2, 3, T, d, b) == 256 + -(-raw // 16) * 16
    per = 1 * 2 * d * m + 4 * d * m + 8 * 10 * d + 11 * 10 * m + 3 * 100
    raw = 4 * (units * per + units * (2 * d * m + 1))
    assert ttt.ttt_mlp_bwd_workspace_bytes(2, 3, 10, d, 64) == 256 + -(-raw // 16) * 16
    assert ttt.ttt_mlp_bwd_workspace_bytes(0, 3, 10, d, 64) == 0


def _mlp_bwd(lib, **kw):
    a = dict(Q=1 * MB, K=2 * MB, V=3 * MB, dt=0, eta=4 * MB, W1=5 * MB, W2=6 * MB, B=2, H=3, T=40, d=16, b=8,
             dZ=7 * MB, dW1o=8 * MB, dW2o=9 * MB, dQ=10 * MB, dK=11 * MB, dV=12 * MB, deta=13 * MB, dW1=14 * MB,
             dW2=15 * MB, ws=32 * MB, wsb=1 << 24, s=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.ttt_mlp_bwd(vp(a["Q"]), vp(a["K"]), vp(a["V"]), a["dt"], vp(a["eta"]), vp(a["W1"]), vp(a["W2"]),
                           a["B"], a["H"], a["T"], a["d"], a["b"], vp(a["dZ"]), vp(a["dW1o"]), vp(a["dW2o"]),
                           vp(a["dQ"]), vp(a["dK"]), vp(a["dV"]), vp(a["deta"]), vp(a["dW1"]), vp(a["dW2"]),
                           vp(a["ws"]), a["wsb"], vp(a["s"]))


@pytest.mark.parametrize("kw,want", [(dict(Q=0), ttt.TTT_ERR_ARG), (dict(dW2o=0), ttt.TTT_ERR_ARG),
                                     (dict(ws=0), ttt.TTT_ERR_ARG), (dict(wsb=4096), ttt.TTT_ERR_ARG),
                                     (dict(b=0), ttt.TTT_ERR_ARG), (dict(dt=3), ttt.TTT_ERR_ARG),
                                     (dict(d=65), ttt.TTT_ERR_UNSUPPORTED), (dict(dQ=1 * MB), ttt.TTT_ERR_ARG),
                                     (dict(dW1=5 * MB), ttt.TTT_ERR_ARG), (dict(ws=9 * MB), ttt.TTT_ERR_ARG),
                                     (dict(dW2=14 * MB + 1024), ttt.TTT_ERR_ARG), (dict(dK=2 * MB + 8), ttt.TTT_ERR_ARG)])
def test_mlp_backward_rejects_bad_arguments(lib, kw, want):
    """Null pointers, no or a short workspace, bad sizes or dtype, d > 64, an output on an input
    (dQ on Q, dW1 on W1_0, the workspace over dW2_out), outputs that overlap (dW2 inside dW1), a
    misaligned output: refused before anything runs."""
    assert _mlp_bwd(lib, **kw) == want
