"""ttt_mlp_fwd_noalloc: the TTT-MLP entry point for callers that cannot
allocate device memory (it takes no workspace and uses the library's fixed
scratch array instead). Called through the C ABI and compared with
ttt_mlp_fwd, which gets a workspace from the caller, on two calls in a row
with different inputs (the shared array must not carry anything over).

Kept in a file pytest collects after the parity tests, so that a run stopping
at the first failure has run them before this one."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import test_sequence_layers_06_b300 as ttt
from ttt_testlib import rel_l2, to64, tolerance, torch_inputs

pytestmark = pytest.mark.gpu


def _noalloc(lib, t, w, Z, W1o, W2o):
    vp = ctypes.c_void_p
    st = lib.ttt_mlp_fwd_noalloc(vp(t["Q"].data_ptr()), vp(t["K"].data_ptr()), vp(t["V"].data_ptr()),
                                 ttt.TTT_BF16 if w.dtype == "bf16" else ttt.TTT_F32, vp(t["eta"].data_ptr()),
                                 vp(t["W1"].data_ptr()), vp(t["W2"].data_ptr()), w.B, w.H, w.T, w.d, w.b,
                                 vp(Z.data_ptr()), vp(W1o.data_ptr()), vp(W2o.data_ptr()),
                                 vp(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_workspace_entry_point_twice():
    lib = ttt.load_library()
    for seed, T in ((11, 80), (12, 45)):
        w = synth.WORKLOADS["mlp_125m"].with_(B=2, H=3, T=T, seed=seed)
        t = torch_inputs(synth.make_inputs(w, want_exact=False))
        Zr, W1r, W2r = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], w.b)
        Z = torch.full_like(t["Q"], float("nan"))
        W1o = torch.full((w.B, w.H, w.d, 4 * w.d), float("nan"), device="cuda")
        W2o = torch.full((w.B, w.H, 4 * w.d, w.d), float("nan"), device="cuda")
        assert _noalloc(lib, t, w, Z, W1o, W2o) == ttt.TTT_OK
        torch.cuda.synchronize()
        for x, r in ((Z, Zr), (W1o, W1r), (W2o, W2r)):
            assert bool(torch.isfinite(x.float()).all())
            assert rel_l2(to64(x), to64(r)) <= tolerance(w)


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = ttt.load_library()
    w = synth.WORKLOADS["mlp_125m"].with_(B=5, H=13, T=16)  # 65 units at d = 64: one more than fits
    t = torch_inputs(synth.make_inputs(w, want_exact=False))
    Z = torch.empty_like(t["Q"])
    W1o = torch.empty((w.B, w.H, w.d, 4 * w.d), device="cuda")
    W2o = torch.empty((w.B, w.H, 4 * w.d, w.d), device="cuda")
    assert _noalloc(lib, t, w, Z, W1o, W2o) == ttt.TTT_ERR_UNSUPPORTED
