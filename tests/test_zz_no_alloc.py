"""ttt_mlp_fwd_noalloc: the TTT-MLP entry point for callers that cannot
allocate device memory (code inside a region that must not synchronise the
device, under a memory pool that hands out only its own tensors, or a plain C
host that owns only its inputs and outputs). It takes no workspace and uses
the library's fixed scratch array instead.

Called through the C ABI on both of its kernels, two calls in a row with
different inputs each (the shared array keeps the last call's contents, which
must not carry over):
  - the tensor-core kernel (bf16, d = 64, b % 16 == 0), which uses only the
    array's status word, against ttt_mlp_fwd (which gets a workspace from the
    caller) and against the oracle;
  - the fp32 SIMT kernel, which writes and reads the array's per-unit snapshot
    region, against the oracle at the 1e-4 bar, and with bf16 operands and
    b % 16 != 0 at the bf16 bar.
The array's status word reads TTT_OK after each call.

Kept in a file pytest collects after the parity tests, so that a run stopping
at the first failure has run them before this one."""
import ctypes

import pytest
import torch

import synth
import test_sequence_layers_06_b300 as ttt
from ttt_testlib import oracle_mlp, rel_err, rel_l2, to64, tolerance, torch_inputs

pytestmark = pytest.mark.gpu


def _outputs(w):
    Z = torch.full((w.B, w.H, w.T, w.d), float("nan"), device="cuda",
                   dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32)
    W1o = torch.full((w.B, w.H, w.d, 4 * w.d), float("nan"), device="cuda")
    W2o = torch.full((w.B, w.H, 4 * w.d, w.d), float("nan"), device="cuda")
    return Z, W1o, W2o


def _noalloc(lib, t, w, Z, W1o, W2o):
    vp = ctypes.c_void_p
    st = lib.ttt_mlp_fwd_noalloc(vp(t["Q"].data_ptr()), vp(t["K"].data_ptr()), vp(t["V"].data_ptr()),
                                 ttt.TTT_BF16 if w.dtype == "bf16" else ttt.TTT_F32, vp(t["eta"].data_ptr()),
                                 vp(t["W1"].data_ptr()), vp(t["W2"].data_ptr()), w.B, w.H, w.T, w.d, w.b,
                                 vp(Z.data_ptr()), vp(W1o.data_ptr()), vp(W2o.data_ptr()),
                                 vp(torch.cuda.current_stream().cuda_stream))
    return st


def _status(lib):
    return lib.ttt_mlp_noalloc_last_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_tensor_kernel_matches_workspace_entry_point_and_oracle_twice():
    lib = ttt.load_library()
    for seed, T in ((11, 80), (12, 45)):
        w = synth.WORKLOADS["mlp_125m"].with_(B=2, H=3, T=T, seed=seed)
        inp = synth.make_inputs(w)
        t = torch_inputs(inp)
        Zr, W1r, W2r = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], w.b)
        Z, W1o, W2o = _outputs(w)
        assert _noalloc(lib, t, w, Z, W1o, W2o) == ttt.TTT_OK
        assert _status(lib) == ttt.TTT_OK
        torch.cuda.synchronize()
        Zo, W1s, W2s = oracle_mlp(inp, w.b)
        for name, x, r, s in (("Z", Z, Zr, Zo), ("W1", W1o, W1r, W1s), ("W2", W2o, W2r, W2s)):
            assert bool(torch.isfinite(x.float()).all())
            assert rel_l2(to64(x), to64(r)) <= tolerance(w)
            assert rel_err(f"noalloc tensor {name}", to64(x), s, tolerance(w)) <= tolerance(w)


@pytest.mark.parametrize("dtype,b,bar", [("f32", 16, 1e-4), ("bf16", 5, 2e-2)])
def test_noalloc_simt_kernel_uses_the_snapshot_region_twice(dtype, b, bar):
    """fp32 operands (or b % 16 != 0) run the SIMT kernel, which keeps each unit's
    chunk-start W1, W2 in the array's snapshot region: two calls in a row with
    different inputs and sizes, each against the oracle."""
    lib = ttt.load_library()
    for seed, (B, H, T) in ((21, (2, 3, 40)), (22, (3, 2, 29))):
        w = synth.WORKLOADS["mlp_125m"].with_(B=B, H=H, T=T, dtype=dtype, b=b, seed=seed)
        inp = synth.make_inputs(w)
        t = torch_inputs(inp)
        Z, W1o, W2o = _outputs(w)
        assert _noalloc(lib, t, w, Z, W1o, W2o) == ttt.TTT_OK
        assert _status(lib) == ttt.TTT_OK
        torch.cuda.synchronize()
        Zo, W1s, W2s = oracle_mlp(inp, b)
        for name, x, r in (("Z", Z, Zo), ("W1", W1o, W1s), ("W2", W2o, W2s)):
            assert rel_err(f"noalloc simt {dtype} {name}", to64(x), r, bar) <= bar


def test_noalloc_limit_applies_to_the_simt_kernel_only():
    """65 units at d = 64: one more than the snapshot region holds. The SIMT kernel
    (fp32 operands) is refused before anything is enqueued; the tensor-core kernel
    needs no snapshot and serves the same sizes."""
    lib = ttt.load_library()
    w = synth.WORKLOADS["mlp_125m"].with_(B=5, H=13, T=16, dtype="f32")
    t = torch_inputs(synth.make_inputs(w, want_exact=False))
    assert _noalloc(lib, t, w, *_outputs(w)) == ttt.TTT_ERR_UNSUPPORTED
    w = w.with_(dtype="bf16")
    t = torch_inputs(synth.make_inputs(w, want_exact=False))
    Z, W1o, W2o = _outputs(w)
    assert _noalloc(lib, t, w, Z, W1o, W2o) == ttt.TTT_OK
    assert _status(lib) == ttt.TTT_OK
    Zr, W1r, W2r = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], w.b)
    torch.cuda.synchronize()
    for x, r in ((Z, Zr), (W1o, W1r), (W2o, W2r)):
        assert rel_l2(to64(x), to64(r)) <= tolerance(w)
