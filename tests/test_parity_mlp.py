"""TTT-MLP on the GPU (through the C ABI) against the fp64 oracle: the
tensor-core kernel (bf16, d = 64, b % 16 == 0) and the fp32 SIMT kernel."""
import numpy as np
import pytest
import torch

import synth
import test_sequence_layers_06_b300 as ttt
from ttt_testlib import oracle_mlp, rel_err, rel_l2, to64, tolerance, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def run_mlp(inp, b):
    t = torch_inputs(inp)
    Z, W1, W2 = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], b)
    torch.cuda.synchronize()
    return to64(Z), to64(W1), to64(W2)


@pytest.mark.parametrize("T,b,dtype,d", [(64, 16, "bf16", 64), (37, 16, "bf16", 64), (20, 5, "f32", 16),
                                         (48, 16, "f32", 64), (1, 16, "bf16", 32)])
def test_mlp_small(T, b, dtype, d):
    w = W["mlp_125m"].with_(B=2, H=2, T=T, d=d, hidden=4 * d, dtype=dtype, seed=300 + T)
    inp = synth.make_inputs(w)
    Z, W1, W2 = run_mlp(inp, b)
    Zr, W1r, W2r = oracle_mlp(inp, b)
    tol = 1e-4 if dtype == "f32" else tolerance(w)
    for name, x, r in (("Z", Z, Zr), ("W1", W1, W1r), ("W2", W2, W2r)):
        assert rel_err(name, x, r, tol) <= tol, rel_l2(x, r)


@pytest.mark.parametrize("T,b", [(96, 32), (80, 48), (130, 64)])
def test_mlp_tensor_path_chunks_of_several_tiles(T, b):
    """Chunks of 2-4 tiles: gradients at the chunk-start weights, read-out with
    the running ones (the tensor-core kernel keeps both bf16 copies)."""
    w = W["mlp_125m"].with_(B=1, H=3, T=T, seed=400 + T + b)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    Z, W1, W2 = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], b,
                                options={"force_path": ttt.PATH_TENSOR})
    torch.cuda.synchronize()
    Zr, W1r, W2r = oracle_mlp(inp, b)
    for name, x, r in (("Z", Z, Zr), ("W1", W1, W1r), ("W2", W2, W2r)):
        assert rel_err(name, to64(x), r, tolerance(w)) <= tolerance(w), rel_l2(to64(x), r)


def test_mlp_simt_path_bf16_agrees_with_tensor_path():
    w = W["mlp_125m"].with_(B=2, H=2, T=64, seed=77)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    outs = [ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], 16, options={"force_path": fp})
            for fp in (ttt.PATH_SIMT, ttt.PATH_TENSOR)]
    torch.cuda.synchronize()
    Zr, W1r, W2r = oracle_mlp(inp, 16)
    for (Z, W1, W2) in outs:
        for x, r in ((Z, Zr), (W1, W1r), (W2, W2r)):
            assert rel_l2(to64(x), r) <= tolerance(w)
    assert rel_l2(to64(outs[0][0]), to64(outs[1][0])) < 2e-2


def test_mlp_full_size_sampled():
    """B4 H12 T8192 d64 hidden 256: GPU over all units, oracle on two sampled ones."""
    w = W["mlp_125m"]
    full = synth.make_inputs(w, want_exact=False)
    t = torch_inputs(full)
    Z, W1, W2 = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], w.b)
    torch.cuda.synchronize()
    units = [(0, 0), (3, 11)]
    sub = synth.make_inputs(w, units=units)
    Zr, W1r, W2r = oracle_mlp(sub, w.b)
    for k, (n, h) in enumerate(units):
        assert rel_err(f"Z unit {n},{h}", to64(Z[n, h]), Zr[0, k], tolerance(w)) <= tolerance(w)
        assert rel_err(f"W1 unit {n},{h}", to64(W1[n, h]), W1r[0, k], tolerance(w)) <= tolerance(w)
        assert rel_err(f"W2 unit {n},{h}", to64(W2[n, h]), W2r[0, k], tolerance(w)) <= tolerance(w)
    assert bool(torch.isfinite(Z.float()).all())


@pytest.mark.parametrize("T", [0, 1, 16, 37, 64, 200])
def test_mlp_b16_one_and_two_ctas_per_unit(T):
    """b = 16: the two-CTA kernel (each CTA of a cluster holds half of the hidden units; the partial
    sums of G and Z cross through distributed shared memory; the automatic choice) and the one-CTA
    kernel, against the oracle: empty, shorter than a tile, ragged and several tiles."""
    w = W["mlp_125m"].with_(B=2, H=3, T=T, seed=500 + T)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    Zr, W1r, W2r = oracle_mlp(inp, 16)
    for fp in (0, ttt.PATH_TENSOR, 3):
        Z, W1, W2 = ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], 16,
                                    options={"force_path": fp})
        torch.cuda.synchronize()
        for name, x, r in (("Z", Z, Zr), ("W1", W1, W1r), ("W2", W2, W2r)):
            if x.numel() == 0:
                continue
            assert rel_err(f"path {fp} {name}", to64(x), r, tolerance(w)) <= tolerance(w), (fp, name)


def test_mlp_two_ctas_refused_where_they_do_not_apply():
    w = W["mlp_125m"].with_(B=1, H=1, T=64, seed=510)
    t = torch_inputs(synth.make_inputs(w))
    with pytest.raises(ttt.TTTError):
        ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], 32, options={"force_path": 3})


@pytest.mark.parametrize("stall,path,b", [(1, 3, 16), (2, 3, 16), (1, ttt.PATH_TENSOR, 16), (1, ttt.PATH_TENSOR, 32)])
def test_mlp_bounded_waits_report_timeout_and_context_survives(stall, path, b):
    """A wait that nothing will end runs out after 1 ms: the loads never start (1), or the second
    CTA of each cluster withholds its G partials (2). The kernel returns, the status says
    TTT_ERR_TIMEOUT, reading clears it, and the next call on the same context matches the oracle."""
    w = W["mlp_125m"].with_(B=1, H=2, T=64, seed=520 + stall)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    args = (t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], b)
    ws = torch.zeros(max(ttt.ttt_workspace_bytes(w.B, w.H, w.T, w.d, b, ttt.TTT_VARIANT_MLP), 256),
                     dtype=torch.uint8, device="cuda")
    ttt.ttt_mlp_fwd(*args, workspace=ws,
                    options={"inject_stall": stall, "wait_timeout_ns": 1_000_000, "force_path": path})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_ERR_TIMEOUT
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    Z, W1, W2 = ttt.ttt_mlp_fwd(*args, workspace=ws, options={"force_path": path})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    Zr, W1r, W2r = oracle_mlp(inp, b)
    for name, x, r in (("Z", Z, Zr), ("W1", W1, W1r), ("W2", W2, W2r)):
        assert rel_err(f"after timeout {name}", to64(x), r, tolerance(w)) <= tolerance(w), name
