"""Backward of TTT-MLP on the GPU (through the C ABI) against the fp64 oracle.

ttt_mlp_bwd returns dQ, dK, dV, d eta, dW1 and dW2 for upstream dZ, dW1_out and
dW2_out; oracle.backward.mlp_backward (pinned by finite differences of the C
primal, autograd and eta = 0 in test_oracle_backward.py) computes the same in
fp64 from the same inputs. Bars: rel-L2 <= 1e-4 per output with fp32 operands,
<= 2e-2 with bf16 operands.
"""
import numpy as np
import pytest
import torch

import synth
import test_sequence_layers_06_b300 as ttt
from oracle.backward import mlp_backward
from ttt_testlib import rel_err, rel_l2, to64, torch_inputs

pytestmark = pytest.mark.gpu

NAMES = ("dQ", "dK", "dV", "deta", "dW1", "dW2")


def run(w, inp, seed, dz_bf16=False):
    g = np.random.default_rng(seed)
    m = 4 * w.d
    dZ = g.standard_normal((w.B, w.H, w.T, w.d)).astype(np.float32)
    if dz_bf16:
        dZ = torch.from_numpy(dZ).to(torch.bfloat16).to(torch.float32).numpy()
    dW1 = (0.5 * g.standard_normal((w.B, w.H, w.d, m))).astype(np.float32)
    dW2 = (0.5 * g.standard_normal((w.B, w.H, m, w.d))).astype(np.float32)
    t = torch_inputs(inp)
    dev = t["Q"].device
    dZt = torch.from_numpy(dZ).to(dev).to(t["Q"].dtype)
    got = ttt.ttt_mlp_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], w.b, dZt,
                          torch.from_numpy(dW1).to(dev), torch.from_numpy(dW2).to(dev))
    torch.cuda.synchronize()
    want = mlp_backward(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W1_64, inp.W2_64, w.b, dZ, dW1, dW2)
    return got, want


@pytest.mark.parametrize("B,H,T,d,b", [(1, 1, 16, 8, 16), (2, 2, 37, 16, 5), (1, 2, 40, 16, 16), (2, 1, 20, 8, 1),
                                       (1, 2, 70, 16, 32), (1, 1, 33, 64, 16), (2, 1, 9, 16, 64)])
def test_mlp_backward_matches_oracle(B, H, T, d, b):
    """fp32 operands: one and many chunks, ragged last chunks, b = 1, a chunk longer than the
    sequence, d = 64 (hidden 256)."""
    w = synth.WORKLOADS["mlp_125m"].with_(B=B, H=H, T=T, d=d, b=b, hidden=4 * d, dtype="f32", w_std=0.3,
                                          eta=("const", 0.2), seed=90 + T + d + b)
    inp = synth.make_inputs(w)
    got, want = run(w, inp, T + b)
    for name, g, r in zip(NAMES, got, want):
        g = to64(g)
        assert np.all(np.isfinite(g)), name
        assert rel_err(f"mlp {name}", g, r, 1e-4) <= 1e-4, (name, rel_l2(g, r))


@pytest.mark.parametrize("B,H,T,d,b", [(1, 2, 64, 64, 16), (2, 1, 50, 32, 16)])
def test_mlp_backward_bf16_matches_oracle(B, H, T, d, b):
    """bf16 operands (fp32 arithmetic; dQ, dK, dV returned in bf16) against the fp64 backward of
    the same bf16 values."""
    w = synth.WORKLOADS["mlp_125m"].with_(B=B, H=H, T=T, d=d, b=b, hidden=4 * d, w_std=0.1,
                                          eta=("uniform", 0.05, 0.3), seed=95 + T + d)
    inp = synth.make_inputs(w)
    got, want = run(w, inp, 3 * T + b, dz_bf16=True)
    assert got[0].dtype == torch.bfloat16
    for name, g, r in zip(NAMES, got, want):
        g = to64(g)
        assert np.all(np.isfinite(g)), name
        assert rel_err(f"mlp bf16 {name}", g, r, 2e-2) <= 2e-2, (name, rel_l2(g, r))


def test_mlp_backward_empty_sequence():
    """T = 0: dW1, dW2 are dW1_out, dW2_out summed over the batch rows and d eta is 0."""
    w = synth.WORKLOADS["mlp_125m"].with_(B=2, H=2, T=0, d=8, b=16, hidden=32, dtype="f32", seed=4)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    dev = t["W1"].device
    g = np.random.default_rng(2)
    dW1 = g.standard_normal((2, 2, 8, 32)).astype(np.float32)
    dW2 = g.standard_normal((2, 2, 32, 8)).astype(np.float32)
    _, _, _, deta, gW1, gW2 = ttt.ttt_mlp_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], 16,
                                               torch.zeros_like(t["Q"]), torch.from_numpy(dW1).to(dev),
                                               torch.from_numpy(dW2).to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(deta.cpu().numpy(), np.zeros(2, np.float32))
    assert np.allclose(gW1.cpu().numpy(), dW1.sum(0), atol=1e-6)
    assert np.allclose(gW2.cpu().numpy(), dW2.sum(0), atol=1e-6)
