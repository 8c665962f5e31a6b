"""Backward of TTT-Linear on the GPU (through the C ABI) against the fp64 oracle.

ttt_linear_bwd returns dQ, dK, dV, d eta and dW0 for upstream dZ and dW_out;
oracle.backward.linear_backward (pinned by finite differences and autograd in
test_oracle_backward.py) computes the same in fp64 from the same fp32 inputs.
Bar: rel-L2 <= 1e-4 per output (fp32 operands).
"""
import numpy as np
import pytest
import torch

import synth
import test_sequence_layers_06_b300 as ttt
from oracle.backward import linear_backward
from ttt_testlib import rel_err, rel_l2, to64, torch_inputs

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def upstream(w, seed):
    g = np.random.default_rng(seed)
    dZ = g.standard_normal((w.B, w.H, w.T, w.d)).astype(np.float32)
    dW = g.standard_normal((w.B, w.H, w.d, w.d)).astype(np.float32)
    return dZ, dW


@pytest.mark.parametrize("B,H,T,d,b,eta", [(1, 1, 64, 16, 16, ("const", 0.5)), (2, 3, 37, 16, 5, ("uniform", 0.05, 0.5)),
                                           (1, 2, 64, 64, 16, ("const", 0.1)), (2, 2, 50, 32, 64, ("const", 0.1)),
                                           (1, 1, 9, 8, 1, ("const", 0.3)), (2, 1, 130, 64, 64, ("const", 0.05))])
def test_backward_matches_oracle(B, H, T, d, b, eta):
    w = W["linear_tiny_f32"].with_(B=B, H=H, T=T, d=d, b=b, eta=eta, w_std=0.02, seed=40 + T + d + b)
    inp = synth.make_inputs(w)
    dZ, dW = upstream(w, seed=T + b)
    t = torch_inputs(inp)
    dev = t["Q"].device
    got = ttt.ttt_linear_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], b, torch.from_numpy(dZ).to(dev),
                             torch.from_numpy(dW).to(dev))
    torch.cuda.synchronize()
    want = linear_backward(inp.q, inp.k, inp.v, inp.eta, inp.W0, b, dZ, dW)
    for name, g, r in zip(("dQ", "dK", "dV", "deta", "dW0"), got, want):
        g = to64(g)
        assert np.all(np.isfinite(g)), name
        assert rel_err(name, g, r, 1e-4) <= 1e-4, (name, rel_l2(g, r))


def test_backward_empty_sequence():
    """T = 0: no tokens, so dW0 is dW_out summed over the batch rows and d eta is 0."""
    w = W["linear_tiny_f32"].with_(B=2, H=2, T=0, d=16, seed=3)
    inp = synth.make_inputs(w)
    dZ, dW = upstream(w, seed=1)
    t = torch_inputs(inp)
    dev = t["W0"].device
    _, _, _, deta, dW0 = ttt.ttt_linear_bwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16,
                                            torch.from_numpy(dZ).to(dev), torch.from_numpy(dW).to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(deta.cpu().numpy(), np.zeros(2, np.float32))
    assert np.allclose(dW0.cpu().numpy(), dW.sum(0), atol=1e-6)
