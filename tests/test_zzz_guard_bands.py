"""Guard bands around every output, and non-finite inputs (GPU).

Out-of-bounds writes are looked for directly, without a memory checker: every
output and workspace of a call is a view into a larger buffer
whose margins hold a known pattern, and the margins must be bit-identical after
the call. A write past either end of an output lands in memory the test owns,
so a bad kernel shows up here as a failed comparison rather than a fault.
Ragged sequence lengths (T not a multiple of 16 or of b) exercise the tails.

A NaN in one unit's inputs must stay in that unit: the call finishes, its
status is OK, and every other (batch row, head) unit is unchanged.

Kept in a file pytest collects last, so that a run stopping at the first
failure has run every other test before this one.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import test_sequence_layers_06_b300 as ttt
from ttt_testlib import oracle_linear, oracle_mlp, rel_l2, to64, tolerance, torch_inputs

pytestmark = pytest.mark.gpu

MARGIN_BYTES = 256  # on each side; keeps every view 16-byte aligned


class Guarded:
    """A tensor of `shape` inside a buffer with MARGIN_BYTES of pattern on each side."""

    def __init__(self, shape, dtype, fill):
        es = torch.empty((), dtype=dtype).element_size()
        self.m = MARGIN_BYTES // es
        self.n = math.prod(shape)
        self.buf = torch.full((self.n + 2 * self.m,), fill, dtype=dtype, device="cuda")
        self.t = self.buf[self.m:self.m + self.n].view(shape)
        self.before = self.buf.clone()

    def margins_intact(self) -> bool:
        torch.cuda.synchronize()
        return torch.equal(self.buf[:self.m], self.before[:self.m]) and \
            torch.equal(self.buf[self.m + self.n:], self.before[self.m + self.n:])


def guarded_workspace(nbytes):
    return Guarded((max(nbytes, 256),), torch.uint8, 0xA5)


@pytest.mark.parametrize("T,b,opts", [(1000, 16, {"force_path": ttt.PATH_SEGMENTED, "seg_len": 256}),
                                      (1300, 32, {"force_path": ttt.PATH_SEGMENTED, "seg_len": 64}),
                                      (72, 32, {"force_path": ttt.PATH_TENSOR}),
                                      (45, 16, {"force_path": ttt.PATH_SIMT})])
def test_linear_forward_writes_inside_its_outputs(T, b, opts):
    w = synth.WORKLOADS["linear_small"].with_(B=1, H=3, T=T, b=b, seed=900 + T)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    Z = Guarded((w.B, w.H, T, w.d), torch.bfloat16, -3.0)
    Wo = Guarded((w.B, w.H, w.d, w.d), torch.float32, -5.0)
    ws = guarded_workspace(ttt.ttt_workspace_bytes(w.B, w.H, T, w.d, b, options=opts))
    ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], b, Z=Z.t, W_out=Wo.t, workspace=ws.t,
                       options=opts)
    assert ttt.ttt_last_device_status(ws.t) == ttt.TTT_OK
    assert Z.margins_intact() and Wo.margins_intact() and ws.margins_intact()
    Zr, Wr = oracle_linear(inp, b)
    assert rel_l2(to64(Z.t), Zr) <= tolerance(w) and rel_l2(to64(Wo.t), Wr) <= tolerance(w)


def test_linear_fp32_forward_writes_inside_its_outputs():
    w = synth.WORKLOADS["linear_tiny_f32"].with_(B=2, H=2, T=37, d=16, b=5)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    Z = Guarded((w.B, w.H, w.T, w.d), torch.float32, -3.0)
    Wo = Guarded((w.B, w.H, w.d, w.d), torch.float32, -5.0)
    ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], w.b, Z=Z.t, W_out=Wo.t)
    assert Z.margins_intact() and Wo.margins_intact()
    Zr, Wr = oracle_linear(inp, w.b)
    assert rel_l2(to64(Z.t), Zr) <= 1e-4 and rel_l2(to64(Wo.t), Wr) <= 1e-4


@pytest.mark.parametrize("T,opts", [(40, None), (37, {"force_path": ttt.PATH_SIMT}), (37, {"force_path": ttt.PATH_TENSOR})])
def test_mlp_forward_writes_inside_its_outputs(T, opts):
    w = synth.WORKLOADS["mlp_125m"].with_(B=1, H=2, T=T, seed=910 + T)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    m = 4 * w.d
    Z = Guarded((w.B, w.H, T, w.d), torch.bfloat16, -3.0)
    A1 = Guarded((w.B, w.H, w.d, m), torch.float32, -5.0)
    A2 = Guarded((w.B, w.H, m, w.d), torch.float32, -7.0)
    ws = guarded_workspace(ttt.ttt_workspace_bytes(w.B, w.H, T, w.d, w.b, ttt.TTT_VARIANT_MLP))
    ttt.ttt_mlp_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W1"], t["W2"], w.b, Z=Z.t, W1_out=A1.t, W2_out=A2.t,
                    workspace=ws.t, options=opts)
    assert ttt.ttt_last_device_status(ws.t) == ttt.TTT_OK
    assert Z.margins_intact() and A1.margins_intact() and A2.margins_intact() and ws.margins_intact()
    Zr, W1r, W2r = oracle_mlp(inp, w.b)
    assert rel_l2(to64(Z.t), Zr) <= tolerance(w) and rel_l2(to64(A1.t), W1r) <= tolerance(w)


def test_momentum_tensor_kernel_writes_inside_its_outputs():
    """The tensor-core momentum kernel (bf16, d = 64, b = 16), a ragged last chunk: Z, W_out, M_out
    and the workspace keep their margins, and the results match the oracle."""
    from oracle.variants import momentum_primal
    w = synth.WORKLOADS["linear_small"].with_(B=1, H=3, T=45, seed=915)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    alpha = torch.full((w.H,), 0.1, device="cuda")
    beta = torch.tensor([0.5, 0.8, 0.0], device="cuda")
    Z = Guarded((w.B, w.H, w.T, w.d), torch.bfloat16, -3.0)
    Wo = Guarded((w.B, w.H, w.d, w.d), torch.float32, -5.0)
    Mo = Guarded((w.B, w.H, w.d, w.d), torch.float32, -7.0)
    ws = guarded_workspace(256)
    o = ttt.ttt_options()
    o.force_path = ttt.PATH_TENSOR
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    st = ttt.load_library().ttt_linear_momentum_fwd_ex(
        p(t["Q"]), p(t["K"]), p(t["V"]), ttt.TTT_BF16, p(alpha), p(beta), p(t["W0"]), w.B, w.H, w.T, w.d, 16, p(Z.t),
        p(Wo.t), p(Mo.t), p(ws.t), 256, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(o))
    assert st == ttt.TTT_OK
    assert ttt.ttt_last_device_status(ws.t) == ttt.TTT_OK
    assert Z.margins_intact() and Wo.margins_intact() and Mo.margins_intact() and ws.margins_intact()
    Zr, Wr, Mr = momentum_primal(inp.q64, inp.k64, inp.v64, alpha.cpu().numpy(), beta.cpu().numpy(), inp.W0_64, 16)
    for x, r in ((Z.t, Zr), (Wo.t, Wr), (Mo.t, Mr)):
        assert rel_l2(to64(x), r) <= tolerance(w)


def test_ln_tensor_kernel_writes_inside_its_outputs():
    """The tensor-core LN + residual kernel (bf16, d = 64, b = 16), a ragged last chunk: Z, W_out and
    the workspace keep their margins, and the results match the oracle."""
    from oracle.variants import ln_residual_primal
    w = synth.WORKLOADS["linear_small"].with_(B=1, H=3, T=45, seed=916)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    g = np.random.default_rng(9)
    gamma = torch.from_numpy((1.0 + 0.2 * g.standard_normal((w.H, 64))).astype(np.float32)).cuda()
    beta = torch.from_numpy((0.1 * g.standard_normal((w.H, 64))).astype(np.float32)).cuda()
    Z = Guarded((w.B, w.H, w.T, w.d), torch.bfloat16, -3.0)
    Wo = Guarded((w.B, w.H, w.d, w.d), torch.float32, -5.0)
    ws = guarded_workspace(256)
    o = ttt.ttt_options()
    o.force_path = ttt.PATH_TENSOR
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    st = ttt.load_library().ttt_linear_ln_fwd_ex(
        p(t["Q"]), p(t["K"]), p(t["V"]), ttt.TTT_BF16, p(t["eta"]), p(t["W0"]), p(gamma), p(beta), w.B, w.H, w.T, w.d,
        16, p(Z.t), p(Wo.t), p(ws.t), 256, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(o))
    assert st == ttt.TTT_OK
    assert ttt.ttt_last_device_status(ws.t) == ttt.TTT_OK
    assert Z.margins_intact() and Wo.margins_intact() and ws.margins_intact()
    Zr, Wr = ln_residual_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, gamma.cpu().numpy(),
                                beta.cpu().numpy(), 16)
    assert rel_l2(to64(Z.t), Zr) <= tolerance(w) and rel_l2(to64(Wo.t), Wr) <= tolerance(w)


def test_decode_writes_inside_its_outputs():
    g = np.random.default_rng(7)
    B, H, d = 2, 3, 64
    q, k, v = (torch.from_numpy(g.standard_normal((B, H, d)).astype(np.float32)).cuda() for _ in range(3))
    eta = torch.full((H,), 0.1, device="cuda")
    Wa = Guarded((B, H, d, d), torch.float32, 0.0)
    Wr = Guarded((B, H, d, d), torch.float32, 0.0)
    z = Guarded((B, H, d), torch.float32, -3.0)
    ttt.ttt_linear_decode_step(q, k, v, eta, Wa.t, Wr.t, 15, 16, z=z.t)
    assert z.margins_intact() and Wa.margins_intact() and Wr.margins_intact()
    zr, _, Wr2 = oracle.linear_decode_step(q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy(), eta.cpu().numpy(),
                                           np.zeros((B, H, d, d)), np.zeros((B, H, d, d)), 15, 16)
    assert rel_l2(to64(z.t), zr) <= 1e-5 and rel_l2(to64(Wr.t), Wr2) <= 1e-6


def test_backward_writes_inside_its_outputs():
    w = synth.WORKLOADS["linear_tiny_f32"].with_(B=2, H=2, T=29, d=16, b=8, eta=("const", 0.3), w_std=0.02)
    x = synth.make_inputs(w)
    t = torch_inputs(x)
    g = np.random.default_rng(5)
    dZ = torch.from_numpy(g.standard_normal((w.B, w.H, w.T, w.d)).astype(np.float32)).cuda()
    dWo = torch.from_numpy(g.standard_normal((w.B, w.H, w.d, w.d)).astype(np.float32)).cuda()
    outs = [Guarded((w.B, w.H, w.T, w.d), torch.float32, -3.0) for _ in range(3)]
    deta = Guarded((w.H,), torch.float32, -5.0)
    dW0 = Guarded((w.H, w.d, w.d), torch.float32, -7.0)
    need = ttt.ttt_linear_bwd_workspace_bytes(w.B, w.H, w.T, w.d, w.b)
    ws = guarded_workspace(need)
    vp = lambda x: ctypes.c_void_p(x.data_ptr())
    st = ttt.load_library().ttt_linear_bwd(vp(t["Q"]), vp(t["K"]), vp(t["V"]), ttt.TTT_F32, vp(t["eta"]),
                                           vp(t["W0"]), w.B, w.H, w.T, w.d, w.b, vp(dZ), vp(dWo), vp(outs[0].t),
                                           vp(outs[1].t), vp(outs[2].t), vp(deta.t), vp(dW0.t), vp(ws.t), need,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ttt.TTT_OK
    assert all(o.margins_intact() for o in outs) and deta.margins_intact() and dW0.margins_intact()
    assert ws.margins_intact()
    from oracle.backward import linear_backward
    want = linear_backward(x.q, x.k, x.v, x.eta, x.W0, w.b, dZ.cpu().numpy(), dWo.cpu().numpy())
    for got, r in zip([o.t for o in outs] + [deta.t, dW0.t], want):
        assert rel_l2(to64(got), r) <= 1e-4


def test_long_chunk_backward_and_mlp_backward_write_inside_their_outputs():
    """The backward for chunks longer than 64 tokens (b = 100) and the TTT-MLP backward, each with
    every output and its workspace inside guard bands."""
    vp = lambda x: ctypes.c_void_p(x.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    lib = ttt.load_library()
    g = np.random.default_rng(6)
    # TTT-Linear, b = 100 over T = 230 (two full chunks and a ragged one)
    w = synth.WORKLOADS["linear_tiny_f32"].with_(B=2, H=2, T=230, d=16, b=100, eta=("const", 0.05), w_std=0.02)
    t = torch_inputs(synth.make_inputs(w))
    dZ = torch.from_numpy(g.standard_normal((w.B, w.H, w.T, w.d)).astype(np.float32)).cuda()
    dWo = torch.from_numpy(g.standard_normal((w.B, w.H, w.d, w.d)).astype(np.float32)).cuda()
    outs = [Guarded((w.B, w.H, w.T, w.d), torch.float32, -3.0) for _ in range(3)]
    deta, dW0 = Guarded((w.H,), torch.float32, -5.0), Guarded((w.H, w.d, w.d), torch.float32, -7.0)
    need = ttt.ttt_linear_bwd_workspace_bytes(w.B, w.H, w.T, w.d, w.b)
    ws = guarded_workspace(need)
    st = lib.ttt_linear_bwd(vp(t["Q"]), vp(t["K"]), vp(t["V"]), ttt.TTT_F32, vp(t["eta"]), vp(t["W0"]), w.B, w.H,
                            w.T, w.d, w.b, vp(dZ), vp(dWo), vp(outs[0].t), vp(outs[1].t), vp(outs[2].t), vp(deta.t),
                            vp(dW0.t), vp(ws.t), need, stream)
    assert st == ttt.TTT_OK
    torch.cuda.synchronize()
    assert all(o.margins_intact() for o in outs) and deta.margins_intact() and dW0.margins_intact()
    assert ws.margins_intact()
    # TTT-MLP, d = 16 (hidden 64), b = 5 over T = 23
    w = synth.WORKLOADS["mlp_125m"].with_(B=2, H=2, T=23, d=16, b=5, hidden=64, dtype="f32", w_std=0.3)
    t = torch_inputs(synth.make_inputs(w))
    dZ = torch.from_numpy(g.standard_normal((w.B, w.H, w.T, w.d)).astype(np.float32)).cuda()
    dW1o = torch.from_numpy(g.standard_normal((w.B, w.H, w.d, 64)).astype(np.float32)).cuda()
    dW2o = torch.from_numpy(g.standard_normal((w.B, w.H, 64, w.d)).astype(np.float32)).cuda()
    outs = [Guarded((w.B, w.H, w.T, w.d), torch.float32, -3.0) for _ in range(3)]
    deta = Guarded((w.H,), torch.float32, -5.0)
    dW1, dW2 = Guarded((w.H, w.d, 64), torch.float32, -7.0), Guarded((w.H, 64, w.d), torch.float32, -9.0)
    need = ttt.ttt_mlp_bwd_workspace_bytes(w.B, w.H, w.T, w.d, w.b)
    ws = guarded_workspace(need)
    st = lib.ttt_mlp_bwd(vp(t["Q"]), vp(t["K"]), vp(t["V"]), ttt.TTT_F32, vp(t["eta"]), vp(t["W1"]), vp(t["W2"]),
                         w.B, w.H, w.T, w.d, w.b, vp(dZ), vp(dW1o), vp(dW2o), vp(outs[0].t), vp(outs[1].t),
                         vp(outs[2].t), vp(deta.t), vp(dW1.t), vp(dW2.t), vp(ws.t), need, stream)
    assert st == ttt.TTT_OK
    torch.cuda.synchronize()
    assert all(o.margins_intact() for o in outs) and deta.margins_intact()
    assert dW1.margins_intact() and dW2.margins_intact() and ws.margins_intact()


@pytest.mark.parametrize("opts", [{"force_path": ttt.PATH_SEGMENTED, "seg_len": 256},
                                  {"force_path": ttt.PATH_TENSOR}, {"force_path": ttt.PATH_SIMT}])
def test_nan_stays_in_its_unit(opts):
    """A NaN key in unit (0, 1) at token 300: the call finishes with status OK, that unit's output is
    NaN from token 300 on, its output before the NaN's chunk (tokens 288-303) equals a clean run, and
    the other units equal a clean run bit for bit. (Inside that chunk a product may carry the NaN into
    earlier rows, NaN x 0 being NaN, so those rows are not checked.)"""
    w = synth.WORKLOADS["linear_small"].with_(B=1, H=3, T=600, b=16, seed=920)
    t = torch_inputs(synth.make_inputs(w))
    ws = torch.zeros(ttt.ttt_workspace_bytes(w.B, w.H, w.T, w.d, w.b, options=opts), dtype=torch.uint8,
                     device="cuda")
    Zc, Wc = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], w.b, workspace=ws, options=opts)
    K = t["K"].clone()
    K[0, 1, 300, 5] = float("nan")
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], K, t["V"], t["eta"], t["W0"], w.b, workspace=ws, options=opts)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    for h in (0, 2):
        assert torch.equal(Z[0, h], Zc[0, h]) and torch.equal(Wo[0, h], Wc[0, h])
    assert torch.equal(Z[0, 1, :288], Zc[0, 1, :288])
    assert torch.isnan(Z[0, 1, 300:].float()).all() and torch.isnan(Wo[0, 1]).any()
