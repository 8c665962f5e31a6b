"""Inner-model variants of TTT-Linear on the GPU (through the C ABI) against the
fp64 oracle of oracle/variants.py (pinned in test_oracle_variants.py): a bias in
f, a learning rate per token, a layer norm and a residual inside f, and
momentum gradient descent with chunk-start gradients. Bars: rel-L2 <= 1e-4 with
fp32 operands, <= 2e-2 with bf16 operands (fp32 state and arithmetic)."""
import numpy as np
import pytest
import torch

import synth
import test_sequence_layers_06_b300 as ttt
from oracle.variants import bias_primal, ln_residual_primal, momentum_primal, token_eta_primal
from ttt_testlib import rel_err, to64, tolerance, torch_inputs

pytestmark = pytest.mark.gpu

CASES = [(16, 40, 16, "f32"), (64, 70, 5, "f32"), (32, 37, 1, "f32"), (64, 100, 16, "bf16"), (63, 50, 64, "bf16"),
         (64, 130, 64, "f32")]


def inputs(d, T, dtype, seed, B=2, H=3):
    w = synth.WORKLOADS["linear_small"].with_(B=B, H=H, T=T, d=d, dtype=dtype, seed=seed)
    inp = synth.make_inputs(w)
    return w, inp, torch_inputs(inp)


def check(name, got, want, w):
    bar = tolerance(w)
    for label, g, r in zip(name.split(","), got, want):
        assert np.all(np.isfinite(to64(g))), label
        assert rel_err(label, to64(g), r, bar) <= bar, label


@pytest.mark.parametrize("d,T,b,dtype", CASES)
def test_bias_matches_oracle(d, T, b, dtype):
    w, inp, t = inputs(d, T, dtype, 700 + d + T + b)
    beta0 = np.random.default_rng(d + T).standard_normal((w.H, d)).astype(np.float32) * 0.3
    got = ttt.ttt_linear_bias_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(beta0).cuda(), b)
    torch.cuda.synchronize()
    want = bias_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, beta0, b)
    check("Z,W_out,beta_out", got, want, w)


@pytest.mark.parametrize("d,T,b,dtype", CASES)
def test_token_eta_matches_oracle(d, T, b, dtype):
    w, inp, t = inputs(d, T, dtype, 710 + d + T + b)
    et = np.random.default_rng(T).uniform(0.0, 0.5, (w.B, w.H, T)).astype(np.float32)
    got = ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(et).cuda(), t["W0"], b)
    torch.cuda.synchronize()
    want = token_eta_primal(inp.q64, inp.k64, inp.v64, et, inp.W0_64, b)
    check("Z,W_out", got, want, w)


@pytest.mark.parametrize("d,T,b,dtype", CASES)
def test_layer_norm_residual_matches_oracle(d, T, b, dtype):
    w, inp, t = inputs(d, T, dtype, 720 + d + T + b)
    g = np.random.default_rng(d * T)
    gamma = (1.0 + 0.2 * g.standard_normal((w.H, d))).astype(np.float32)
    beta = (0.1 * g.standard_normal((w.H, d))).astype(np.float32)
    got = ttt.ttt_linear_ln_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(gamma).cuda(),
                                torch.from_numpy(beta).cuda(), b)
    torch.cuda.synchronize()
    want = ln_residual_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, gamma, beta, b)
    check("Z,W_out", got, want, w)


@pytest.mark.parametrize("d,T,b,dtype", CASES)
def test_momentum_matches_oracle(d, T, b, dtype):
    w, inp, t = inputs(d, T, dtype, 730 + d + T + b)
    g = np.random.default_rng(d + 2 * T)
    alpha = g.uniform(0.05, 0.3, w.H).astype(np.float32)
    beta = g.uniform(0.5, 0.9, w.H).astype(np.float32)
    got = ttt.ttt_linear_momentum_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(alpha).cuda(),
                                      torch.from_numpy(beta).cuda(), t["W0"], b)
    torch.cuda.synchronize()
    want = momentum_primal(inp.q64, inp.k64, inp.v64, alpha, beta, inp.W0_64, b)
    check("Z,W_out,M_out", got, want, w)


def test_variants_reduce_to_plain_ttt_linear():
    """Two variants at settings where they are plain TTT-Linear (a per-token rate equal to the
    head's eta everywhere; momentum with beta = 0 and alpha = eta) equal the library's plain
    fp32 SIMT path on the same inputs within fp32 rounding."""
    w, inp, t = inputs(64, 96, "f32", 741)
    Zp, Wp = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16,
                                options={"force_path": ttt.PATH_SIMT})
    et = t["eta"][None, :, None].expand(w.B, w.H, w.T).contiguous()
    Zt, Wt = ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], et, t["W0"], 16)
    Zm, Wm, _ = ttt.ttt_linear_momentum_fwd(t["Q"], t["K"], t["V"], t["eta"], torch.zeros_like(t["eta"]), t["W0"], 16)
    torch.cuda.synchronize()
    for Z, Wo in ((Zt, Wt), (Zm, Wm)):
        assert float((Z - Zp).abs().max()) < 1e-5 and float((Wo - Wp).abs().max()) < 1e-5


@pytest.mark.parametrize("variant", ["bias", "token_eta", "ln", "momentum"])
def test_variants_medium_bf16(variant):
    """B1 H2 T1024 d64 b16, bf16 operands: every unit against the oracle."""
    w, inp, t = inputs(64, 1024, "bf16", 750, B=1, H=2)
    g = np.random.default_rng(7)
    if variant == "bias":
        beta0 = (0.3 * g.standard_normal((w.H, 64))).astype(np.float32)
        got = ttt.ttt_linear_bias_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(beta0).cuda(), 16)
        want, names = bias_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, beta0, 16), "Z,W_out,beta_out"
    elif variant == "token_eta":
        et = g.uniform(0.0, 0.5, (1, w.H, w.T)).astype(np.float32)
        got = ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(et).cuda(), t["W0"], 16)
        want, names = token_eta_primal(inp.q64, inp.k64, inp.v64, et, inp.W0_64, 16), "Z,W_out"
    elif variant == "ln":
        gamma = (1.0 + 0.2 * g.standard_normal((w.H, 64))).astype(np.float32)
        beta = (0.1 * g.standard_normal((w.H, 64))).astype(np.float32)
        got = ttt.ttt_linear_ln_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(gamma).cuda(),
                                    torch.from_numpy(beta).cuda(), 16)
        want, names = ln_residual_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, gamma, beta, 16), "Z,W_out"
    else:
        alpha = np.full(w.H, 0.1, np.float32)
        beta = np.array([0.6, 0.9], np.float32)
        got = ttt.ttt_linear_momentum_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(alpha).cuda(),
                                          torch.from_numpy(beta).cuda(), t["W0"], 16)
        want, names = momentum_primal(inp.q64, inp.k64, inp.v64, alpha, beta, inp.W0_64, 16), "Z,W_out,M_out"
    torch.cuda.synchronize()
    check(names, got, want, w)


FAST_BIAS = [(63, 50, 16, 2, 3), (16, 40, 16, 2, 3), (32, 130, 64, 2, 2), (1, 33, 16, 1, 2), (48, 2048, 16, 1, 2)]


@pytest.mark.parametrize("d,T,b,B,H", FAST_BIAS)
def test_bias_fast_path_matches_oracle(d, T, b, B, H):
    """ttt_linear_bias_fwd_ex with bf16 operands: padded inputs through the tensor-core kernels
    (T = 2048 takes the segment-parallel plan), against the oracle; the status word is clean."""
    w, inp, t = inputs(d, T, "bf16", 760 + d + T + b, B=B, H=H)
    beta0 = np.random.default_rng(d + T).standard_normal((w.H, d)).astype(np.float32) * 0.3
    need = ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_BIAS, ttt.TTT_BF16, B, H, T, d, b)
    assert need > 256
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    got = ttt.ttt_linear_bias_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(beta0).cuda(), b,
                                  fast=True, workspace=ws)
    torch.cuda.synchronize()
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    want = bias_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, beta0, b)
    check("Z,W_out,beta_out", got, want, w)


FAST_TOK = [(64, 100, 16, 2, 3), (64, 2048, 16, 1, 2), (40, 70, 32, 2, 2), (64, 37, 64, 1, 3), (16, 48, 16, 1, 1)]


@pytest.mark.parametrize("d,T,b,B,H", FAST_TOK)
def test_token_eta_fast_path_matches_oracle(d, T, b, B, H):
    """ttt_linear_token_eta_fwd_ex with bf16 operands: sqrt(eta_t)-scaled keys and values through
    the tensor-core kernels (in place at d = 64, padded below), against the oracle."""
    w, inp, t = inputs(d, T, "bf16", 770 + d + T + b, B=B, H=H)
    et = np.random.default_rng(T + d).uniform(0.0, 0.5, (B, H, T)).astype(np.float32)
    ws = torch.empty(ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, ttt.TTT_BF16, B, H, T, d, b),
                     dtype=torch.uint8, device="cuda")
    got = ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(et).cuda(), t["W0"], b, fast=True,
                                       workspace=ws)
    torch.cuda.synchronize()
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    want = token_eta_primal(inp.q64, inp.k64, inp.v64, et, inp.W0_64, b)
    check("Z,W_out", got, want, w)


@pytest.mark.parametrize("d,T,b,dtype", [(16, 40, 16, "f32"), (64, 70, 5, "bf16")])
def test_fast_calls_run_the_variant_kernel_where_padding_does_not_apply(d, T, b, dtype):
    """fp32 operands or b % 16 != 0: the *_ex calls take the fp32 variant kernel (a 256-byte
    workspace) and match the oracle at that dtype's bar."""
    w, inp, t = inputs(d, T, dtype, 780 + d + T + b)
    et = np.random.default_rng(T).uniform(0.0, 0.5, (w.B, w.H, T)).astype(np.float32)
    code = ttt.TTT_BF16 if dtype == "bf16" else ttt.TTT_F32
    assert ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, code, w.B, w.H, T, d, b) == 256
    got = ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(et).cuda(), t["W0"], b, fast=True)
    torch.cuda.synchronize()
    check("Z,W_out", got, token_eta_primal(inp.q64, inp.k64, inp.v64, et, inp.W0_64, b), w)


def test_fast_token_eta_reports_a_negative_rate():
    """A negative per-token rate has no square root: the call finishes and the status word says
    TTT_ERR_DEVICE_CHECK; the next call with valid rates is clean again."""
    w, inp, t = inputs(64, 48, "bf16", 790, B=1, H=2)
    et = np.full((1, 2, 48), 0.2, np.float32)
    et[0, 1, 17] = -0.1
    ws = torch.empty(ttt.ttt_linear_variant_workspace_bytes(ttt.TTT_INNER_TOKEN_ETA, ttt.TTT_BF16, 1, 2, 48, 64, 16),
                     dtype=torch.uint8, device="cuda")
    ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(et).cuda(), t["W0"], 16, fast=True,
                                 workspace=ws)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_ERR_DEVICE_CHECK
    et[0, 1, 17] = 0.1
    got = ttt.ttt_linear_token_eta_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(et).cuda(), t["W0"], 16, fast=True,
                                       workspace=ws)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    check("Z,W_out", got, token_eta_primal(inp.q64, inp.k64, inp.v64, et, inp.W0_64, 16), w)


FAST_MOM = [(1, 2, 1, 0.6, 16), (1, 2, 3, 0.6, 16), (2, 3, 16, 0.9, 16), (2, 3, 37, 0.5, 16),
            (1, 2, 100, 0.0, 16), (1, 2, 1024, 0.8, 16), (1, 2, 2048, 0.95, 16), (2, 3, 100, 0.7, 32),
            (1, 2, 1000, 0.5, 64), (1, 2, 600, 0.5, 256)]


@pytest.mark.parametrize("B,H,T,beta,b", FAST_MOM)
def test_momentum_fast_path_matches_oracle(B, H, T, beta, b):
    """bf16, d = 64, b a multiple of 16 on the tensor-core momentum kernel (forced, so that no other
    kernel can serve): a single short chunk, ragged last chunks, beta = 0 (plain TTT-Linear with the
    last token's gradient as M), strong momentum, sequences of 64 and 128 chunks, and chunks of 2,
    4 and 16 tiles (each tile's E from the chunk-start W)."""
    w, inp, t = inputs(64, T, "bf16", 800 + T + b, B=B, H=H)
    alpha = np.linspace(0.05, 0.15, H).astype(np.float32)
    betas = (beta * (1.0 - 0.05 * np.arange(H))).astype(np.float32)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    got = ttt.ttt_linear_momentum_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(alpha).cuda(),
                                      torch.from_numpy(betas).cuda(), t["W0"], b, fast=True, workspace=ws,
                                      options={"force_path": ttt.PATH_TENSOR})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    want = momentum_primal(inp.q64, inp.k64, inp.v64, alpha, betas, inp.W0_64, b)
    check("Z,W_out,M_out", got, want, w)


def test_momentum_fast_call_takes_the_variant_kernel_elsewhere():
    """fp32 operands (or d != 64, b != 16): ttt_linear_momentum_fwd_ex runs the fp32 variant kernel
    and matches the oracle at the fp32 bar."""
    w, inp, t = inputs(32, 45, "f32", 820)
    alpha = np.full(w.H, 0.1, np.float32)
    betas = np.full(w.H, 0.7, np.float32)
    got = ttt.ttt_linear_momentum_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(alpha).cuda(),
                                      torch.from_numpy(betas).cuda(), t["W0"], 16, fast=True)
    torch.cuda.synchronize()
    check("Z,W_out,M_out", got, momentum_primal(inp.q64, inp.k64, inp.v64, alpha, betas, inp.W0_64, 16), w)


def test_momentum_fast_path_bounded_wait_reports_timeout():
    """The load pipeline never fills: the tensor kernel's waits run out after 1 ms, the status says
    TTT_ERR_TIMEOUT, reading clears it, and the next call on the same context matches the oracle."""
    w, inp, t = inputs(64, 64, "bf16", 830, B=1, H=2)
    alpha, betas = np.full(w.H, 0.1, np.float32), np.full(w.H, 0.8, np.float32)
    args = (t["Q"], t["K"], t["V"], torch.from_numpy(alpha).cuda(), torch.from_numpy(betas).cuda(), t["W0"], 16)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ttt.ttt_linear_momentum_fwd(*args, fast=True, workspace=ws,
                                options={"inject_stall": 1, "wait_timeout_ns": 1_000_000, "force_path": ttt.PATH_TENSOR})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_ERR_TIMEOUT
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    got = ttt.ttt_linear_momentum_fwd(*args, fast=True, workspace=ws)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    check("Z,W_out,M_out", got, momentum_primal(inp.q64, inp.k64, inp.v64, alpha, betas, inp.W0_64, 16), w)


FAST_LN = [(1, 2, 1, 16), (1, 2, 3, 16), (2, 3, 16, 16), (2, 3, 37, 16), (1, 2, 100, 16), (1, 2, 1024, 16),
           (1, 2, 2048, 16), (2, 3, 100, 32), (1, 2, 512, 64), (1, 2, 600, 256)]


def ln_params(H, seed):
    g = np.random.default_rng(seed)
    return ((1.0 + 0.2 * g.standard_normal((H, 64))).astype(np.float32),
            (0.1 * g.standard_normal((H, 64))).astype(np.float32))


@pytest.mark.parametrize("B,H,T,b", FAST_LN)
def test_ln_fast_path_matches_oracle(B, H, T, b):
    """bf16, d = 64, b a multiple of 16 on the tensor-core LN + residual kernel (forced, so that no
    other kernel can serve): a single short chunk, ragged last chunks, sequences of 64 and 128 chunks,
    and chunks of 2, 4 and 16 tiles (each tile's Y and E from the chunk-start W)."""
    w, inp, t = inputs(64, T, "bf16", 840 + T + b, B=B, H=H)
    gamma, beta = ln_params(w.H, T)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    got = ttt.ttt_linear_ln_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(gamma).cuda(),
                                torch.from_numpy(beta).cuda(), b, fast=True, workspace=ws,
                                options={"force_path": ttt.PATH_TENSOR})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    want = ln_residual_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, gamma, beta, b)
    check("Z,W_out", got, want, w)


def test_ln_fast_call_takes_the_variant_kernel_elsewhere():
    """fp32 operands (or d != 64, b != 16): ttt_linear_ln_fwd_ex runs the fp32 variant kernel and
    matches the oracle at the fp32 bar."""
    w, inp, t = inputs(32, 45, "f32", 850)
    g = np.random.default_rng(3)
    gamma = (1.0 + 0.2 * g.standard_normal((w.H, 32))).astype(np.float32)
    beta = (0.1 * g.standard_normal((w.H, 32))).astype(np.float32)
    got = ttt.ttt_linear_ln_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(gamma).cuda(),
                                torch.from_numpy(beta).cuda(), 16, fast=True)
    torch.cuda.synchronize()
    check("Z,W_out", got, ln_residual_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, gamma, beta, 16), w)


def test_ln_fast_path_bounded_wait_reports_timeout():
    """The load pipeline never fills: the tensor kernel's waits run out after 1 ms, the status says
    TTT_ERR_TIMEOUT, reading clears it, and the next call on the same context matches the oracle."""
    w, inp, t = inputs(64, 64, "bf16", 860, B=1, H=2)
    gamma, beta = ln_params(w.H, 5)
    args = (t["Q"], t["K"], t["V"], t["eta"], t["W0"], torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda(),
            16)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ttt.ttt_linear_ln_fwd(*args, fast=True, workspace=ws,
                          options={"inject_stall": 1, "wait_timeout_ns": 1_000_000, "force_path": ttt.PATH_TENSOR})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_ERR_TIMEOUT
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    got = ttt.ttt_linear_ln_fwd(*args, fast=True, workspace=ws)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    check("Z,W_out", got, ln_residual_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, gamma, beta, 16), w)


@pytest.mark.parametrize("variant", ["momentum", "ln"])
def test_variant_tensor_kernels_full_size_sampled(variant):
    """B8 H12 T8192 d64 bf16 (the 125M-shaped workload the benchmark times): the momentum and
    LN + residual tensor kernels over all 96 units, the oracle on two sampled ones."""
    w = synth.WORKLOADS["linear_125m"]
    full = synth.make_inputs(w, want_exact=False)
    t = torch_inputs(full)
    units = [(0, 0), (7, 11)]
    sub = synth.make_inputs(w, units=units)
    heads = [h for _, h in units]
    if variant == "momentum":
        alpha = np.full(w.H, 0.1, np.float32)  # alpha / (1 - beta) <= 1: a stable step at unit-norm keys
        beta = np.linspace(0.5, 0.9, w.H).astype(np.float32)
        got = ttt.ttt_linear_momentum_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(alpha).cuda(),
                                          torch.from_numpy(beta).cuda(), t["W0"], 16, fast=True,
                                          options={"force_path": ttt.PATH_TENSOR})
        want = momentum_primal(sub.q64, sub.k64, sub.v64, alpha[heads], beta[heads], sub.W0_64, 16)
        names = ("Z", "W_out", "M_out")
    else:
        gamma, beta = ln_params(w.H, 11)
        eta = np.full(w.H, 0.05, np.float32)
        got = ttt.ttt_linear_ln_fwd(t["Q"], t["K"], t["V"], torch.from_numpy(eta).cuda(), t["W0"],
                                    torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda(), 16, fast=True,
                                    options={"force_path": ttt.PATH_TENSOR})
        want = ln_residual_primal(sub.q64, sub.k64, sub.v64, eta[heads], sub.W0_64, gamma[heads], beta[heads], 16)
        names = ("Z", "W_out")
    torch.cuda.synchronize()
    bar = tolerance(w)
    for k, (n, h) in enumerate(units):
        for name, g, r in zip(names, got, want):
            assert rel_err(f"{variant} {name} unit {n},{h}", to64(g[n, h]), r[0, k], bar) <= bar, (name, n, h)
    assert bool(torch.isfinite(got[0].float()).all())
