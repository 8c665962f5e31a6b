"""TTT-Linear on the GPU (through the C ABI) against the fp64 oracle.

Small cases run the oracle over every unit; the full-size workloads run the
GPU on everything and the oracle on sampled (batch row, head) units, which the
counter-based generator can draw on their own. Bars: rel-L2 <= 1e-4 with fp32
operands, <= 2e-2 with bf16 operands (fp32 state and accumulation).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import test_sequence_layers_06_b300 as ttt
from ttt_testlib import oracle_linear, rel_err, rel_l2, to64, tolerance, torch_inputs, worst_unit_rel

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def run_linear(inp, b, path=ttt.PATH_AUTO):
    t = torch_inputs(inp)
    opts = None if path == ttt.PATH_AUTO else {"force_path": path}
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], b, options=opts)
    torch.cuda.synchronize()
    return to64(Z), to64(Wo)


def check(inp, b, path=ttt.PATH_AUTO, tol=None):
    tol = tolerance(inp.w) if tol is None else tol
    Z, Wo = run_linear(inp, b, path)
    Zr, Wr = oracle_linear(inp, b)
    ez, ew = rel_err("Z", Z, Zr, tol), rel_err("W_out", Wo, Wr, tol)
    assert np.all(np.isfinite(Z)) and np.all(np.isfinite(Wo))
    assert ez <= tol and ew <= tol, (ez, ew, worst_unit_rel(Z, Zr))
    return ez, ew


def test_tiny_fp32_workload():
    """B1 H1 T64 d16 b16, fp32 operands: the 1e-4 bar."""
    inp = synth.make_inputs(W["linear_tiny_f32"])
    ez, ew = check(inp, 16)
    assert ez < 1e-5 and ew < 1e-5


def test_small_bf16_workload_tensor_path():
    """B2 H4 T2048 d64 b16, bf16: the tensor-core kernel."""
    inp = synth.make_inputs(W["linear_small"])
    check(inp, 16, ttt.PATH_TENSOR)


def test_small_bf16_workload_automatic_plan():
    """B2 H4 T2048 d64 b16, bf16, with no forced path: 8 units are too few to fill the
    GPU, so the library's own plan is the segment-parallel form (tcgen05 affine maps,
    combine, per-segment read-out). Every unit against the oracle."""
    w = W["linear_small"]
    plan = ttt.ttt_linear_plan(w.B, w.H, w.T, w.d, w.b)
    assert plan["path"] == ttt.PATH_SEGMENTED and plan["seg_count"] >= 2 and plan["affine"] == 2, plan
    check(synth.make_inputs(w), w.b)


def test_small_bf16_workload_simt_path():
    inp = synth.make_inputs(W["linear_small"])
    check(inp, 16, ttt.PATH_SIMT)


@pytest.mark.parametrize("T,b", [(1, 16), (15, 16), (17, 16), (50, 16), (100, 32), (130, 64), (300, 256),
                                 (64, 48), (0, 16), (1000, 512)])
def test_tensor_path_ragged_and_chunk_sizes(T, b):
    """Several 16-token tiles with a ragged tail; chunks of 1, 2, 3 and 16 tiles."""
    w = W["linear_small"].with_(B=1, H=3, T=T, seed=100 + T)
    inp = synth.make_inputs(w)
    if T == 0:
        Z, Wo = run_linear(inp, b, ttt.PATH_TENSOR)
        assert Z.size == 0 and np.array_equal(Wo[0], inp.W0.astype(np.float64))
        return
    check(inp, b, ttt.PATH_TENSOR)


@pytest.mark.parametrize("T,b,seg", [(1024, 16, 256), (1000, 16, 256), (64, 16, 32), (777, 16, 16),
                                     (2048, 64, 512), (2560, 256, 512), (2048, 128, 512), (1300, 32, 64),
                                     (4096, 16, 1024), (4096, 1024, 2048), (6144, 2048, 2048)])
def test_segment_parallel_path(T, b, seg):
    """Segment-parallel form: per-segment affine maps, the combine, and a read-out
    per segment from its start state. Full, ragged and one-tile segments; chunks
    of 1, 2, 4, 8 and 16 tiles (one to four 64-token steps per chunk); per-head eta."""
    w = W["linear_125m"].with_(B=2, H=3, T=T, seed=300 + T + b + seg)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    opts = {"force_path": ttt.PATH_SEGMENTED, "seg_len": seg}
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], b, options=opts)
    torch.cuda.synchronize()
    Zr, Wr = oracle_linear(inp, b)
    ez, ew = rel_err("Z", to64(Z), Zr, tolerance(w)), rel_err("W_out", to64(Wo), Wr, tolerance(w))
    assert ez <= tolerance(w) and ew <= tolerance(w), (ez, ew, worst_unit_rel(to64(Z), Zr))


@pytest.mark.parametrize("pieces,T,seg", [(2, 4096, 512), (3, 4096, 512), (5, 2560, 256), (8, 2048, 256)])
def test_segment_pieces_are_bit_identical_to_one_piece(pieces, T, seg):
    """Cutting the segments into pieces (the affine maps of piece p + 1 on a second
    stream beside the read-out of piece p, the combine continued piece by piece from
    the stored start states) changes only when each kernel runs, not what it computes:
    Z and W_out are bit-identical to the one-piece run, and that run matches the oracle."""
    w = W["linear_125m"].with_(B=2, H=3, T=T, seed=500 + pieces)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    base = {"force_path": ttt.PATH_SEGMENTED, "seg_len": seg}
    assert ttt.ttt_linear_plan(w.B, w.H, T, w.d, 16, options=dict(base, pieces=pieces))["pieces"] == pieces
    Z1, W1 = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16, options=dict(base, pieces=1))
    Zp, Wp = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16, options=dict(base, pieces=pieces))
    torch.cuda.synchronize()
    assert torch.equal(Z1.view(torch.int16), Zp.view(torch.int16)) and torch.equal(W1, Wp)
    Zr, Wr = oracle_linear(inp, 16)
    assert rel_err("Z", to64(Zp), Zr, tolerance(w)) <= tolerance(w)
    assert rel_err("W_out", to64(Wp), Wr, tolerance(w)) <= tolerance(w)


def test_concurrent_calls_on_two_streams_are_bit_identical():
    """Two independent calls on two streams at once, and the piecewise form, put tcgen05
    affine-map CTAs on the same SMs as read-out CTAs. Every result must be bit-identical to a
    lone call. (A read-out warp that released its stage to the next TMA load before its last
    load from that stage had completed read the next tile's K once in about eight such runs;
    a stage is now released only after all of its loaded registers are consumed.)"""
    w = W["linear_long"].with_(T=32768, seed=61)
    t = torch_inputs(synth.make_inputs(w, want_exact=False))
    opts = {"force_path": ttt.PATH_SEGMENTED, "seg_len": 1024}

    def call(stream=None, **extra):
        Z = torch.empty_like(t["Q"])
        Wo = torch.empty((w.B, w.H, w.d, w.d), device="cuda")
        ws = torch.empty(ttt.ttt_workspace_bytes(w.B, w.H, w.T, w.d, w.b, 0, opts), dtype=torch.uint8, device="cuda")
        ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], w.b, Z=Z, W_out=Wo, workspace=ws,
                           stream=stream, options=dict(opts, **extra))
        return Z, Wo, ws

    Zr, Wr, _ = call()
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    runs = []
    for _ in range(24):
        runs += [call(s1), call(s2)]
    for _ in range(8):
        runs.append(call(pieces=4))
    torch.cuda.synchronize()
    for Z, Wo, ws in runs:
        assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
        assert torch.equal(Z.view(torch.int16), Zr.view(torch.int16)) and torch.equal(Wo, Wr)


def test_segment_parallel_equals_one_pass():
    """The two tensor-core forms agree with each other within bf16 rounding."""
    w = W["linear_small"].with_(B=2, H=4, T=2048, seed=41)
    t = torch_inputs(synth.make_inputs(w, want_exact=False))
    Z1, W1 = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16,
                                options={"force_path": ttt.PATH_TENSOR})
    Z2, W2 = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16,
                                options={"force_path": ttt.PATH_SEGMENTED, "seg_len": 256})
    torch.cuda.synchronize()
    assert rel_l2(to64(Z2), to64(Z1)) < 1e-2 and rel_l2(to64(W2), to64(W1)) < 1e-2


def test_segment_parallel_bounded_wait_reports_timeout():
    w = W["linear_small"].with_(B=1, H=2, T=512)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    opts = {"force_path": ttt.PATH_SEGMENTED, "seg_len": 128}
    ws = torch.zeros(ttt.ttt_workspace_bytes(1, 2, 512, 64, 16, 0, opts), dtype=torch.uint8, device="cuda")
    ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16, workspace=ws,
                       options=dict(opts, inject_stall=1, wait_timeout_ns=1_000_000))
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_ERR_TIMEOUT
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16, workspace=ws, options=opts)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
    Zr, Wr = oracle_linear(inp, 16)
    assert rel_l2(to64(Z), Zr) <= 2e-2 and rel_l2(to64(Wo), Wr) <= 2e-2


@pytest.mark.parametrize("d,T,b,dtype", [(16, 40, 16, "f32"), (32, 37, 5, "f32"), (64, 33, 1, "f32"),
                                         (16, 64, 16, "bf16"), (32, 70, 7, "bf16"), (64, 19, 3, "bf16"),
                                         (8, 23, 4, "f32")])
def test_simt_path_shapes(d, T, b, dtype):
    w = W["linear_small"].with_(B=2, H=2, T=T, d=d, dtype=dtype, seed=200 + d + T)
    check(synth.make_inputs(w), b)


def test_fp32_bigger_workload_meets_1e4():
    w = W["linear_tiny_f32"].with_(B=2, H=3, T=512, d=64, w_std=0.02, q_mode="normalized")
    check(synth.make_inputs(w), 16)


@pytest.mark.parametrize("name,units", [("linear_125m", [(0, 0), (3, 7), (7, 11)])])
def test_full_size_125m_sampled(name, units):
    """B8 H12 T8192: GPU over all 96 units, oracle on sampled ones; per-head eta differs."""
    w = W[name]
    full = synth.make_inputs(w, want_exact=False)
    t = torch_inputs(full)
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], w.b)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(Z.float()).all()) and bool(torch.isfinite(Wo).all())
    sub = synth.make_inputs(w, units=units)
    Zr, Wr = oracle_linear(sub, w.b)
    for k, (n, h) in enumerate(units):
        assert rel_err(f"Z unit {n},{h}", to64(Z[n, h]), Zr[0, k], tolerance(w)) <= tolerance(w)
        assert rel_err(f"W_out unit {n},{h}", to64(Wo[n, h]), Wr[0, k], tolerance(w)) <= tolerance(w)


@pytest.mark.parametrize("b", [16, 64, 256])
def test_full_size_long_context_sampled(b):
    """B1 H32 T131072 at b in {16, 64, 256} (the automatic plan runs the
    segment-parallel form here, as the benchmark does): oracle on two sampled heads."""
    w = W["linear_long"].with_(b=b)
    full = synth.make_inputs(w, want_exact=False)
    t = torch_inputs(full)
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], b)
    torch.cuda.synchronize()
    units = [(0, 5), (0, 31)]
    sub = synth.make_inputs(w, units=units)
    Zr, Wr = oracle_linear(sub, b)
    for k, (n, h) in enumerate(units):
        ez = rel_err(f"Z head {h}", to64(Z[n, h]), Zr[0, k], tolerance(w))
        ew = rel_err(f"W_out head {h}", to64(Wo[n, h]), Wr[0, k], tolerance(w))
        assert ez <= tolerance(w) and ew <= tolerance(w), (h, ez, ew)
    # every head: finite and bounded (the state update contracts for these eta)
    assert bool(torch.isfinite(Z.float()).all()) and float(Wo.abs().max()) < 10.0

    # One decode token from the final state (T % b == 0, so anchor = running = W_out and
    # pos = T), for every head on the GPU; the oracle continues from its own W_out.
    tok = synth.make_inputs(w.with_(T=1, seed=w.seed + 7919))
    tt = torch_inputs(tok)
    Wa, Wrun = Wo.clone(), Wo.clone()
    z = ttt.ttt_linear_decode_step(tt["Q"][:, :, 0].contiguous(), tt["K"][:, :, 0].contiguous(),
                                   tt["V"][:, :, 0].contiguous(), t["eta"], Wa, Wrun, w.T, b)
    torch.cuda.synchronize()
    hs = [h for _, h in units]
    zq, Wa2, Wr2 = oracle.linear_decode_step(tok.q64[:, hs, 0], tok.k64[:, hs, 0], tok.v64[:, hs, 0], sub.eta64,
                                              Wr, Wr, w.T, b)
    for k, h in enumerate(hs):
        ez = rel_err(f"decode z head {h}", to64(z[0, h]), zq[0, k], tolerance(w))
        ew = rel_err(f"decode W_run head {h}", to64(Wrun[0, h]), Wr2[0, k], tolerance(w))
        assert ez <= tolerance(w) and ew <= tolerance(w), ("decode", h, ez, ew)
        assert rel_l2(to64(Wa[0, h]), Wa2[0, k]) <= tolerance(w)


def test_chain_two_calls_equal_one():
    w = W["linear_small"].with_(B=1, H=2, T=96, seed=9)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    Z, Wo = ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16)
    Za, Wa = ttt.ttt_linear_fwd(t["Q"][:, :, :48].contiguous(), t["K"][:, :, :48].contiguous(),
                                t["V"][:, :, :48].contiguous(), t["eta"], t["W0"], 16)
    Zb, Wb = ttt.ttt_linear_fwd(t["Q"][:, :, 48:].contiguous(), t["K"][:, :, 48:].contiguous(),
                                t["V"][:, :, 48:].contiguous(), t["eta"], Wa[0].contiguous(), 16)
    torch.cuda.synchronize()
    assert rel_l2(to64(torch.cat([Za, Zb], 2)), to64(Z)) < 1e-2
    assert rel_l2(to64(Wb), to64(Wo)) < 1e-3


def test_decode_continues_forward():
    """Prefill T1 (b | T1), then decode N tokens one by one: equals the oracle over T1 + N."""
    T1, N = 32, 20
    w = W["linear_small"].with_(B=2, H=3, T=T1 + N, seed=77)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    _, Wp = ttt.ttt_linear_fwd(t["Q"][:, :, :T1].contiguous(), t["K"][:, :, :T1].contiguous(),
                               t["V"][:, :, :T1].contiguous(), t["eta"], t["W0"], 16)
    Wa, Wr = Wp.clone(), Wp.clone()
    zs = []
    for s in range(N):
        tt = T1 + s
        zs.append(ttt.ttt_linear_decode_step(t["Q"][:, :, tt].contiguous(), t["K"][:, :, tt].contiguous(),
                                             t["V"][:, :, tt].contiguous(), t["eta"], Wa, Wr, tt, 16))
    torch.cuda.synchronize()
    Zr, Wref = oracle_linear(inp, 16)
    assert rel_err("decoded z", to64(torch.stack(zs, 2)), Zr[:, :, T1:], 2e-2) <= 2e-2
    assert rel_err("W_run", to64(Wr), Wref, 2e-2) <= 2e-2


@pytest.mark.parametrize("dtype,d,N", [("bf16", 64, 37), ("f32", 64, 50), ("f32", 40, 21), ("bf16", 64, 1)])
def test_decode_many_tokens_in_one_launch_continues_forward(dtype, d, N):
    """Prefill T1 (b | T1), then decode N tokens in one ttt_linear_decode launch (the
    anchor moves at every chunk boundary inside the launch): equals the oracle over
    T1 + N; a state width that is not a multiple of 16 leaves a partial column slice."""
    T1, b = 32, 16
    w = W["linear_small"].with_(B=2, H=3, T=T1 + N, d=d, dtype=dtype, seed=90 + N + d)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    sl = lambda x, a, e: x[:, :, a:e].contiguous()
    _, Wp = ttt.ttt_linear_fwd(sl(t["Q"], 0, T1), sl(t["K"], 0, T1), sl(t["V"], 0, T1), t["eta"], t["W0"], b)
    Wa, Wr = Wp.clone(), Wp.clone()
    z = ttt.ttt_linear_decode(sl(t["Q"], T1, T1 + N), sl(t["K"], T1, T1 + N), sl(t["V"], T1, T1 + N), t["eta"],
                              Wa, Wr, T1, b)
    torch.cuda.synchronize()
    Zr, Wref = oracle_linear(inp, b)
    bar = tolerance(w)
    assert rel_err("decoded z (one launch)", to64(z), Zr[:, :, T1:], bar) <= bar
    assert rel_err("W_run (one launch)", to64(Wr), Wref, bar) <= bar
    # the anchor is the state at the start of the current chunk
    n_full = ((T1 + N) // b) * b
    _, Wanc = oracle.linear_primal(inp.q64[:, :, :n_full], inp.k64[:, :, :n_full], inp.v64[:, :, :n_full],
                                   inp.eta64, inp.W0_64, b)
    assert rel_l2(to64(Wa), Wanc) <= bar
    # no tokens: nothing changes
    Wa2, Wr2 = Wa.clone(), Wr.clone()
    e = torch.empty((w.B, w.H, 0, d), dtype=t["Q"].dtype, device="cuda")
    ttt.ttt_linear_decode(e, e, e, t["eta"], Wa2, Wr2, T1 + N, b)
    torch.cuda.synchronize()
    assert torch.equal(Wa2, Wa) and torch.equal(Wr2, Wr)


def test_decode_fp32_single_token_matches_oracle():
    g = np.random.default_rng(3)
    B, H, d = 2, 4, 64
    q, k, v = (g.standard_normal((B, H, d)).astype(np.float32) for _ in range(3))
    eta = g.uniform(0.05, 0.5, H).astype(np.float32)
    Wa = (0.05 * g.standard_normal((B, H, d, d))).astype(np.float32)
    Wr = (0.05 * g.standard_normal((B, H, d, d))).astype(np.float32)
    for pos, b in ((5, 16), (15, 16)):
        z, Wa2, Wr2 = oracle.linear_decode_step(q, k, v, eta, Wa, Wr, pos, b)
        tq = [torch.from_numpy(x).cuda() for x in (q, k, v, eta)]
        ta, tr = torch.from_numpy(Wa).cuda(), torch.from_numpy(Wr).cuda()
        zz = ttt.ttt_linear_decode_step(*tq[:3], tq[3], ta, tr, pos, b)
        torch.cuda.synchronize()
        assert rel_err("decode z fp32", to64(zz), z, 1e-4) < 1e-5
        assert rel_err("decode W_run fp32", to64(tr), Wr2, 1e-4) < 1e-6 and rel_l2(to64(ta), Wa2) < 1e-6


def test_bounded_wait_reports_timeout_and_context_survives():
    """The load pipeline is told never to fill: the consumers' wait runs out
    after 1 ms, the kernel returns, the status says TTT_ERR_TIMEOUT, and the
    next call on the same context works."""
    w = W["linear_small"].with_(B=1, H=2, T=64)
    inp = synth.make_inputs(w)
    t = torch_inputs(inp)
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16, workspace=ws,
                       options={"inject_stall": 1, "wait_timeout_ns": 1_000_000, "force_path": ttt.PATH_TENSOR})
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_ERR_TIMEOUT
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK  # reading clears it
    check(inp, 16, ttt.PATH_TENSOR)
    ttt.ttt_linear_fwd(t["Q"], t["K"], t["V"], t["eta"], t["W0"], 16, workspace=ws)
    assert ttt.ttt_last_device_status(ws) == ttt.TTT_OK
