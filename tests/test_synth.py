"""The seeded input generator: rounding, counters and recipes (CPU only)."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch_on_fp32_values():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32).astype(np.float64)
    bits, back = synth.round_bf16(x)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(bits.view(np.int16), ref)
    assert np.array_equal(back, synth.bf16_bits_to_f64(bits))


def test_bf16_ties_round_to_even_from_fp64():
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -40])
    _, back = synth.round_bf16(x)
    assert back.tolist() == [1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7]


def test_counter_slices_match_full_draw():
    full = synth.normal(5, 2, 1000)
    assert np.array_equal(synth.normal(5, 2, 77, first=333), full[333:410])
    assert np.array_equal(synth.normal(5, 2, 1, first=999), full[999:])
    assert not np.array_equal(synth.normal(6, 2, 1000), full)
    assert abs(full.mean()) < 0.15 and abs(full.std() - 1) < 0.1
    u = synth.uniform(1, 1, 100000)
    assert u.min() > 0 and u.max() <= 1 and abs(u.mean() - 0.5) < 0.01


def test_workload_recipes():
    w = synth.WORKLOADS["linear_small"].with_(T=64)
    x = synth.make_inputs(w)
    assert x.q.dtype == np.uint16 and x.q.shape == (2, 4, 64, 64)
    n = np.linalg.norm(x.k64, axis=-1)
    assert np.all(np.abs(n - 1) < 1e-2)
    assert np.allclose(x.eta, 0.1) and x.W0.shape == (4, 64, 64)
    y = synth.make_inputs(w, units=[(1, 3), (0, 0)])
    assert np.array_equal(y.q[0, 0], x.q[1, 3]) and np.array_equal(y.v64[0, 1], x.v64[0, 0])
    assert np.array_equal(y.W0[0], x.W0[3])
    t = synth.make_inputs(synth.WORKLOADS["linear_tiny_f32"])
    assert t.q.dtype == np.float32 and np.all(t.W0 == 0) and t.eta[0] == np.float32(0.5)
    e = synth.make_eta(synth.WORKLOADS["linear_125m"])[0]
    assert e.min() >= 0.05 and e.max() <= 0.5 and len(set(e.tolist())) == 12
