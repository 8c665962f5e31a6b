"""Shared helpers for the parity tests: move synthetic inputs to the GPU, call
the library through its binding, call the oracle, compare."""
from __future__ import annotations

import os

import numpy as np

import oracle
import synth


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


# Every parity comparison's measured error, printed by conftest.py at the end of the run.
MARGINS: list = []


def record_margin(what: str, err: float, bar: float) -> float:
    """Keep one comparison's rel-L2 and its bar for the end-of-run margin table; returns err."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    MARGINS.append({"test": test, "what": what, "err": float(err), "bar": float(bar)})
    return err


def rel_err(what: str, x, ref, bar: float) -> float:
    """rel_l2(x, ref), recorded against `bar` (the caller still asserts)."""
    return record_margin(what, rel_l2(x, ref), bar)


def worst_unit_rel(x, ref) -> float:
    """Largest rel-L2 over (batch row, head) units (a diagnostic)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    B, H = ref.shape[:2]
    return max(rel_l2(x[n, h], ref[n, h]) for n in range(B) for h in range(H))


def torch_inputs(inp: synth.Inputs, device="cuda"):
    import torch
    if inp.q.dtype == np.uint16:
        cv = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        cv = lambda a: torch.from_numpy(a).to(device)
    out = dict(Q=cv(inp.q), K=cv(inp.k), V=cv(inp.v), eta=torch.from_numpy(inp.eta).to(device))
    if inp.W0 is not None:
        out["W0"] = torch.from_numpy(inp.W0).to(device)
    if inp.W1 is not None:
        out["W1"] = torch.from_numpy(inp.W1).to(device)
        out["W2"] = torch.from_numpy(inp.W2).to(device)
    return out


def to64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def tolerance(w: synth.Workload) -> float:
    """rel-L2 bars: 1e-4 for fp32 operands, 2e-2 for bf16 operands (fp32 state and accumulation)."""
    return 1e-4 if w.dtype == "f32" else 2e-2


def oracle_linear(inp: synth.Inputs, b: int):
    return oracle.linear_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, b)


def oracle_mlp(inp: synth.Inputs, b: int):
    return oracle.mlp_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W1_64, inp.W2_64, b)
