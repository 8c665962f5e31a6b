import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


@pytest.fixture(scope="session")
def has_gpu():
    import torch
    return torch.cuda.is_available()


def pytest_terminal_summary(terminalreporter):
    """Print every parity comparison's measured rel-L2 beside its bar (the margin), and
    write them as JSON lines to $TTT_PARITY_LOG when that is set."""
    try:
        import ttt_testlib
    except ImportError:
        return
    rows = ttt_testlib.MARGINS
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity margins: rel-L2 against the oracle, and the bar")
    for r in rows:
        tr.write_line(f"{r['err']:.3e} / {r['bar']:.0e} ({r['err'] / r['bar']:6.1%})  {r['what']:<28} {r['test']}")
    worst = max(rows, key=lambda r: r["err"] / r["bar"])
    tr.write_line(f"worst: {worst['err']:.3e} of {worst['bar']:.0e} ({worst['err'] / worst['bar']:.1%}) "
                  f"{worst['what']} {worst['test']}")
    path = os.environ.get("TTT_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            for r in rows:
                f.write(json.dumps(r) + "\n")
