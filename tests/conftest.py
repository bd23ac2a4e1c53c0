import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Per test, the largest relative L2 error of its outputs against the oracle
    rounded to bf16 (the gate) and against the unrounded FP64 oracle (the margin
    the bf16 output rounding takes), from every comparison the test made."""
    helpers = sys.modules.get("tests.helpers")
    rows = getattr(helpers, "REPORT", None)
    if not rows:
        return
    worst = {}
    for name, eb, eu in rows:
        b, u = worst.get(name, (0.0, 0.0))
        worst[name] = (max(b, eb), max(u, eu))
    tr = terminalreporter
    tr.write_sep("-", "rel-L2 against the oracle: bf16(oracle) (gated at 2e-3) / unrounded")
    for name, (b, u) in sorted(worst.items()):
        tr.write_line(f"{b:.2e} / {u:.2e}  {name}")
    tr.write_line(f"max over {len(rows)} comparisons: {max(r[1] for r in rows):.2e} / "
                  f"{max(r[2] for r in rows):.2e}")
