import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture
def golden():
    return read_golden


def pytest_terminal_summary(terminalreporter):
    """Record how many stochastic positions the parity tests compared and how
    many of those the margin rule excused (the bound is under 0.01 %)."""
    mod = sys.modules.get("tests.gpu_parity")
    if mod is None or mod.SESSION.rows == 0:
        return
    t = mod.SESSION
    terminalreporter.write_line(
        f"stochastic parity: {t.rows} positions in {t.sequences} sequences compared, "
        f"{t.margin_rows} excused by the margin rule ({100.0 * t.margin_rows / t.rows:.4f} %)")
