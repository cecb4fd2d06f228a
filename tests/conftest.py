import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(autouse=True)
def _parity_recorder(record_property):
    """Lets the parity helpers attach the errors they measured to the test."""
    import _parity_log
    _parity_log.RECORD = record_property
    yield
    _parity_log.RECORD = None


def pytest_terminal_summary(terminalreporter):
    """One line per GPU test with the errors it measured against the oracle."""
    lines = []
    for outcome in ("passed", "failed"):
        for rep in terminalreporter.stats.get(outcome, []):
            for name, val in getattr(rep, "user_properties", []):
                if name == "parity" and isinstance(val, dict):
                    errs = " ".join(f"{k}={v:.2e}" for k, v in val.items())
                    lines.append(f"{rep.nodeid.split('::', 1)[-1]} [{outcome}]: {errs}")
    if lines:
        terminalreporter.write_sep("-", "measured errors against the oracle (bounds in tests/test_parity_gpu.py)")
        for line in lines:
            terminalreporter.write_line(line)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    from chunked_lm_head_linear_gb300 import lce
    lce.load()
    return lce
