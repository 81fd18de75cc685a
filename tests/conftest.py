import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import speculative_verify_paged_gb300 as sv
    return sv


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Excused sampling decisions (uniform within 1e-5 of a boundary where the
    GPU and the oracle differ), counted over every comparison of the run."""
    try:
        import parity_utils
    except ImportError:
        return
    rows = parity_utils.EXCUSALS
    if not rows:
        return
    exc = sum(r[1] for r in rows)
    dec = sum(r[2] for r in rows)
    terminalreporter.write_line("sampling parity: %d excused sequences over %d decisions in %d comparisons "
                                "(bar: < %.2g of the decisions of each comparison)"
                                % (exc, dec, len(rows), parity_utils.MAX_EXCUSED_FRACTION))
    for name, e, d in rows:
        if e:
            terminalreporter.write_line("  %s: %d excused of %d decisions" % (name, e, d))
