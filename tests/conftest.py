import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Raw errors of the workload parity checks made in this session (worst over the
    sampled slices): the O error before and after the storage allowance, how many
    elements needed it, the LSE error and the gradients' relative Frobenius errors."""
    try:
        from parity import RECORD
    except ImportError:
        return
    if not RECORD:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the fp64 oracle (worst over sampled slices)")
    for label, r in RECORD.items():
        grads = " ".join(f"{n} {r[n]:.2e}" for n in ("dq", "dk", "dv") if n in r)
        tr.write_line(
            f"{label}: slices {r['slices']}, O max {r['o_max']:.4f} "
            f"(|O_ref|<2: {r['o_max_below2']:.4f}), elements over 1e-2 {r['o_allowance_used']}, "
            f"LSE {r.get('lse_max', float('nan')):.2e}, {grads}")
