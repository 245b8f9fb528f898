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
    """The C-ABI library, loaded through the binding (built on first use)."""
    from transformer_attention_backward_gb300 import _binding
    return _binding.load()


def pytest_terminal_summary(terminalreporter):
    """Both error figures of every GPU-vs-oracle comparison made through
    tests.helpers.checked: max |g - r| / max |r| (the bound) and the
    per-element max |g - r| / (|r| + 1e-6 max |r|) (reported only)."""
    from tests.helpers import PARITY_LOG
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.section("parity errors (max_rel = bound; elem_rel = per-element, reported)")
    worst = {}
    for tag, name, e, pe in PARITY_LOG:
        k = (tag, name)
        a, b = worst.get(k, (0.0, 0.0))
        worst[k] = (max(a, e), max(b, pe))
    for (tag, name), (e, pe) in sorted(worst.items()):
        tr.write_line(f"{tag:48s} {name:10s} max_rel {e:.3e}  elem_rel {pe:.3e}")
