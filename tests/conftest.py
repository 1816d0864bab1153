import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")


def pytest_terminal_summary(terminalreporter):
    """The oracle-parity checks of this session: rows compared and every
    near-tie exception (a decision that differs from the oracle's where the
    oracle's two candidates lie within the logits' tolerance)."""
    try:
        from tests.gpu_helpers import PARITY_REPORT
    except ImportError:
        return
    if not PARITY_REPORT:
        return
    rows = sum(n for _, n, _ in PARITY_REPORT)
    listed = [(label, e) for label, _, exc in PARITY_REPORT for e in exc]
    tr = terminalreporter
    tr.write_sep("-", "oracle parity: near-tie exceptions (listed, not hidden)")
    for label, e in listed:
        tr.write_line(f"  {label}: {e}")
    tr.write_line(f"oracle parity: {len(PARITY_REPORT)} checks, {rows} rows compared, "
                  f"{len(listed)} near-tie exceptions listed above")
