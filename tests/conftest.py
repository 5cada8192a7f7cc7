import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.lib()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Totals of the attention parity checks of the session: rows compared with the oracle, the worst
    row-normwise error (the bar) and the worst element-wise error (floor 1e-3 of the row's maximum)."""
    mod = sys.modules.get("tests.gpu_util")
    rec = getattr(mod, "RECORD", None) if mod else None
    if not rec:
        return
    rows = sum(r.compared for r in rec)
    flagged = sum(r.flagged for r in rec)
    terminalreporter.write_line(
        f"attention parity: {len(rec)} checks, {rows} rows compared, {flagged} flagged; worst row-normwise "
        f"{max(r.worst for r in rec):.3e}, worst element-wise {max(r.worst_elem for r in rec):.3e}")
