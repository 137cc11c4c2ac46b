import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmoe.so")
    config.addinivalue_line("markers", "slow: longer oracle runs")


def pytest_terminal_summary(terminalreporter):
    """Per output-parity check: rel-L2, the bare max|err|/rms and the max error
    beyond the rounding-point allowance / rms (the figure held to 1e-2)."""
    try:
        from tests.tolerances import RECORDS
    except Exception:  # noqa: BLE001 - the summary is informational
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", f"output parity: {len(RECORDS)} checks (rel-L2 <= 5e-3; max beyond allowance <= 1e-2 rms)")
    tr.write_line(f"{'check':<60} {'rel-L2':>10} {'max|err|/rms':>13} {'beyond/rms':>11}")
    for what, r in RECORDS:
        tr.write_line(f"{what[:60]:<60} {r['rel_l2']:>10.3e} {r['max_err_over_rms']:>13.3e} "
                      f"{r['max_beyond_over_rms']:>11.3e}")
    worst = max(r["max_err_over_rms"] for _, r in RECORDS)
    tr.write_line(f"largest bare max|err|/rms: {worst:.3e}; largest rel-L2: {max(r['rel_l2'] for _, r in RECORDS):.3e}")
