import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Measured parity errors of every comparison the GPU tests made."""
    try:
        from tests.gpu_common import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.section("measured parity errors (max |err|, max err/bound, elements over bound)")
    agg = {}
    for r in PARITY_LOG:
        key = (r["test"].split("::")[-1], r["name"])
        a = agg.setdefault(key, {"n": 0, "max_abs": 0.0, "ratio": 0.0, "over": 0, "ulps": 0.0,
                                 "rms": 0.0})
        a["n"] += r["n"]
        a["max_abs"] = max(a["max_abs"], r["max_abs"])
        a["ratio"] = max(a["ratio"], r["max_over_bound"])
        a["over"] += r["n_over_bound"]
        a["ulps"] = max(a["ulps"], r["max_ulps"])
        a["rms"] = max(a["rms"], r.get("max_over_row_rms", 0.0))
    for (t, n), a in sorted(agg.items()):
        tr.write_line(f"{t:60s} {n:10s} n={a['n']:9d} max_abs={a['max_abs']:.3e} "
                      f"max/bound={a['ratio']:.3f} over={a['over']} ulps={a['ulps']:.1f} "
                      f"/rowrms={a['rms']:.2e}")
