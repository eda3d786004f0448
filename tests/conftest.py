import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity report of the GPU tests that recorded one (max / mean |err|, and
    the error in ULPs of the output format where |ref| >= 2^-6), printed at
    the end and written as JSON to $PARITY_REPORT when that is set."""
    try:
        from tests.helpers import PARITY
    except Exception:
        return
    if not PARITY:
        return
    tr = terminalreporter
    tr.section("parity vs the fp64 oracle")
    for r in PARITY:
        tr.write_line(f"{r['case']:<48} n={r['elements']:>9}  max|err|={r['max_abs']:.2e}  "
                      f"mean|err|={r['mean_abs']:.2e}  ULP (|ref|>=2^-6) max={r['max_ulp']:.1f} "
                      f"p99.9={r['p999_ulp']:.2f}")
    path = os.environ.get("PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(PARITY, f, indent=1)
