import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst parity errors per test (normwise, gated at 2e-3; elementwise with
    a floor, for information), so that a quiet run's output shows the
    magnitudes and not only the pass count."""
    try:
        from parity_util import RECORD
    except ImportError:
        return
    if not RECORD:
        return
    tr = terminalreporter
    tr.write_line("parity vs the fp64 oracle (worst over cases; normwise | elementwise):")
    for name in sorted(RECORD):
        r = RECORD[name]
        parts = []
        for q in ("o", "S", "A", "zk"):
            if q in r:
                el = r.get(q + "_el")
                parts.append(f"{q} {r[q]:.1e}" + (f"|{el:.1e}" if el is not None else ""))
        extra = [f"{k} {v:.1e}" for k, v in sorted(r.items())
                 if k not in ("n", "o", "S", "A", "zk") and not k.endswith("_el")]
        tr.write_line(f"  {name} (n={r['n']}): " + " ".join(parts + extra))
