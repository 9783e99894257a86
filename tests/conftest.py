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
    """Per check: the literal max|err|/RMS(ref) next to the bound applied, and
    the near-tie tokens each routing comparison tolerated (GPU runs)."""
    try:
        import parity
    except ImportError:
        return
    if not parity.RECORDS and not parity.TIE_RECORDS:
        return
    tr = terminalreporter
    tr.section("parity statistics (against the fp64 oracle)")
    if parity.RECORDS:
        worst = max(r[1] for r in parity.RECORDS)
        n_over = sum(1 for r in parity.RECORDS if r[1] > parity.MAX_REL_RMS)
        tr.write_line("%d float checks; strict max|err|/RMS: worst %.4g, %d above 2e-2 "
                      "(those pass through the bf16 allowance)" % (len(parity.RECORDS), worst, n_over))
        tr.write_line("%-34s %12s %16s %10s" % ("check", "max|err|/RMS", "beyond-allow/RMS", "rel L1"))
        seen = {}
        for name, strict, beyond, l1 in parity.RECORDS:   # worst case per check name
            if name not in seen or strict > seen[name][0]:
                seen[name] = (strict, beyond, l1)
        for name in sorted(seen, key=lambda n: -seen[n][0]):
            strict, beyond, l1 = seen[name]
            tr.write_line("%-34s %12.4g %16.4g %10.3g" % (name[:34], strict, beyond, l1))
    if parity.TIE_RECORDS:
        tr.write_line("near-tie tokens tolerated per routing comparison: " +
                      ", ".join("%s %d" % r for r in parity.TIE_RECORDS))
