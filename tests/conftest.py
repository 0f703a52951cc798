import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The largest flat forward error max|O - O_ref| over the elements with |O_ref| < 2
    (where the flat 1e-2 is asserted) and over |O_ref| < 4, across every forward parity
    check of the session (dropout checks, whose bound is relative to the output scale,
    listed apart), and the checks that came closest."""
    from tests import helpers
    log = helpers.FORWARD_LOG
    if not log:
        return
    tr = terminalreporter
    plain = [r for r in log if not r[5]]
    drop = [r for r in log if r[5]]
    tr.write_sep("-", "forward parity: flat max|O - O_ref|")
    for name, rows in (("no dropout", plain), ("dropout", drop)):
        if not rows:
            continue
        w2 = max(rows, key=lambda r: r[1])
        w4 = max(rows, key=lambda r: r[2])
        n_el = sum(r[3] for r in rows)
        n_over = sum(r[4] for r in rows)
        tr.write_line(f"{name}: {len(rows)} checks, {n_el} elements; |O_ref| < 2: "
                      f"{w2[1]:.3e} ({w2[0]}); |O_ref| < 4: {w4[2]:.3e} ({w4[0]}); "
                      f"elements at 2 <= |O_ref| < 4 above 1e-2: {n_over}")
    for what, m2, m4, n, over, dropped in sorted(plain, key=lambda r: -r[1])[:6]:
        tr.write_line(f"  {m2:.3e} (< 2)  {m4:.3e} (< 4)  {what}  ({n} elements)")
