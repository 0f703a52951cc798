import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The largest flat forward error max|O - O_ref| (elements with |O_ref| < 4) over every
    forward parity check of the session, and the checks that came closest to 1e-2."""
    from tests import helpers
    log = helpers.FORWARD_LOG
    if not log:
        return
    worst = sorted(log, key=lambda r: -r[1])
    n_el = sum(r[2] for r in log)
    n_big = sum(r[3] for r in log)
    tr = terminalreporter
    tr.write_sep("-", "forward parity: flat max|O - O_ref| over |O_ref| < 4")
    tr.write_line(f"{len(log)} checks, {n_el} elements ({n_big} with |O_ref| >= 4); "
                  f"largest flat max|dO| = {worst[0][1]:.3e} ({worst[0][0]})")
    for what, flat_max, n, big in worst[:8]:
        tr.write_line(f"  {flat_max:.3e}  {what}  ({n} elements, {big} at |O_ref| >= 4)")
