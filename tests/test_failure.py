"""The failure path every kernel shares, made to run on the GPU without a fault: a
bounded wait on a barrier that nothing completes gives up after the library's limit,
the device status word reports ATTN_ERR_DEVICE_TIMEOUT once, and the context stays
usable (the next call runs and reports a clean status)."""
import time

import numpy as np
import pytest
import torch

from tests import helpers as H
from workloads import TINY, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_gives_up_reports_and_recovers():
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import _lib
    assert ea.device_status() == 0
    t0 = time.perf_counter()
    ea.selftest_wait_timeout()
    status = ea.device_status()  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == 7 and _lib.STATUS_NAMES[7] == "ATTN_ERR_DEVICE_TIMEOUT"
    assert 1.5 < elapsed < 30.0, elapsed  # the limit is 2 s of the device clock
    assert ea.device_status() == 0  # reported once, then cleared
    # the context is still usable: a forward runs and matches the oracle
    inputs = make_inputs(TINY)
    o, lse = H.run_forward(TINY, "tc", inputs)
    o_ref, l_ref = H.oracle_forward(TINY, inputs)
    H.check_forward(o, lse, o_ref, l_ref, "after the timeout")
    assert np.isfinite(o).all()
    torch.cuda.synchronize()


@pytest.mark.parametrize("offs,n,ok", [
    ([0, 100, 250, 300], 300, True),
    ([0, 0, 300], 300, True),             # an empty document is allowed
    ([0, 200, 100, 300], 300, False),     # not non-decreasing
    ([0, 100, 250], 300, False),          # does not end at N
    ([5, 100, 300], 300, False),          # does not start at 0
    ([0, 100, 400], 300, False),          # ends past N
])
def test_document_offsets_check(offs, n, ok):
    """attn_check_doc_offsets records a bad table in the device status word
    (ATTN_ERR_DEVICE_INPUT, reported once by attn_device_status); a good one leaves it
    clean. The check kernel reads the table only."""
    import exact_io_aware_13_gb300 as ea
    assert ea.device_status() == 0
    ea.check_doc_offsets(torch.tensor(offs, dtype=torch.int32, device="cuda"), n)
    assert ea.device_status() == (0 if ok else 8)
    assert ea.device_status() == 0


def test_checked_mode_checks_every_document_call():
    """With ATTN_CHECKED=1 in the environment, a call with the document mask checks its
    table first: run in a fresh process, a tile classification (a kernel that reads the
    table within its bounds and writes only the class array) on a table that does not
    end at N reports ATTN_ERR_DEVICE_INPUT, and one on a good table reports nothing.
    Without the variable the table is trusted and nothing is reported."""
    import os
    import subprocess
    import sys
    code = (
        "import torch, exact_io_aware_13_gb300 as ea\n"
        "good = torch.tensor([0, 100, 300], dtype=torch.int32, device='cuda')\n"
        "bad = torch.tensor([0, 100, 250], dtype=torch.int32, device='cuda')\n"
        "ea.classify_tiles(ea.MASK_DOCUMENT_CAUSAL, 300, 300, doc_offsets=good)\n"
        "a = ea.device_status()\n"
        "ea.classify_tiles(ea.MASK_DOCUMENT_CAUSAL, 300, 300, doc_offsets=bad)\n"
        "b = ea.device_status()\n"
        "print(a, b)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for env_value, want in (("1", "0 8"), ("0", "0 0")):
        env = dict(os.environ, ATTN_CHECKED=env_value)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                           cwd=root, env=env, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        assert r.stdout.split()[-2:] == want.split(), (env_value, r.stdout)
