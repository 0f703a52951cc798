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
