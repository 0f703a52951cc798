"""attn_bwd_static_workspace: the backward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the backward pass (their device
memory is already handed out to another allocator, or their runtime forbids new
allocations after start-up). This entry point serves them: it takes the same
inputs and outputs as attn_bwd but keeps the backward's scratch in an array inside
the library. The test calls it through the C ABI twice in a row, on two different
problems, and checks each result against attn_bwd on the same inputs, with the
tolerance of the other parity tests. It also checks that an oversized problem is
refused before anything runs.

The file name sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import helpers as H
from workloads import MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, SCORE_ALIBI, SCORE_SOFTCAP, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_13_gb300 import _lib
    return _lib.load()


def _static_backward(lib, w, qd, kd, vd, o, lse, dod, dt):
    from exact_io_aware_13_gb300 import _lib
    dq = torch.empty_like(qd)
    dk = torch.empty_like(kd)
    dv = torch.empty_like(vd)
    mp = _lib.MaskParams(w.window, None if dt is None else dt.data_ptr(),
                         0 if dt is None else dt.numel() - 1)
    sp = _lib.ScoreParams(w.softcap)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.attn_bwd_static_workspace(
        p(qd), p(kd), p(vd), p(o), p(lse), p(dod), p(dq), p(dk), p(dv), w.B, w.Hq, w.Hkv,
        w.Nq, w.Nkv, w.d, ctypes.c_float(w.scale), w.mask_kind, ctypes.byref(mp),
        w.score_kind, ctypes.byref(sp), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.attn_strerror(rc).decode()
    return dq, dk, dv


def test_static_workspace_backward_matches_attn_bwd_twice(lib):
    import exact_io_aware_13_gb300 as ea
    problems = [
        H.small_workload("static-1", MASK_CAUSAL, B=2, Hq=4, Hkv=2, N=700, d=128, seed=11),
        H.small_workload("static-2", MASK_DOCUMENT_CAUSAL, SCORE_ALIBI | SCORE_SOFTCAP, B=1,
                         Hq=2, Hkv=1, N=333, d=64, softcap=30.0, seed=12),
    ]
    for w in problems:  # two calls in a row; the second reuses the array the first filled
        q, k, v, do, offs = make_inputs(w, with_dout=True)
        qd, kd, vd, dod = H.to_dev(q, k, v, do)
        dt = H.doc_tensor(offs)
        kw = H.mask_kwargs(w, offs)
        o, lse = ea.forward(qd, kd, vd, scale=w.scale, doc_offsets=dt, **kw)
        ref = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, doc_offsets=dt, **kw)
        got = _static_backward(lib, w, qd, kd, vd, o, lse, dod, dt)
        torch.cuda.synchronize()
        assert ea.device_status() == 0
        H.check_grads([t.float().cpu().numpy() for t in got],
                      [t.float().cpu().numpy().astype(np.float64) for t in ref], w.name)


def test_static_workspace_rejects_oversized_problems(lib):
    from exact_io_aware_13_gb300 import _lib
    rows_max = 1 << 21
    dummy = ctypes.c_void_p(256)
    # B * Hq * Nq128 = 2 * 16 * 65664 > 2^21: refused before any pointer is touched
    rc = lib.attn_bwd_static_workspace(*([dummy] * 9), 2, 16, 16, 65537, 65537, 128,
                                       ctypes.c_float(0.1), 0, None, 0, None, None)
    assert rc == 5 and 2 * 16 * 65664 > rows_max  # ATTN_ERR_WORKSPACE
    assert "workspace" in lib.attn_strerror(rc).decode()
    assert _lib.header_functions().count("attn_bwd_static_workspace") == 1
