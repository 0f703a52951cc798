"""attn_bwd_static_workspace: the backward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the backward pass (their device
memory is already handed out to another allocator, or their runtime forbids new
allocations after start-up). This entry point serves them: it takes the same
inputs and outputs as attn_bwd but keeps the backward's scratch in an array inside
the library. The test calls it through the C ABI several times in a row, on different
problems (d = 64, 128 and 256), and checks each result against attn_bwd on the same
inputs: both run the same deterministic kernels in the same order, so dq, dk and dv
must be bit for bit equal (the gradient tolerance of the other parity tests is checked
as well). It also checks that an oversized problem is refused before anything runs.

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


def _static_backward(lib, w, qd, kd, vd, o, lse, dod, dt, outs=None):
    from exact_io_aware_13_gb300 import _lib
    if outs is None:
        outs = (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd))
    dq, dk, dv = outs
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
        H.small_workload("static-3", MASK_CAUSAL, SCORE_ALIBI, B=1, Hq=2, Hkv=1, N=300,
                         d=256, seed=13),
    ]
    for w in problems:  # calls in a row; each reuses the array the one before filled
        q, k, v, do, offs = make_inputs(w, with_dout=True)
        qd, kd, vd, dod = H.to_dev(q, k, v, do)
        dt = H.doc_tensor(offs)
        kw = H.mask_kwargs(w, offs)
        o, lse = ea.forward(qd, kd, vd, scale=w.scale, doc_offsets=dt, **kw)
        ref = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, doc_offsets=dt, **kw)
        got = _static_backward(lib, w, qd, kd, vd, o, lse, dod, dt)
        torch.cuda.synchronize()
        assert ea.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g, r), f"{w.name}: {name} differs from attn_bwd"
        H.check_grads([t.float().cpu().numpy() for t in got],
                      [t.float().cpu().numpy().astype(np.float64) for t in ref], w.name,
                      d=w.d)


def test_static_workspace_backward_writes_only_its_outputs(lib):
    """dq, dk and dv as views inside buffers of sentinel guard bytes (ragged lengths,
    GQA): the entry point writes nothing outside them."""
    import exact_io_aware_13_gb300 as ea
    from tests.test_canaries import Guarded
    w = H.small_workload("static-guard", MASK_CAUSAL, SCORE_SOFTCAP, B=1, Hq=4, Hkv=2, N=513,
                         Nkv=513, d=128, softcap=20.0, seed=14)
    q, k, v, do, offs = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    kw = H.mask_kwargs(w, offs)
    o, lse = ea.forward(qd, kd, vd, scale=w.scale, **kw)
    ref = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, **kw)
    bufs = [Guarded(qd.shape, torch.bfloat16), Guarded(kd.shape, torch.bfloat16),
            Guarded(vd.shape, torch.bfloat16)]
    _static_backward(lib, w, qd, kd, vd, o, lse, dod, None, outs=[g.view for g in bufs])
    assert all(g.intact() for g in bufs)
    for g, r in zip(bufs, ref):
        assert torch.equal(g.view, r)


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
