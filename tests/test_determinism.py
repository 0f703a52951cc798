"""Bitwise determinism of the forward and backward passes (same inputs, same bits)."""
import pytest
import torch

from tests import helpers as H
from workloads import MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, SCORE_ALIBI, SCORE_SOFTCAP, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("mask,score", [(MASK_CAUSAL, 0),
                                        (MASK_DOCUMENT_CAUSAL, SCORE_ALIBI | SCORE_SOFTCAP)])
def test_forward_and_backward_are_bitwise_repeatable(mask, score):
    import exact_io_aware_13_gb300 as ea
    w = H.small_workload("det", mask, score, B=2, Hq=8, Hkv=2, N=1500, d=128,
                         softcap=30.0 if score else 0.0, doc_lo=100, doc_hi=700)
    q, k, v, do, offs = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    dt = H.doc_tensor(offs)
    kw = H.mask_kwargs(w, offs)
    runs = []
    for _ in range(3):
        o, lse = ea.forward(qd, kd, vd, scale=w.scale, doc_offsets=dt, **kw)
        dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, doc_offsets=dt, **kw)
        runs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    torch.cuda.synchronize()
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)


def test_backward_phases_equal_attn_bwd():
    """attn_bwd_phases run kernel by kernel gives the same bits as attn_bwd."""
    import exact_io_aware_13_gb300 as ea
    w = H.small_workload("phases", MASK_CAUSAL, B=1, Hq=4, Hkv=2, N=640, d=128)
    q, k, v, do, offs = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    kw = H.mask_kwargs(w, offs)
    o, lse = ea.forward(qd, kd, vd, scale=w.scale, **kw)
    ref = ea.backward(qd, kd, vd, o, lse, dod, scale=w.scale, **kw)
    got = [torch.empty_like(t) for t in ref]
    ws = torch.empty(ea.bwd_workspace_size(qd, kd), dtype=torch.uint8, device="cuda")
    for ph in (ea.BWD_ROWDOT, ea.BWD_DQ, ea.BWD_DKDV):  # dq before dkdv: independent
        ea.bwd_phases_into(ph, qd, kd, vd, o, lse, dod, *got, ws, scale=w.scale, **kw)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
