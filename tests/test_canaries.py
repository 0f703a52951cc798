"""Guard bytes around every buffer the library writes: no entry point may write outside
the outputs and workspace it is given.

Each output (and each caller workspace) is an offset view into a larger device buffer
whose bytes before and after the view hold a sentinel pattern. After the call the test
checks that every guard byte still holds the sentinel, and that the guarded outputs are
bit for bit those of the same call on plainly allocated buffers (so the view offsets
changed nothing). The cases are the ones whose epilogues handle ragged edges: lengths of
1, 129, 300 and 513 rows, unequal query and key lengths, d = 64, 128 and 256, dropout,
the FP8 quantiser and forward on a ragged tail, and paged decode with pages of 8 and 64
keys in split mode. The views start 4 KiB into their buffers, so they keep the 16-byte
(indeed 256-byte) alignment the library requires.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import helpers as H
from workloads import (MASK_CAUSAL, MASK_DOCUMENT_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW,
                       SCORE_ALIBI, SCORE_SOFTCAP, DecodeWorkload, make_decode_inputs,
                       make_inputs)

pytestmark = pytest.mark.gpu

GUARD = 4096          # guard bytes before and after each view
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


class Guarded:
    """A device buffer of GUARD sentinel bytes, the view's bytes (also set to the
    sentinel) and GUARD more sentinel bytes, rounded up to 256 bytes."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        total = GUARD + (n + 255) // 256 * 256 + GUARD
        self.raw = torch.full((total,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.view = self.raw[GUARD:GUARD + n].view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        before = self.raw[:GUARD]
        after = self.raw[GUARD + self.n:]
        return bool((before == SENTINEL).all()) and bool((after == SENTINEL).all())


def _check_all(bufs, what):
    bad = [name for name, g in bufs.items() if not g.intact()]
    assert not bad, f"{what}: guard bytes overwritten around {bad}"


FWD_CASES = [
    # (name, mask, score, B, Hq, Hkv, Nq, Nkv, d, window, dropout_p)
    ("n1", MASK_NONE, 0, 1, 2, 1, 1, 129, 128, 0, 0.0),
    ("n129", MASK_CAUSAL, 0, 2, 2, 1, 129, 129, 64, 0, 0.0),
    ("n300win", MASK_SLIDING_WINDOW, SCORE_ALIBI, 1, 4, 2, 300, 300, 128, 100, 0.0),
    ("n513docs", MASK_DOCUMENT_CAUSAL, SCORE_ALIBI | SCORE_SOFTCAP, 1, 2, 2, 513, 513, 64, 0,
     0.0),
    ("nq450nkv200", MASK_CAUSAL, 0, 1, 2, 1, 450, 200, 128, 0, 0.0),
    ("nq200nkv450", MASK_NONE, SCORE_SOFTCAP, 1, 2, 2, 200, 450, 128, 0, 0.0),
    ("d256n300", MASK_CAUSAL, SCORE_ALIBI, 1, 2, 1, 300, 300, 256, 0, 0.0),
    ("d256n129", MASK_NONE, 0, 1, 2, 2, 129, 513, 256, 0, 0.0),
    ("drop300", MASK_CAUSAL, SCORE_ALIBI, 1, 4, 2, 300, 300, 128, 0, 0.2),
    ("drop513d64", MASK_SLIDING_WINDOW, 0, 1, 2, 1, 513, 513, 64, 200, 0.5),
]


def _workload(case):
    name, mask, score, B, Hq, Hkv, Nq, Nkv, d, window, p = case
    w = H.small_workload(f"guard {name}", mask, score, B=B, Hq=Hq, Hkv=Hkv, N=Nq, Nkv=Nkv,
                         d=d, window=window, softcap=20.0 if score & SCORE_SOFTCAP else 0.0,
                         seed=500 + Nq + Nkv + d, doc_lo=60, doc_hi=200)
    if p > 0:
        w = w.replace(dropout_p=p, dropout_seed=0x1234_5678_9ABC)
    return w


def _impls(w):
    simt_ok = w.d <= 128 and w.dropout_p == 0
    return ["tc", "simt"] if simt_ok else ["tc"]


@pytest.mark.parametrize("case", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_forward_writes_only_its_outputs(case):
    """attn_fwd (and attn_fwd_simt where it applies)."""
    import exact_io_aware_13_gb300 as ea
    w = _workload(case)
    q, k, v, _, offs = make_inputs(w)
    qd, kd, vd = H.to_dev(q, k, v)
    dt = H.doc_tensor(offs)
    kw = dict(scale=w.scale, doc_offsets=dt, **H.mask_kwargs(w, offs))
    for impl in _impls(w):
        o_ref, l_ref = ea.forward(qd, kd, vd, impl=impl, **kw)
        bufs = {"o": Guarded(qd.shape, torch.bfloat16),
                "lse": Guarded(qd.shape[:-1], torch.float32)}
        ea.fwd_into(qd, kd, vd, bufs["o"].view, bufs["lse"].view, impl=impl, **kw)
        _check_all(bufs, f"{w.name} {impl}")
        assert torch.equal(bufs["o"].view, o_ref) and torch.equal(bufs["lse"].view, l_ref)
        assert ea.device_status() == 0


@pytest.mark.parametrize("case", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_backward_writes_only_its_outputs_and_workspace(case):
    """attn_bwd (and attn_bwd_simt where it applies), workspace guarded too."""
    import exact_io_aware_13_gb300 as ea
    w = _workload(case)
    q, k, v, do, offs = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    dt = H.doc_tensor(offs)
    kw = dict(scale=w.scale, doc_offsets=dt, **H.mask_kwargs(w, offs))
    o, lse = ea.forward(qd, kd, vd, **kw)
    ws_bytes = ea.bwd_workspace_size(qd, kd)
    for impl in _impls(w):
        ref = ea.backward(qd, kd, vd, o, lse, dod, impl=impl, **kw)
        bufs = {"dq": Guarded(qd.shape, torch.bfloat16), "dk": Guarded(kd.shape, torch.bfloat16),
                "dv": Guarded(vd.shape, torch.bfloat16),
                "workspace": Guarded((ws_bytes,), torch.uint8)}
        ea.bwd_into(qd, kd, vd, o, lse, dod, bufs["dq"].view, bufs["dk"].view, bufs["dv"].view,
                    bufs["workspace"].view, impl=impl, **kw)
        _check_all(bufs, f"{w.name} {impl}")
        for name, r in zip(("dq", "dk", "dv"), ref):
            assert torch.equal(bufs[name].view, r), f"{w.name} {impl}: {name}"
        assert ea.device_status() == 0


@pytest.mark.parametrize("case", [c for c in FWD_CASES if c[0] in ("n300win", "d256n300",
                                                                    "drop513d64", "n1")],
                         ids=["n300win", "d256n300", "drop513d64", "n1"])
def test_backward_phases_write_only_their_outputs(case):
    """attn_bwd_phases, one kernel per call: the row kernel writes only the workspace,
    the dK/dV kernel only dk and dv, the dQ kernel only dq."""
    import exact_io_aware_13_gb300 as ea
    w = _workload(case)
    q, k, v, do, offs = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = H.to_dev(q, k, v, do)
    dt = H.doc_tensor(offs)
    kw = dict(scale=w.scale, doc_offsets=dt, **H.mask_kwargs(w, offs))
    o, lse = ea.forward(qd, kd, vd, **kw)
    ref = ea.backward(qd, kd, vd, o, lse, dod, **kw)
    bufs = {"dq": Guarded(qd.shape, torch.bfloat16), "dk": Guarded(kd.shape, torch.bfloat16),
            "dv": Guarded(vd.shape, torch.bfloat16),
            "workspace": Guarded((ea.bwd_workspace_size(qd, kd),), torch.uint8)}
    untouched = {n: bufs[n].raw.clone() for n in ("dq", "dk", "dv")}
    ea.bwd_phases_into(ea.BWD_ROWDOT, qd, kd, vd, o, lse, dod, bufs["dq"].view, bufs["dk"].view,
                       bufs["dv"].view, bufs["workspace"].view, **kw)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv"):  # the row kernel writes the workspace only
        assert torch.equal(bufs[n].raw, untouched[n]), f"row kernel wrote into {n}"
    for ph in (ea.BWD_DKDV, ea.BWD_DQ):
        ea.bwd_phases_into(ph, qd, kd, vd, o, lse, dod, bufs["dq"].view, bufs["dk"].view,
                           bufs["dv"].view, bufs["workspace"].view, **kw)
        _check_all(bufs, f"{w.name} phase {ph}")
    for name, r in zip(("dq", "dk", "dv"), ref):
        assert torch.equal(bufs[name].view, r), f"{w.name}: {name}"
    assert ea.device_status() == 0


@pytest.mark.parametrize("n", [1, 129, 300])
def test_fp8_quantiser_and_forward_write_only_their_outputs(n):
    """attn_quantize_fp8 (both layouts) and attn_fwd_fp8 on ragged lengths."""
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import _lib
    w = H.small_workload(f"guard fp8 {n}", MASK_CAUSAL, SCORE_ALIBI, B=1, Hq=2, Hkv=1, N=n,
                         d=128, seed=600 + n)
    q, k, v, _, _ = make_inputs(w)
    qd, kd, vd = H.to_dev(q, k, v)
    lib = _lib.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    quant = {}
    for name, x, layout in (("q", qd, ea.FP8_TILES), ("k", kd, ea.FP8_TILES),
                            ("v", vd, ea.FP8_V_TRANSPOSED)):
        B, Hh, N, d = x.shape
        codes_ref, scales_ref = ea.quantize_fp8(x, layout)
        bufs = {"codes": Guarded(codes_ref.shape, torch.uint8),
                "scales": Guarded(scales_ref.shape, torch.float32)}
        rc = lib.attn_quantize_fp8(ctypes.c_void_p(x.data_ptr()),
                                   ctypes.c_void_p(bufs["codes"].view.data_ptr()),
                                   ctypes.c_void_p(bufs["scales"].view.data_ptr()),
                                   B * Hh, N, d, layout, st)
        assert rc == 0
        _check_all(bufs, f"quantise {name} n={n}")
        assert torch.equal(bufs["codes"].view, codes_ref)
        assert torch.equal(bufs["scales"].view, scales_ref)
        quant[name] = (codes_ref, scales_ref)
    (q8, sq), (k8, sk), (v8t, sv) = quant["q"], quant["k"], quant["v"]
    kw = dict(Nkv=w.Nkv, scale=w.scale, mask_kind=w.mask_kind, score_kind=w.score_kind)
    o_ref = torch.empty_like(qd)
    l_ref = torch.empty(qd.shape[:-1], dtype=torch.float32, device="cuda")
    ea.fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o_ref, l_ref, **kw)
    bufs = {"o": Guarded(qd.shape, torch.bfloat16), "lse": Guarded(qd.shape[:-1], torch.float32)}
    ea.fwd_fp8_into(q8, sq, k8, sk, v8t, sv, bufs["o"].view, bufs["lse"].view, **kw)
    _check_all(bufs, f"fp8 forward n={n}")
    assert torch.equal(bufs["o"].view, o_ref) and torch.equal(bufs["lse"].view, l_ref)
    assert ea.device_status() == 0


@pytest.mark.parametrize("page_size", [8, 64])
@pytest.mark.parametrize("nq", [1, 3])
def test_decode_writes_only_its_outputs_and_workspace(page_size, nq):
    """attn_decode_paged in split mode (several key chunks, so the partials go through
    the workspace and the combine kernel)."""
    import exact_io_aware_13_gb300 as ea
    lengths = (0, 1, 63, 65, 700)
    w = DecodeWorkload(name="guard decode", seed=70 + page_size + nq, B=len(lengths), Hq=8,
                       Hkv=2, Nq=nq, d=128, len_min=0, len_max=max(lengths), page_size=page_size,
                       lengths=lengths, mask_kind=MASK_CAUSAL, score_kind=SCORE_ALIBI)
    q, kc, vc, table, lens = [t.cuda() for t in make_decode_inputs(w, poison_unused=True)]
    msl = int(table.shape[1] * page_size)
    split = 128
    kw = dict(max_seq_len=msl, split_keys=split, scale=w.scale, mask_kind=w.mask_kind,
              score_kind=w.score_kind)
    o_ref, l_ref = ea.decode_paged(q, kc, vc, table, lens, **kw)
    ws_bytes = ea.decode_workspace_size(w.B, w.Hq, w.Hkv, nq, w.d, msl, split)
    assert ws_bytes > 0
    bufs = {"o": Guarded(q.shape, torch.bfloat16), "lse": Guarded(q.shape[:-1], torch.float32),
            "workspace": Guarded((ws_bytes,), torch.uint8)}
    ea.decode_paged_into(q, kc, vc, table, lens, bufs["o"].view, bufs["lse"].view,
                         bufs["workspace"].view, **kw)
    _check_all(bufs, f"decode page {page_size} nq {nq}")
    assert torch.equal(bufs["o"].view, o_ref) and torch.equal(bufs["lse"].view, l_ref)
    assert ea.device_status() == 0
